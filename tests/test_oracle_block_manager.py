"""Pins for the oracle's block manager and cache operations (CPU only).

* the capacity model the pages print (128-block pool: contiguous reservation admits 4
  sequences, paged allocation 13 using 118 blocks);
* the two block-table figures (shared prefix block with ref_cnt 2; A=[3,0], B=[5,1,6], C=[2]);
* copy-on-write on a write into a shared block, fork of 4 children (ref_cnt 4);
* the waste bound and the return of every block to the free queue;
* KV write and block copy change exactly the addressed bytes.
"""
import json
import os

import numpy as np
import pytest

from oracle.block_manager import BlockManagerModel, NoBlocks, InvalidArg
from oracle.cache_ops import kv_write, copy_blocks
from oracle.paged_attention import slot_of_position


def _ceil(a, b):
    return -(-a // b)


def test_capacity_model_printed_output(golden_dir):
    fx = json.load(open(os.path.join(golden_dir, "capacity_model.json")))
    bs, pool, max_len, lens = fx["block_size"], fx["pool_blocks"], fx["max_len"], fx["lens"]
    exp = fx["expected"]
    # contiguous reservation: arithmetic only
    reserve = _ceil(max_len, bs)
    used = admitted = 0
    for L in lens:
        if used + reserve > pool:
            break
        used += reserve
        admitted += 1
    assert (reserve, admitted, used) == (exp["contiguous_reserve_per_seq"], exp["contiguous_admitted"],
                                          exp["contiguous_reserved_blocks"])
    assert sum(_ceil(L, bs) for L in lens[:admitted]) == exp["contiguous_really_used_blocks"]
    # paged: the block manager admits while the free queue can cover the prompt
    bm = BlockManagerModel(pool, bs)
    n = 0
    for i, L in enumerate(lens):
        try:
            bm.allocate(i, L)
        except NoBlocks:
            break
        n += 1
    assert n == exp["paged_admitted"]
    assert pool - bm.num_free() == exp["paged_used_blocks"]


def test_lecture33_shared_prefix_figure(golden_dir):
    fx = json.load(open(os.path.join(golden_dir, "block_table_diagrams.json")))["lecture33_figure"]
    bm = BlockManagerModel(fx["num_blocks"], fx["block_size"])
    for sid, (name, s) in enumerate(fx["seqs"].items()):
        bm.import_seq(sid, s["blocks"], s["tokens"])
    for b, r in fx["ref_cnt"].items():
        assert bm.ref_cnt[int(b)] == r
    tables, lens = bm.export([0, 1], 3)
    assert tables == [[7, 2, 5], [7, 9, -1]] and lens == [10, 6]
    # A's next token (position 10) lands in its half-full private block 5 at offset 2
    slot, cow = bm.append_slot(0)
    assert cow is None and slot == 5 * 4 + 2
    # B's next token (position 6) lands in block 9 at offset 2
    slot, cow = bm.append_slot(1)
    assert cow is None and slot == 9 * 4 + 2


def test_virtual_memory_figure_tables(golden_dir):
    fx = json.load(open(os.path.join(golden_dir, "block_table_diagrams.json")))["virtual_memory_figure"]
    bm = BlockManagerModel(fx["num_blocks"], fx["block_size"])
    for sid, s in enumerate(fx["seqs"].values()):
        bm.import_seq(sid, s["blocks"], 16 * len(s["blocks"]))
    assert bm.num_free() == 8 - 6
    assert sorted(bm.free_queue) == [4, 7]
    tables, _ = bm.export([0, 1, 2], 3)
    assert tables == [[3, 0, -1], [5, 1, 6], [2, -1, -1]]
    bm.free(1)                                          # B finishes: its blocks go to the tail
    assert list(bm.free_queue) == [4, 7, 5, 1, 6]


def test_decode_growth_one_block_at_a_time():
    bm = BlockManagerModel(8, 4)
    bm.allocate(0, 3)
    assert bm.tables[0] == [0]
    slots = [bm.append_slot(0)[0] for _ in range(6)]   # positions 3..8
    assert bm.tables[0] == [0, 1, 2]
    assert slots == [3, 4, 5, 6, 7, 8]
    assert [slot_of_position(bm.tables[0], p, 4) for p in range(3, 9)] == slots


def test_fork_then_copy_on_write():
    bs = 16
    bm = BlockManagerModel(16, bs)
    bm.allocate(0, 40)                                  # 3 blocks, last one half full
    for c in range(1, 5):                               # 4 parallel samples share everything
        bm.fork(0, c)
    assert all(bm.ref_cnt[b] == 5 for b in bm.tables[0])
    free_before = bm.num_free()
    slot, cow = bm.append_slot(1)                       # child 1 writes into the shared last block
    old = bm.tables[0][2]
    assert cow is not None and cow[0] == old and cow[1] == bm.tables[1][2] != old
    assert bm.ref_cnt[old] == 4 and bm.ref_cnt[cow[1]] == 1
    assert bm.tables[1][:2] == bm.tables[0][:2]
    assert slot == cow[1] * bs + 40 % bs
    assert bm.num_free() == free_before - 1
    slot, cow = bm.append_slot(1)                       # now private: no second copy
    assert cow is None


def test_exhaustion_and_errors_leave_state_unchanged():
    bm = BlockManagerModel(2, 16)
    bm.allocate(0, 32)
    with pytest.raises(NoBlocks):
        bm.append_slot(0)
    assert bm.num_tokens[0] == 32 and bm.tables[0] == [0, 1]
    with pytest.raises(NoBlocks):
        bm.allocate(1, 1)
    with pytest.raises(InvalidArg):
        bm.allocate(0, 1)


def test_random_workload_invariants():
    rng = np.random.default_rng(0)
    bs, nb = 16, 400
    bm = BlockManagerModel(nb, bs)
    live = []
    nxt = 0
    for step in range(2000):
        op = rng.integers(0, 4)
        try:
            if op == 0 or not live:
                bm.allocate(nxt, int(rng.integers(1, 100))); live.append(nxt); nxt += 1
            elif op == 1:
                bm.append_slot(int(rng.choice(live)))
            elif op == 2:
                bm.fork(int(rng.choice(live)), nxt); live.append(nxt); nxt += 1
            else:
                s = int(rng.choice(live)); bm.free(s); live.remove(s)
        except NoBlocks:
            pass
        # invariants: counts equal table references; free <=> count 0; waste bound
        refs = np.zeros(nb, dtype=int)
        for s in live:
            for b in bm.tables[s]:
                refs[b] += 1
            assert len(bm.tables[s]) * bs - bm.num_tokens[s] <= bs - 1
        assert list(refs) == bm.ref_cnt
        assert sorted(bm.free_queue) == [b for b in range(nb) if refs[b] == 0]
    for s in list(live):
        bm.free(s)
    assert bm.num_free() == nb and all(r == 0 for r in bm.ref_cnt)


def test_kv_write_touches_only_addressed_rows():
    rng = np.random.default_rng(2)
    k = rng.integers(0, 1 << 16, size=(10, 3, 16, 8), dtype=np.uint16)
    v = rng.integers(0, 1 << 16, size=(10, 3, 16, 8), dtype=np.uint16)
    kn = rng.integers(0, 1 << 16, size=(4, 3, 8), dtype=np.uint16)
    vn = rng.integers(0, 1 << 16, size=(4, 3, 8), dtype=np.uint16)
    slots = [37, -1, 160 - 1, 0]
    k2, v2 = kv_write(k, v, kn, vn, slots)
    touched = np.zeros((10, 16), dtype=bool)
    for t, s in enumerate(slots):
        if s < 0:
            continue
        assert np.array_equal(k2[s // 16, :, s % 16], kn[t])
        assert np.array_equal(v2[s // 16, :, s % 16], vn[t])
        touched[s // 16, s % 16] = True
    keep = ~touched[:, None, :, None].repeat(3, 1).repeat(8, 3)
    assert np.array_equal(k2[keep], k[keep]) and np.array_equal(v2[keep], v[keep])


def test_copy_blocks_copies_whole_blocks_only():
    rng = np.random.default_rng(3)
    k = rng.integers(0, 256, size=(12, 2, 16, 8), dtype=np.uint8)
    v = rng.integers(0, 256, size=(12, 2, 16, 8), dtype=np.uint8)
    pairs = [(1, 7), (1, 8), (4, 2)]
    k2, v2 = copy_blocks(k, v, pairs)
    for s, d in pairs:
        assert np.array_equal(k2[d], k[s]) and np.array_equal(v2[d], v[s])
    untouched = [b for b in range(12) if b not in (7, 8, 2)]
    assert np.array_equal(k2[untouched], k[untouched]) and np.array_equal(v2[untouched], v[untouched])
    with pytest.raises(AssertionError):
        copy_blocks(k, v, [(1, 2), (2, 3)])              # chained pair rejected
