"""CPU tests of the C ABI library: every declared symbol is exported, argument checks
refuse bad inputs without a GPU, and the C++ block manager matches the oracle's block
manager model bit for bit (and the pages' printed capacity numbers)."""
import ctypes
import json
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_symbols():
    src = open(os.path.join(ROOT, "include", "pkv.h")).read()
    return sorted(set(re.findall(r"PKV_API[^;(]*?\b(pkv_\w+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    import paged_kv_cache_160_gb300 as pkv
    names = _declared_symbols()
    assert len(names) >= 20
    raw = ctypes.CDLL(pkv._binding._LIB_PATH)
    for n in names:
        assert hasattr(raw, n), f"{n} declared in include/pkv.h but not exported"


def test_status_strings_and_version():
    import paged_kv_cache_160_gb300 as pkv
    assert pkv.lib.pkv_status_string(0) == b"ok"
    assert pkv.lib.pkv_status_string(5) == b"no free blocks"
    assert pkv.lib.pkv_version() >= 1


def test_decode_sm_budget_setting():
    """The decode SM budget is a host setting: 0 (every SM) by default, any n >= 0 is kept,
    a negative value is refused and leaves the budget as it was."""
    import paged_kv_cache_160_gb300 as pkv
    L = pkv.lib
    assert L.pkv_get_decode_sm_budget() == 0
    try:
        assert L.pkv_set_decode_sm_budget(64) == 0
        assert L.pkv_get_decode_sm_budget() == 64
        assert L.pkv_set_decode_sm_budget(-1) == 1              # PKV_ERR_INVALID_ARG
        assert L.pkv_get_decode_sm_budget() == 64
        pkv.pkv_set_decode_sm_budget(100000)                    # clamped to the SM count at launch
        assert pkv.pkv_get_decode_sm_budget() == 100000
        with pytest.raises(pkv.PkvError):
            pkv.pkv_set_decode_sm_budget(-5)
        # the workspace is sized for every SM whatever the budget
        args = (64, 28, 4, 128, 16, 2048, 0)
        pkv.pkv_set_decode_sm_budget(0)
        full = pkv.pkv_decode_workspace_bytes(*args)
        pkv.pkv_set_decode_sm_budget(1)
        assert pkv.pkv_decode_workspace_bytes(*args) == full > 0
    finally:
        pkv.pkv_set_decode_sm_budget(0)
    assert L.pkv_get_decode_sm_budget() == 0


def test_argument_checks_run_on_host_without_gpu():
    import paged_kv_cache_160_gb300 as pkv
    from paged_kv_cache_160_gb300._binding import CacheDesc
    L = pkv.lib
    desc = CacheDesc(64, 4, 16, 128, 1, None, None)
    # bad GQA split
    assert L.pkv_paged_decode(16, 16, 1, 4, 6, 16, 16, ctypes.byref(desc), 16, 8, 16, 128, 0.1, 0, 16, 1 << 20,
                              None) == 1
    # partition not a multiple of the block size
    assert L.pkv_paged_decode(16, 16, 1, 4, 8, 16, 16, ctypes.byref(desc), 16, 8, 16, 128, 0.1, 24, 16, 1 << 20,
                              None) == 1
    # unsupported head_dim
    d96 = CacheDesc(64, 4, 16, 96, 1, None, None)
    assert L.pkv_paged_decode(16, 16, 1, 4, 8, 16, 16, ctypes.byref(d96), 16, 8, 16, 128, 0.1, 0, 16, 1 << 20,
                              None) == 2
    # tile indices must fit 32 bits: 4 kv heads x 65536 sequences x 8192 tiles = 2^31
    assert L.pkv_paged_decode(16, 16, 1, 65536, 8, 16, 16, ctypes.byref(desc), 16, 8192, 16, 131072, 0.1, 0, 16,
                              1 << 20, None) == 2
    # fused append: both new-row pointers are required and 16-byte aligned
    assert L.pkv_paged_decode_append(16, 16, 1, 4, 8, None, 16, 16, 16, ctypes.byref(desc), 16, 8, 16, 128, 0.1,
                                     0, 16, 1 << 20, None) == 1
    assert L.pkv_paged_decode_append(16, 16, 1, 4, 8, 16, 24, 16, 16, ctypes.byref(desc), 16, 8, 16, 128, 0.1,
                                     0, 16, 1 << 20, None) == 1
    # misaligned pointer
    assert L.pkv_kv_write(17, 16, 1, 4, 16, 16, 16, ctypes.byref(desc), None) == 1
    # e4m3 cache without scales
    d8 = CacheDesc(64, 4, 16, 128, 2, None, None)
    assert L.pkv_copy_blocks(16, 16, ctypes.byref(d8), 16, 1, None) == 1
    # nothing to do is fine
    assert L.pkv_kv_write(16, 16, 1, 0, 16, 16, 16, ctypes.byref(desc), None) == 0
    assert L.pkv_copy_blocks(16, 16, ctypes.byref(desc), 16, 0, None) == 0
    assert L.pkv_decode_workspace_bytes(4, 6, 4, 128, 16, 100, 0) == 0       # bad split -> 0
    # swap_blocks: misaligned host pool, empty destination pool, missing pairs; no pairs is fine
    assert L.pkv_swap_blocks(16, 16, 8, 24, 16, 8, ctypes.byref(desc), 16, 2, None) == 1
    assert L.pkv_swap_blocks(16, 16, 0, 16, 16, 8, ctypes.byref(desc), 16, 2, None) == 1
    assert L.pkv_swap_blocks(16, 16, 8, 16, 16, 8, ctypes.byref(desc), None, 2, None) == 1
    assert L.pkv_swap_blocks(16, 16, 8, 16, 16, 8, ctypes.byref(desc), 16, 0, None) == 0
    # the tile-stream measurement: misaligned pool, missing rows or checksum; no tiles is fine
    assert L.pkv_stream_tiles(24, 16, ctypes.byref(desc), 16, 4, 16, None) == 1
    assert L.pkv_stream_tiles(16, 16, ctypes.byref(desc), None, 4, 16, None) == 1
    assert L.pkv_stream_tiles(16, 16, ctypes.byref(desc), 16, 4, None, None) == 1
    assert L.pkv_stream_tiles(16, 16, ctypes.byref(desc), 16, 0, 16, None) == 0
    # prefill: (out, q, q_dtype, cu_q_lens, q_start_pos, num_chunks, total_q, max_q_len, num_heads,
    #          k, v, desc, tables, max_blocks_per_seq, scale, stream)
    assert L.pkv_paged_prefill_chunk(16, 16, 1, 16, 16, 1, 8, 8, 6, 16, 16, ctypes.byref(desc), 16, 8, 0.1,
                                     None) == 1                               # bad GQA split
    assert L.pkv_paged_prefill_chunk(16, 16, 1, 16, 16, 1, 8, 8, 8, 16, 16, ctypes.byref(d96), 16, 8, 0.1,
                                     None) == 2                               # head_dim 96
    assert L.pkv_paged_prefill_chunk(16, 16, 0, 16, 16, 1, 8, 8, 8, 16, 16, ctypes.byref(desc), 16, 8, 0.1,
                                     None) == 2                               # f16 q over a bf16 cache
    assert L.pkv_paged_prefill_chunk(16, 16, 1, 16, 16, 1, 8, 8, 8, 16, 16, ctypes.byref(desc), 16, 1 << 27, 0.1,
                                     None) == 2                               # table width x block_size >= 2^31
    assert L.pkv_paged_prefill_chunk(16, 16, 1, 16, 16, 1, 8, 8, 8, 16, 16, ctypes.byref(desc), 16, 8, 0.0,
                                     None) == 1                               # scale must be positive
    assert L.pkv_paged_prefill_chunk(16, 16, 1, 16, 16, 0, 0, 0, 8, 16, 16, ctypes.byref(desc), 16, 8, 0.1,
                                     None) == 0                               # nothing to do
    # the bounded-wait diagnostic takes a limit in (0, 1 s]
    assert L.pkv_check_bounded_wait(0, None) == 1
    assert L.pkv_check_bounded_wait(2_000_000_000, None) == 1


def test_noalloc_decode_returns_the_same_status_as_the_workspace_call():
    """Invalid arguments give the same status from pkv_paged_decode_noalloc as from
    pkv_paged_decode (both run the same host checks before anything else); nothing here
    reaches the GPU."""
    import paged_kv_cache_160_gb300 as pkv
    from paged_kv_cache_160_gb300._binding import CacheDesc
    L = pkv.lib
    good = CacheDesc(64, 4, 16, 128, 1, None, None)
    cases = [
        # (description, out, q, q_dtype, num_seqs, num_heads, k, v, desc, tables, max_blocks, lens, max_len, part)
        ("null out", None, 16, 1, 4, 8, 16, 16, good, 16, 8, 16, 128, 0),
        ("null q", 16, None, 1, 4, 8, 16, 16, good, 16, 8, 16, 128, 0),
        ("null lengths", 16, 16, 1, 4, 8, 16, 16, good, 16, 8, None, 128, 0),
        ("misaligned k", 16, 16, 1, 4, 8, 24, 16, good, 16, 8, 16, 128, 0),
        ("bad GQA split", 16, 16, 1, 4, 6, 16, 16, good, 16, 8, 16, 128, 0),
        ("group above 8", 16, 16, 1, 4, 36, 16, 16, good, 16, 8, 16, 128, 0),
        ("block size 8", 16, 16, 1, 4, 8, 16, 16, CacheDesc(64, 4, 8, 128, 1, None, None), 16, 8, 16, 128, 0),
        ("head_dim 96", 16, 16, 1, 4, 8, 16, 16, CacheDesc(64, 4, 16, 96, 1, None, None), 16, 8, 16, 128, 0),
        ("partition 24", 16, 16, 1, 4, 8, 16, 16, good, 16, 8, 16, 128, 24),
        ("q dtype e4m3", 16, 16, 2, 4, 8, 16, 16, good, 16, 8, 16, 128, 0),
        ("negative seqs", 16, 16, 1, -1, 8, 16, 16, good, 16, 8, 16, 128, 0),
        ("no table columns", 16, 16, 1, 4, 8, 16, 16, good, 16, 0, 16, 128, 0),
        ("e4m3 without scales", 16, 16, 1, 4, 8, 16, 16, CacheDesc(64, 4, 16, 128, 2, None, None), 16, 8, 16,
         128, 0),
        ("tile count past 2^31", 16, 16, 1, 65536, 8, 16, 16, good, 16, 8192, 16, 131072, 0),
        ("nothing to do", 16, 16, 1, 0, 8, 16, 16, good, 16, 8, 16, 128, 0),
    ]
    for name, out, q, qd, S, H, k, v, d, tb, mb, ln, ml, part in cases:
        a = L.pkv_paged_decode(out, q, qd, S, H, k, v, ctypes.byref(d), tb, mb, ln, ml, 0.1, part, 16, 1 << 30,
                               None)
        b = L.pkv_paged_decode_noalloc(out, q, qd, S, H, k, v, ctypes.byref(d), tb, mb, ln, ml, 0.1, part, None)
        assert a == b, (name, a, b)
        assert (a == 0) == (name == "nothing to do"), (name, a)


# ---------------------------------------------------------------------------------------
# block manager: pins and parity with the oracle model
# ---------------------------------------------------------------------------------------

def test_capacity_model_printed_output(golden_dir):
    from paged_kv_cache_160_gb300 import BlockManager, NoBlocksError
    fx = json.load(open(os.path.join(golden_dir, "capacity_model.json")))
    bm = BlockManager(fx["pool_blocks"], fx["block_size"])
    n = 0
    for i, L in enumerate(fx["lens"]):
        try:
            bm.allocate(i, L)
        except NoBlocksError:
            break
        n += 1
    assert n == fx["expected"]["paged_admitted"]
    assert fx["pool_blocks"] - bm.num_free() == fx["expected"]["paged_used_blocks"]


def test_lecture33_figure_and_cow(golden_dir):
    from paged_kv_cache_160_gb300 import BlockManager
    fx = json.load(open(os.path.join(golden_dir, "block_table_diagrams.json")))["lecture33_figure"]
    bm = BlockManager(fx["num_blocks"], fx["block_size"])
    bm.import_seq(0, [7, 2, 5], 10)
    bm.import_seq(1, [7, 9], 6)
    for b, r in fx["ref_cnt"].items():
        assert bm.ref_cnt(int(b)) == r
    # fork B, then the child writes into the shared, half-full block 9 -> copy-on-write
    bm.fork(1, 2)
    assert bm.ref_cnt(9) == 2 and bm.ref_cnt(7) == 3
    slot, cow = bm.append_slot(2)
    assert cow is not None and cow[0] == 9
    assert bm.ref_cnt(9) == 1 and bm.ref_cnt(cow[1]) == 1
    assert slot == cow[1] * 4 + 2


def test_step_decode_is_all_or_nothing():
    from paged_kv_cache_160_gb300 import BlockManager, NoBlocksError
    bm = BlockManager(3, 16)
    bm.allocate(0, 16)
    bm.allocate(1, 16)
    before = bm.free_queue()
    with pytest.raises(NoBlocksError):          # both sequences need a new block, only one is free
        bm.step_decode([0, 1], 4)
    assert bm.free_queue() == before and bm.export([0, 1], 4)[1] == [16, 16]


def _random_ops(seed, n_ops=3000, nb=300, bs=16):
    rng = np.random.default_rng(seed)
    ops = []
    live, nxt = [], 0
    for _ in range(n_ops):
        r = rng.random()
        if live and r > 0.93:                   # preemption by swapping, and the way back
            ops.append(("swap_out" if r < 0.965 else "swap_in", int(rng.choice(live))))
            continue
        if r < 0.2 or not live:
            ops.append(("allocate", nxt, int(rng.integers(0, 120)))); live.append(nxt); nxt += 1
        elif r < 0.55:
            ops.append(("append_slot", int(rng.choice(live))))
        elif r < 0.65:
            ops.append(("append_slots", int(rng.choice(live)), int(rng.integers(1, 40))))
        elif r < 0.75:
            ops.append(("fork", int(rng.choice(live)), nxt)); live.append(nxt); nxt += 1
        elif r < 0.85:
            k = int(rng.integers(1, min(8, len(live)) + 1))
            ops.append(("step_decode", [int(x) for x in rng.choice(live, size=k, replace=False)]))
        else:
            s = int(rng.choice(live)); ops.append(("free", s)); live.remove(s)
    return ops


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_block_manager_matches_oracle_model(seed):
    from oracle.block_manager import BlockManagerModel, NoBlocks
    from paged_kv_cache_160_gb300 import BlockManager, NoBlocksError
    nb, bs, mb, nh = 300, 16, 64, 200
    model, prod = BlockManagerModel(nb, bs), BlockManager(nb, bs)
    model.set_host_pool(nh)
    prod.set_host_pool(nh)
    live = set()
    for op in _random_ops(seed, nb=nb, bs=bs):
        kind = op[0]
        if kind == "step_decode":
            seqs = [s for s in op[1] if s in live and not model.swapped.get(s)]
            if not seqs:
                continue
            # the model has no batch call: all-or-nothing on the number of blocks needed
            try:
                got = prod.step_decode(seqs, mb)
            except NoBlocksError:
                got = None
            if got is None:
                continue
            slots, cows = [], []
            for s in seqs:
                sl, c = model.append_slot(s)
                slots.append(sl)
                if c is not None:
                    cows.append(c)
            tables, lens = model.export(seqs, mb)
            assert got == (slots, cows, tables, lens)
            continue
        if kind in ("append_slot", "append_slots", "free", "fork", "swap_out", "swap_in") and op[1] not in live:
            continue
        if kind in ("append_slot", "append_slots", "fork", "swap_out") and model.swapped.get(op[1]):
            continue
        if kind == "swap_in" and not model.swapped.get(op[1]):
            continue
        res = {}
        for name, side in (("m", model), ("p", prod)):
            try:
                if kind == "allocate":
                    side.allocate(op[1], op[2]); res[name] = "ok"
                elif kind == "append_slot":
                    res[name] = side.append_slot(op[1])
                elif kind == "append_slots":
                    res[name] = side.append_slots(op[1], op[2])
                elif kind == "fork":
                    side.fork(op[1], op[2]); res[name] = "ok"
                elif kind == "free":
                    side.free(op[1]); res[name] = "ok"
                elif kind == "swap_out":
                    res[name] = side.swap_out(op[1])
                elif kind == "swap_in":
                    res[name] = side.swap_in(op[1])
            except (NoBlocks, NoBlocksError):
                res[name] = "noblocks"
        assert res["m"] == res["p"], op
        if res["p"] == "ok":
            if kind == "allocate":
                live.add(op[1])
            elif kind == "fork":
                live.add(op[2])
            elif kind == "free":
                live.discard(op[1])
        assert prod.num_free() == model.num_free()
        assert prod.num_free_host() == len(model.host_free)
    assert prod.free_queue() == list(model.free_queue)
    assert all(prod.is_swapped(s) == int(bool(model.swapped.get(s))) for s in live)
    assert [prod.ref_cnt(b) for b in range(nb)] == model.ref_cnt
    seqs = sorted(s for s in live if not model.swapped.get(s))
    assert prod.export(seqs, mb) == model.export(seqs, mb)


def test_swap_out_and_in_follow_the_preemption_steps():
    """Lecture 33 §5.2: the victim's blocks go to host memory, its device blocks return to
    the pool for others, and later it comes back into fresh device blocks."""
    from paged_kv_cache_160_gb300 import BlockManager, NoBlocksError, PkvError
    bm = BlockManager(8, 4)
    bm.set_host_pool(3)
    bm.allocate(0, 10)                           # blocks 0, 1, 2
    bm.allocate(1, 4)                            # block 3
    bm.fork(1, 2)                                # block 3 shared by 1 and 2
    assert bm.swap_out(0) == [(0, 0), (1, 1), (2, 2)]
    assert bm.free_queue() == [4, 5, 6, 7, 0, 1, 2] and bm.num_free_host() == 0
    with pytest.raises(PkvError):                # a swapped sequence neither appends nor exports
        bm.append_slot(0)
    with pytest.raises(PkvError):
        bm.export([0], 4)
    with pytest.raises(NoBlocksError):           # the host pool is full
        bm.swap_out(1)
    bm.allocate(3, 16)                           # reuses 4, 5, 6, 7
    with pytest.raises(NoBlocksError):           # needs 4 device blocks, only 0, 1, 2 are free
        bm.allocate(4, 13)
    assert bm.swap_in(0) == [(0, 0), (1, 1), (2, 2)]
    assert bm.export([0], 4) == ([[0, 1, 2, -1]], [10]) and bm.num_free_host() == 3
    bm.free(3)
    assert bm.swap_out(2) == [(3, 0)]            # shared block: stays for sequence 1, copied for 2
    assert bm.ref_cnt(3) == 1
    assert bm.swap_in(2) == [(0, 4)]
    assert bm.export([1, 2], 2) == ([[3, -1], [4, -1]], [4, 4])


def test_synthetic_plans_agree_on_both_sides():
    """The tiny workload's step: copy-on-write for sequence 0, a new block for sequence 3."""
    import synth
    from tests.harness import oracle_plan, product_plan
    case = synth.tiny_config()
    po, pp = oracle_plan(case), product_plan(case)
    assert po == pp
    assert len(pp.cows) == 1 and pp.cows[0][0] == case.seq_blocks[0][0]
    assert pp.lens == [11, 7, 38, 17]
    assert pp.tables[3][0] == case.seq_blocks[3][0] != pp.tables[0][0]
    # sequence 2's new token is token 37: logical block 2, offset 5 (the worked example)
    assert pp.slots[2] == case.seq_blocks[2][2] * 16 + 5
