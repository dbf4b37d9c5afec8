"""Pins of the swapping path of the oracle (Lecture 33 §5.2: a preempted sequence's blocks
go to host memory, its device blocks serve others, and it later resumes from fresh device
blocks).  The decode output of the sequence must be the same, bit for bit, before the swap
and after the round trip, whatever the freed blocks held meanwhile; every block the swap
does not name keeps its bytes."""
import numpy as np
import pytest

from oracle import cache_ops, paged_attention as pa
from oracle.block_manager import BlockManagerModel, NoBlocks


def _pool(rng, nb, hkv, bs, d):
    return (rng.integers(0, 1 << 16, size=(nb, hkv, bs, d), dtype=np.uint16) & 0x3BFF,   # finite f16 codes
            rng.integers(0, 1 << 16, size=(nb, hkv, bs, d), dtype=np.uint16) & 0x3BFF)


def test_swap_round_trip_preserves_the_sequence_and_nothing_else():
    rng = np.random.default_rng(11)
    nb, nh, hkv, bs, d, hq = 12, 6, 2, 4, 8, 4
    k, v = _pool(rng, nb, hkv, bs, d)
    hk, hv = _pool(rng, nh, hkv, bs, d)                # host pool starts with junk
    bm = BlockManagerModel(nb, bs)
    bm.set_host_pool(nh)
    bm.allocate(0, 9)                                  # 3 blocks
    bm.allocate(1, 6)
    q = rng.standard_normal((1, hq, d))
    tab, lens = bm.export([0], 3)
    before = pa.decode_attention(q, k, v, "f16", tab, lens, 0.35)

    out_pairs = bm.swap_out(0)
    assert [dv for dv, _ in out_pairs] == tab[0]
    hk2, hv2 = cache_ops.swap_blocks(hk, hv, k, v, out_pairs)
    named = {h for _, h in out_pairs}
    for b in range(nh):                                # only the named host blocks change
        if b not in named:
            assert np.array_equal(hk2[b], hk[b]) and np.array_equal(hv2[b], hv[b])
    # others reuse the freed device blocks and overwrite them
    bm.allocate(2, 4 * bm.num_free())
    tab2, _ = bm.export([2], 16)
    slots = [tab2[0][j // bs] * bs + j % bs for j in range(4 * len([x for x in tab2[0] if x >= 0]))]
    kn, vn = _pool(rng, len(slots), hkv, 1, d)
    k, v = cache_ops.kv_write(k, v, kn[:, :, 0, :], vn[:, :, 0, :], slots)
    bm.free(2)

    in_pairs = bm.swap_in(0)
    assert [h for h, _ in in_pairs] == [h for _, h in out_pairs]
    k3, v3 = cache_ops.swap_blocks(k, v, hk2, hv2, in_pairs)
    dst = {dv for _, dv in in_pairs}
    for b in range(nb):
        if b not in dst:
            assert np.array_equal(k3[b], k[b]) and np.array_equal(v3[b], v[b])
    tab3, lens3 = bm.export([0], 3)
    after = pa.decode_attention(q, k3, v3, "f16", tab3, lens3, 0.35)
    assert lens3 == lens and np.array_equal(after, before)


def test_swap_needs_room_on_both_sides():
    bm = BlockManagerModel(4, 2)
    bm.set_host_pool(1)
    bm.allocate(0, 3)
    with pytest.raises(NoBlocks):
        bm.swap_out(0)                                 # 2 blocks, 1 host block
    assert bm.num_free() == 2 and not bm.swapped.get(0)
    bm.set_host_pool(2)
    bm.swap_out(0)
    bm.allocate(1, 7)                                  # takes all 4 device blocks
    with pytest.raises(NoBlocks):
        bm.swap_in(0)
    bm.free(1)
    assert [dv for _, dv in bm.swap_in(0)] == [2, 3]   # the free queue after the swap-out was 2, 3, 0, 1
