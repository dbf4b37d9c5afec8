"""GPU parity of preemption by swapping (Lecture 33 §5.2) through the C ABI.

A sequence's blocks go from the device pool to a pinned host pool with pkv_swap_blocks
(pairs from the host block manager); another sequence then reuses and overwrites the freed
device blocks; the first sequence is swapped back into fresh device blocks.  After every
copy both pools must equal the oracle's byte copies exactly, and the sequence's decode
output must be bit-identical before and after the round trip.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import cache_ops
from oracle.block_manager import BlockManagerModel
from tests.harness import codes

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")


def _pairs(pairs, dev):
    return torch.tensor(pairs, dtype=torch.int32, device=dev).reshape(-1, 2)


@pytest.mark.parametrize("kv", ["bf16", "e4m3"])
def test_swap_round_trip_through_pinned_host_memory(kv):
    import paged_kv_cache_160_gb300 as pkv
    dev = torch.device("cuda")
    nb, nh, hkv, hq, d, bs = 96, 40, 4, 28, 128, 16
    case = synth.make_decode_case("swap", 90, [300, 200, 500], hq, hkv, d, "bf16", kv, num_blocks=nb, write=False)
    k0, v0 = case.k_cache.clone(), case.v_cache.clone()
    kc, vc = k0.to(dev), v0.to(dev)
    ks = case.k_scale.to(dev) if case.k_scale is not None else None
    vs = case.v_scale.to(dev) if case.v_scale is not None else None
    desc = pkv.cache_desc(kc, ks, vs)
    hk = torch.zeros((nh,) + tuple(k0.shape[1:]), dtype=k0.dtype).pin_memory()
    hv = torch.zeros_like(hk).pin_memory()

    bm, model = pkv.BlockManager(nb, bs), BlockManagerModel(nb, bs)
    for side in (bm, model):
        side.set_host_pool(nh)
        for i, blocks in enumerate(case.seq_blocks):
            side.import_seq(i, blocks, case.context_lens[i])
    q = case.q.to(dev)
    mb = max(len(b) for b in case.seq_blocks) + 8

    def decode(seqs):
        tab, lens = bm.export(seqs, mb)
        out = torch.empty((len(seqs), hq, d), dtype=torch.bfloat16, device=dev)
        ws = torch.zeros(pkv.pkv_decode_workspace_bytes(len(seqs), hq, hkv, d, 16, max(lens), 0), dtype=torch.uint8,
                         device=dev)
        pkv.pkv_paged_decode(out, q[seqs], kc, vc, desc, torch.tensor(tab, dtype=torch.int32, device=dev),
                             torch.tensor(lens, dtype=torch.int32, device=dev), max(lens), case.scale, 0, ws)
        return out

    before = decode([2])
    ok, ov = codes(k0), codes(v0)
    ohk, ohv = codes(hk), codes(hv)

    out_pairs = bm.swap_out(2)
    assert out_pairs == model.swap_out(2)
    pkv.pkv_swap_blocks(hk, hv, kc, vc, desc, _pairs(out_pairs, dev))
    torch.cuda.synchronize()
    ohk, ohv = cache_ops.swap_blocks(ohk, ohv, ok, ov, out_pairs)
    assert np.array_equal(codes(hk), ohk) and np.array_equal(codes(hv), ohv)

    # a newcomer takes every free device block (the victim's among them) and overwrites it
    n_free = bm.num_free()
    for side in (bm, model):
        side.allocate(7, n_free * bs)
    tab7, _ = bm.export([7], n_free)
    junk_k = torch.randn((n_free,) + tuple(k0.shape[1:]), generator=torch.Generator().manual_seed(5)).to(k0.dtype) \
        if kv != "e4m3" else torch.randint(0, 0x78, (n_free,) + tuple(k0.shape[1:]), dtype=torch.uint8)
    dst = torch.tensor(tab7[0], dtype=torch.long)
    kc[dst.to(dev)] = junk_k.to(dev)
    vc[dst.to(dev)] = junk_k.to(dev)
    ok, ov = ok.copy(), ov.copy()
    ok[dst.numpy()] = codes(junk_k)
    ov[dst.numpy()] = codes(junk_k)
    for side in (bm, model):
        side.free(7)

    in_pairs = bm.swap_in(2)
    assert in_pairs == model.swap_in(2)
    pkv.pkv_swap_blocks(kc, vc, hk, hv, desc, _pairs(in_pairs, dev))
    torch.cuda.synchronize()
    ok, ov = cache_ops.swap_blocks(ok, ov, ohk, ohv, in_pairs)
    assert np.array_equal(codes(kc.cpu()), ok) and np.array_equal(codes(vc.cpu()), ov)
    after = decode([2])
    assert torch.equal(after, before)
    assert pkv.pkv_get_device_error() == 0


def test_swap_skips_and_flags_bad_pairs():
    import paged_kv_cache_160_gb300 as pkv
    dev = torch.device("cuda")
    k = torch.randn((8, 2, 16, 64)).to(torch.float16)
    kc, vc = k.to(dev), (k + 1).to(dev)
    desc = pkv.cache_desc(kc)
    hk = torch.zeros((4, 2, 16, 64), dtype=torch.float16).pin_memory()
    hv = torch.zeros_like(hk).pin_memory()
    pkv.pkv_get_device_error()
    # (1 -> 0) fine; (2 -> 3) and (5 -> 3) write the same dst; (6 -> 9) dst outside the host pool
    pkv.pkv_swap_blocks(hk, hv, kc, vc, desc, _pairs([(1, 0), (2, 3), (5, 3), (6, 9)], dev))
    torch.cuda.synchronize()
    assert pkv.pkv_get_device_error() == pkv.DEVERR["copy_pair"]
    assert torch.equal(hk[0], k[1]) and torch.equal(hv[0], k[1] + 1)
    assert torch.count_nonzero(hk[1:]) == 0 and torch.count_nonzero(hv[1:]) == 0
