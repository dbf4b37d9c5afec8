"""GPU parity of the fused append + decode call (pkv_paged_decode_append).

The oracle side is the unfused step: kv_write of each sequence's new row at its last
position, then decode.  Caches must match it bit for bit, outputs within the dtype's
tolerance; the fused and unfused device paths must agree exactly.
"""
import numpy as np
import pytest
import torch

import synth
from tests.harness import TOL, append_slots, codes, device_run, max_abs_err, oracle_plan, oracle_run, product_plan
from tests.test_gpu_parity import BS32, SMALL, _random_decode_shape

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import paged_kv_cache_160_gb300  # noqa: F401


def _check_fused(case, partition_size=None, decode_rows=None, append_inputs=None, compare_unfused=True):
    po, pp = oracle_plan(case), product_plan(case)
    assert pp == po
    assert append_slots(case, pp) == list(pp.slots)
    dev = device_run(case, pp, partition_size=partition_size, fused_append=True, append_inputs=append_inputs)
    ref = oracle_run(case, po, decode_rows=decode_rows)
    assert dev.device_error == 0, f"device error word {dev.device_error:#x}"
    assert np.array_equal(codes(dev.k_cache), ref.k_cache), "K cache differs from kv_write"
    assert np.array_equal(codes(dev.v_cache), ref.v_cache), "V cache differs from kv_write"
    err = max_abs_err(dev.decode, ref.decode)
    assert err <= TOL[case.kv_dtype], f"decode max abs err {err:.3e}"
    if compare_unfused and append_inputs is None:
        un = device_run(case, pp, partition_size=partition_size)
        # bit patterns (unused pool rows may hold NaN)
        assert np.array_equal(codes(un.k_cache), codes(dev.k_cache))
        assert np.array_equal(codes(un.v_cache), codes(dev.v_cache))
        assert torch.equal(un.decode, dev.decode), "fused and unfused outputs differ"
    return dev, ref


def test_tiny_with_copy_on_write():
    _check_fused(synth.tiny_config())


@pytest.mark.parametrize("part", [0, 512])
def test_qwen7b_gqa_full(part):
    _check_fused(synth.qwen7b_gqa_config(), partition_size=part)


def test_mha13b_sampled():
    case = synth.mha13b_config()
    rows = [(i, h) for i in range(case.num_seqs) for h in (0, 21, 39)]
    _check_fused(case, decode_rows=rows, compare_unfused=False)


_WRITE_SMALL = [s for s in SMALL if s[6] != "e4m3"]


@pytest.mark.parametrize("name,lens,hq,hkv,d,qd,kd,part", _WRITE_SMALL, ids=[s[0] for s in _WRITE_SMALL])
def test_small_cases(name, lens, hq, hkv, d, qd, kd, part):
    _check_fused(synth.make_decode_case(name, 177, lens, hq, hkv, d, qd, kd, partition_size=part,
                                        unused_fill="nan"))


_BS32 = [s for s in BS32 if s[6] != "e4m3"]


@pytest.mark.parametrize("name,lens,hq,hkv,d,qd,kd,part", _BS32, ids=[s[0] for s in _BS32])
def test_block_size_32(name, lens, hq, hkv, d, qd, kd, part):
    _check_fused(synth.make_decode_case(name, 183, lens, hq, hkv, d, qd, kd, block_size=32, partition_size=part,
                                        unused_fill="nan"))


def _e4m3_case(name, seed, lens, hq, hkv, qd, bs, part):
    """An e4m3 cache whose new rows arrive as f16/bf16: the oracle writes the codes of the
    fp32 quotient x / scale (round to nearest even, saturating), as pkv_kv_write does."""
    from oracle.formats import encode_e4m3
    case = synth.make_decode_case(name, seed, lens, hq, hkv, 128, qd, "e4m3", block_size=bs, partition_size=part,
                                  unused_fill="nan")
    g = torch.Generator().manual_seed(seed + 1)
    tdt = torch.bfloat16 if qd == "bf16" else torch.float16
    xs = []
    for which, sc in (("k", case.k_scale), ("v", case.v_scale)):
        x = (torch.randn((case.num_seqs, hkv, 128), generator=g) * 2).to(tdt)
        if which == "k":
            # saturates to code +-448.  Only in K: a saturated V row would make outputs of
            # magnitude ~900, whose rounding to the q dtype alone exceeds the absolute tolerance.
            x[0, 0, :2] = torch.tensor([1e4, -1e4]).to(tdt)
        q32 = (x.to(torch.float32) / sc.view(1, hkv, 1)).numpy().astype(np.float64)
        xs.append((x, torch.from_numpy(encode_e4m3(q32).astype(np.uint8))))
    case.k_new, case.v_new = xs[0][1], xs[1][1]
    return case, (xs[0][0], xs[1][0])


@pytest.mark.parametrize("qd,bs,part", [("bf16", 16, 512), ("f16", 16, 0), ("bf16", 32, 0), ("f16", 32, 48)])
def test_e4m3_cache_quantises_the_new_rows(qd, bs, part):
    case, xin = _e4m3_case(f"app_e4m3_{qd}_{bs}", 190 + bs, [1, 16, 17, 511, 513, 900], 32, 8, qd, bs, part)
    _check_fused(case, append_inputs=xin)


@pytest.mark.parametrize("seed", range(6))
def test_random_shapes(seed):
    name, lens, hq, hkv, d, qd, kd, part, bs = _random_decode_shape(seed)
    lens = [max(1, L) for L in lens]                                      # every sequence appends
    if kd == "e4m3":
        case, xin = _e4m3_case(name, 950 + seed, lens, hq, hkv, qd, bs, part)
        _check_fused(case, append_inputs=xin)
    else:
        _check_fused(synth.make_decode_case(name, 950 + seed, lens, hq, hkv, d, qd, kd, block_size=bs,
                                            partition_size=part, unused_fill="nan"))


def test_clamped_length_writes_nothing_and_is_flagged():
    import paged_kv_cache_160_gb300 as pkv
    case = synth.make_decode_case("app_clamp", 191, [20, 40], 4, 2, 64, "f16", "f16")
    plan = product_plan(case)
    dev = torch.device("cuda")
    kc, vc = case.k_cache.to(dev), case.v_cache.to(dev)
    k0, v0 = kc.clone(), vc.clone()
    desc = pkv.cache_desc(kc)
    q = case.q.to(dev)
    out = torch.empty_like(q)
    tables = torch.tensor(plan.tables, dtype=torch.int32, device=dev)
    lens = torch.tensor(plan.lens, dtype=torch.int32, device=dev)       # 21 and 41
    ws = torch.zeros(pkv.pkv_decode_workspace_bytes(2, 4, 2, 64, 16, 30, 0), dtype=torch.uint8, device=dev)
    pkv.pkv_get_device_error()
    pkv.pkv_paged_decode_append(out, q, case.k_new.to(dev), case.v_new.to(dev), kc, vc, desc, tables, lens,
                                30, case.scale, 0, ws)
    err = pkv.pkv_get_device_error()
    assert err & pkv.DEVERR["context_len"]
    s0 = append_slots(case, plan)[0]
    ch = (kc != k0).nonzero()
    blk, off = s0 // 16, s0 % 16
    # only sequence 0 (length 21 <= 30) wrote its row
    assert torch.equal(kc[blk, :, off], case.k_new[0].to(dev))
    assert all(int(b) == blk and int(o) == off for b, _, o, _ in ch.tolist())
    assert torch.equal((vc != v0).nonzero()[:, [0, 2]].unique(dim=0).cpu(), torch.tensor([[blk, off]]))


@pytest.mark.parametrize("fused", [True, False])
def test_pinned_host_inputs_and_output_match_device_ones(fused):
    """out, q, new K/V, tables and lengths in pinned host memory are read and written in
    place by the kernels; results are bit-identical to device-resident buffers."""
    import paged_kv_cache_160_gb300 as pkv
    case = synth.make_decode_case("pinned", 193, [1, 15, 16, 17, 300, 1000], 28, 4, 128, "bf16", "bf16")
    plan = product_plan(case)
    dev = torch.device("cuda")
    max_len = max(plan.lens)
    ws = torch.zeros(pkv.pkv_decode_workspace_bytes(case.num_seqs, 28, 4, 128, 16, max_len, 0), dtype=torch.uint8,
                     device=dev)
    tables = torch.tensor(plan.tables, dtype=torch.int32)
    lens = torch.tensor(plan.lens, dtype=torch.int32)
    results = []
    for where in ("device", "pinned"):
        kc, vc = case.k_cache.to(dev), case.v_cache.to(dev)
        desc = pkv.cache_desc(kc)
        if where == "device":
            q, tb, ln, kn, vn = case.q.to(dev), tables.to(dev), lens.to(dev), case.k_new.to(dev), case.v_new.to(dev)
            out = torch.empty(case.q.shape, dtype=case.q.dtype, device=dev)
        else:
            q, tb, ln = case.q.clone().pin_memory(), tables.clone().pin_memory(), lens.clone().pin_memory()
            kn, vn = case.k_new.clone().pin_memory(), case.v_new.clone().pin_memory()
            out = torch.empty(case.q.shape, dtype=case.q.dtype).pin_memory()
        if fused:
            pkv.pkv_paged_decode_append(out, q, kn, vn, kc, vc, desc, tb, ln, max_len, case.scale, 0, ws)
        else:
            pkv.pkv_paged_decode(out, q, kc, vc, desc, tb, ln, max_len, case.scale, 0, ws)
        torch.cuda.synchronize()
        results.append((out.cpu(), kc.cpu(), vc.cpu()))
    assert pkv.pkv_get_device_error() == 0
    assert torch.equal(results[0][0], results[1][0])
    assert torch.isfinite(results[0][0].float()).all()
    assert np.array_equal(codes(results[0][1]), codes(results[1][1]))
    assert np.array_equal(codes(results[0][2]), codes(results[1][2]))


def test_very_large_batch_takes_the_four_warp_layout():
    """4500 sequences (the four-warp layout): fused and unfused agree exactly; sampled rows
    match the oracle."""
    rng = np.random.default_rng(16)
    lens = [int(x) for x in rng.integers(1, 40, size=4500)]
    case = synth.make_decode_case("huge_batch_fused", 182, lens, 4, 1, 128, "bf16", "bf16")
    rows = sorted({(int(s), int(h)) for s, h in zip(rng.integers(0, 4500, 300), rng.integers(0, 4, 300))})
    _check_fused(case, decode_rows=rows)
