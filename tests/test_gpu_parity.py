"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Caches, tables, slots and copy-on-write pairs must match bit for bit; attention
outputs must be within the stated max-abs tolerance of the float64 oracle
(fp16 2e-3, bf16 1e-2, e4m3 KV 3e-2) after the GPU's rounding to the query dtype.
"""
import math

import numpy as np
import pytest
import torch

import synth
from tests.harness import (TOL, codes, device_run, max_abs_err, oracle_plan, oracle_run, product_plan)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import paged_kv_cache_160_gb300  # noqa: F401  (fails loudly if the library is missing)


def _check_case(case, partition_size=None, decode_rows=None, prefill_rows=None, prefill_heads=None,
                compare_caches=True, run_prefill=True):
    po, pp = oracle_plan(case), product_plan(case)
    assert pp == po, "block manager plans differ"
    dev = device_run(case, pp, partition_size=partition_size, keep_intermediate=compare_caches,
                     run_prefill=run_prefill)
    ref = oracle_run(case, po, decode_rows=decode_rows, prefill_rows=prefill_rows, prefill_heads=prefill_heads)
    assert dev.device_error == 0, f"device error word {dev.device_error:#x}"
    if compare_caches:
        assert np.array_equal(codes(dev.k_cache), ref.k_cache), "K cache differs after copy/write"
        assert np.array_equal(codes(dev.v_cache), ref.v_cache), "V cache differs after copy/write"
        assert np.array_equal(codes(dev.k_final), ref.k_final)
        assert np.array_equal(codes(dev.v_final), ref.v_final)
    tol = TOL[case.kv_dtype]
    err = max_abs_err(dev.decode, ref.decode)
    assert err <= tol, f"decode max abs err {err:.3e} > {tol}"
    if case.chunk is not None and dev.prefill is not None:
        perr = max_abs_err(dev.prefill, ref.prefill)
        assert perr <= tol, f"prefill max abs err {perr:.3e} > {tol}"
    return dev, ref, err


# ---------------------------------------------------------------------------------------
# the five workloads at full size
# ---------------------------------------------------------------------------------------

def test_tiny_with_copy_on_write():
    case = synth.tiny_config()
    dev, ref, _ = _check_case(case)
    # sequence 3 shares sequence 0's first block; sequence 0's write goes to a private copy,
    # so sequence 3's output must equal a run in which sequence 0 writes nothing.
    import copy
    plan2 = copy.deepcopy(product_plan(case))
    plan2.slots[0] = -1                                     # padding: sequence 0 writes nothing
    plan2.cows = []
    plan2.tables[0][0] = case.seq_blocks[0][0]
    dev2 = device_run(case, plan2)
    assert torch.equal(dev.decode[3], dev2.decode[3])


@pytest.mark.parametrize("part", [0, 512, 16])
def test_qwen7b_gqa_full(part):
    case = synth.qwen7b_gqa_config()
    _check_case(case, partition_size=part)


def test_mha13b_full_sampled():
    case = synth.mha13b_config()
    heads = [0, 17, 39]
    rows = [(i, h) for i in range(case.num_seqs) for h in heads]
    dev, ref, _ = _check_case(case, decode_rows=rows)
    # sequences sharing the 1024-token prefix read the same physical blocks
    sh = case.meta["sharers"]
    assert len(sh) == 64


@pytest.mark.parametrize("part", [512, 0])
def test_long_splitkv_e4m3_sampled(part):
    case = synth.long_splitkv_config()
    rows = [(i, h) for i in range(case.num_seqs) for h in (0, 13, 31)]
    _check_case(case, partition_size=part, decode_rows=rows, compare_caches=False)


def test_mixed_step_decode_and_copies():
    case = synth.mixed_config()
    _check_case(case, prefill_rows=[0, 1, 255, 511], prefill_heads=[0, 6, 27])


# ---------------------------------------------------------------------------------------
# small cases spanning several tiles, ragged tails and edge cases
# ---------------------------------------------------------------------------------------

SMALL = [
    # name, lens, Hq, Hkv, D, q dtype, kv dtype, partition
    ("mha_f16_d64", [1, 15, 16, 17, 31, 33, 200], 4, 4, 64, "f16", "f16", 0),
    ("gqa7_bf16", [5, 16, 100, 257, 1000], 28, 4, 128, "bf16", "bf16", 0),
    ("gqa8_bf16_d64", [3, 48, 49, 300], 16, 2, 64, "bf16", "bf16", 32),
    ("gqa3_f16", [2, 64, 65, 129], 6, 2, 128, "f16", "f16", 64),
    ("e4m3_bf16q", [1, 17, 511, 512, 513, 2000], 32, 8, 128, "bf16", "e4m3", 512),
    ("e4m3_f16q_balanced", [7, 16, 130, 900], 8, 2, 128, "f16", "e4m3", 0),
    # six workers in one CTA merge sixteen (segment, head) items
    ("few_workers_gqa8", [80, 80], 8, 1, 128, "bf16", "bf16", 32),
    ("gqa5_many_seqs", [int(x) for x in np.random.default_rng(5).integers(1, 80, size=300)], 10, 2, 128,
     "bf16", "bf16", 0),
]


@pytest.mark.parametrize("name,lens,hq,hkv,d,qd,kd,part", SMALL, ids=[s[0] for s in SMALL])
def test_small_cases(name, lens, hq, hkv, d, qd, kd, part):
    case = synth.make_decode_case(name, 77, lens, hq, hkv, d, qd, kd, partition_size=part)
    _check_case(case)


def test_very_large_batch_takes_the_four_warp_layout():
    """4500 sequences: the per-sequence prefix arrays no longer fit beside twelve warps'
    stages, so the kernel runs with four worker warps per CTA; sampled rows vs the oracle."""
    rng = np.random.default_rng(6)
    lens = [int(x) for x in rng.integers(1, 40, size=4500)]
    case = synth.make_decode_case("huge_batch", 82, lens, 4, 1, 128, "bf16", "bf16")
    rows = sorted({(int(s), int(h)) for s, h in zip(rng.integers(0, 4500, 300), rng.integers(0, 4, 300))})
    _check_case(case, decode_rows=rows, compare_caches=False)


BS32 = [
    # 32-token blocks: each is two 16-row tiles.  Lengths straddle tile and block edges;
    # a 48-token partition ends inside a block.
    ("bs32_gqa7_bf16", [1, 16, 17, 31, 32, 33, 100, 700], 28, 4, 128, "bf16", "bf16", 0),
    ("bs32_e4m3_part512", [5, 511, 512, 513, 1500], 32, 8, 128, "bf16", "e4m3", 512),
    ("bs32_f16_d64_part48", [3, 47, 48, 49, 250], 8, 2, 64, "f16", "f16", 48),
]


@pytest.mark.parametrize("name,lens,hq,hkv,d,qd,kd,part", BS32, ids=[s[0] for s in BS32])
def test_block_size_32(name, lens, hq, hkv, d, qd, kd, part):
    case = synth.make_decode_case(name, 83, lens, hq, hkv, d, qd, kd, block_size=32, partition_size=part,
                                  unused_fill="nan")
    _check_case(case)


def _random_decode_shape(seed):
    """A seeded random decode configuration within the supported envelope."""
    rng = np.random.default_rng(seed)
    kd = ["f16", "bf16", "e4m3"][seed % 3]
    d = 128 if kd == "e4m3" else int(rng.choice([64, 128]))
    qd = "bf16" if kd == "bf16" else ("f16" if kd == "f16" else str(rng.choice(["f16", "bf16"])))
    hkv = int(rng.integers(1, 5))
    g = int(rng.integers(1, 9))
    bs = int(rng.choice([16, 32]))
    n = int(rng.integers(1, 40))
    lens = [int(x) for x in rng.integers(0, 1500, n)]
    lens[int(rng.integers(0, n))] = int(rng.integers(1, 3))             # a very short one
    part = int(rng.choice([0, 0, 16, 48, 256]))
    return f"rand{seed}", lens, g * hkv, hkv, d, qd, kd, part, bs


@pytest.mark.parametrize("seed", range(12))
def test_random_shapes(seed):
    """Random group sizes, head dims, dtypes, splits, block sizes and ragged lengths (some
    sequences may be empty), with NaN in every unused pool row."""
    name, lens, hq, hkv, d, qd, kd, part, bs = _random_decode_shape(seed)
    case = synth.make_decode_case(name, 900 + seed, lens, hq, hkv, d, qd, kd, block_size=bs, partition_size=part,
                                  unused_fill="nan")
    _check_case(case)


@pytest.mark.parametrize("kd", ["bf16", "e4m3"])
def test_unused_slots_hold_nan(kd):
    """Rows past each sequence's end hold NaN; they must never reach the output."""
    qd = "bf16"
    case = synth.make_decode_case("nan_tail", 78, [1, 7, 16, 33, 250], 8, 2, 128, qd, kd, unused_fill="nan",
                                  partition_size=0 if kd == "bf16" else 32)
    _check_case(case)


def test_empty_sequences_give_zeros():
    case = synth.make_decode_case("empty", 79, [0, 40, 0, 3], 8, 8, 64, "f16", "f16", write=False)
    dev, ref, _ = _check_case(case)
    assert torch.count_nonzero(dev.decode[0]) == 0 and torch.count_nonzero(dev.decode[2]) == 0


def test_all_empty():
    case = synth.make_decode_case("all_empty", 80, [0, 0], 4, 4, 64, "f16", "f16", write=False)
    dev, _, _ = _check_case(case)
    assert torch.count_nonzero(dev.decode) == 0


def test_workspace_needs_no_init_and_repeat_is_deterministic():
    import paged_kv_cache_160_gb300 as pkv
    case = synth.qwen7b_gqa_config()
    plan = product_plan(case)
    dev = torch.device("cuda")
    kc, vc = case.k_cache.to(dev), case.v_cache.to(dev)
    desc = pkv.cache_desc(kc)
    q = case.q.to(dev)
    tables = torch.tensor(plan.tables, dtype=torch.int32, device=dev)
    lens = torch.tensor(plan.lens, dtype=torch.int32, device=dev)
    outs = []
    for part in (0, 0, 0, 512):
        ws_bytes = pkv.pkv_decode_workspace_bytes(case.num_seqs, 28, 4, 128, 16, max(plan.lens), part)
        ws = torch.full((ws_bytes,), 0xFF, dtype=torch.uint8, device=dev)     # garbage, not zeros
        out = torch.empty_like(q)
        pkv.pkv_paged_decode(out, q, kc, vc, desc, tables, lens, max(plan.lens), case.scale, part, ws)
        outs.append(out)
        out2 = torch.empty_like(q)                                            # the same workspace again
        pkv.pkv_paged_decode(out2, q, kc, vc, desc, tables, lens, max(plan.lens), case.scale, part, ws)
        torch.cuda.synchronize()
        assert torch.equal(out2, out)
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])
    assert (outs[3].float() - outs[0].float()).abs().max().item() < 2e-2
    assert pkv.pkv_get_device_error() == 0


def test_a_wait_that_runs_out_reports_a_timeout_and_the_context_survives():
    """The bounded wait every kernel uses, on a barrier nothing arrives on: after 2 ms it
    gives up, sets the timeout bit, and later calls on the same context still work."""
    import time
    import paged_kv_cache_160_gb300 as pkv
    pkv.pkv_get_device_error()
    t0 = time.perf_counter()
    pkv.pkv_check_bounded_wait(2_000_000)
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 1.0
    assert pkv.pkv_get_device_error() == pkv.DEVERR["timeout"]
    assert pkv.pkv_get_device_error() == 0                  # reading clears the word
    case = synth.make_decode_case("after_timeout", 84, [5, 40], 4, 2, 64, "f16", "f16")
    _check_case(case)


def test_device_checks_flag_bad_tables_without_faulting():
    import paged_kv_cache_160_gb300 as pkv
    case = synth.make_decode_case("bad", 81, [40, 40], 4, 4, 64, "f16", "f16", write=False)
    dev = torch.device("cuda")
    kc, vc = case.k_cache.to(dev), case.v_cache.to(dev)
    desc = pkv.cache_desc(kc)
    q = case.q.to(dev)
    tables = torch.tensor([b + [-1] for b in case.seq_blocks], dtype=torch.int32, device=dev)
    tables[1, 1] = case.num_blocks + 5                     # a block id outside the pool
    lens = torch.tensor([40, 40], dtype=torch.int32, device=dev)
    ws = torch.zeros(pkv.pkv_decode_workspace_bytes(2, 4, 4, 64, 16, 64, 0), dtype=torch.uint8, device=dev)
    out = torch.empty_like(q)
    pkv.pkv_get_device_error()
    pkv.pkv_paged_decode(out, q, kc, vc, desc, tables, lens, 64, case.scale, 0, ws)
    assert pkv.pkv_get_device_error() & pkv.DEVERR["block_id"]
    lens[0] = 4 * 16 + 1                                   # longer than the block table allows
    pkv.pkv_paged_decode(out, q, kc, vc, desc, tables, lens, 80, case.scale, 0, ws)
    assert pkv.pkv_get_device_error() & pkv.DEVERR["context_len"]
    # a slot beyond the pool and a chaining copy pair are skipped and flagged
    slots = torch.tensor([case.num_blocks * 16 + 3], dtype=torch.int64, device=dev)
    kn = torch.zeros((1, 4, 64), dtype=torch.float16, device=dev)
    before = kc.clone()
    pkv.pkv_kv_write(kn, kn, slots, kc, vc, desc)
    assert pkv.pkv_get_device_error() & pkv.DEVERR["slot"]
    pkv.pkv_copy_blocks(kc, vc, desc, torch.tensor([[1, 2], [2, 3]], dtype=torch.int32, device=dev))
    assert pkv.pkv_get_device_error() & pkv.DEVERR["copy_pair"]
    assert torch.equal(kc[2], before[2])                   # (1, 2) skipped: its dst is a src
    assert torch.equal(kc[3], before[2])                   # (2, 3) is valid and applied
    # the context is still usable
    pkv.pkv_paged_decode(out, q, kc, vc, desc, torch.tensor([b + [-1] for b in case.seq_blocks],
                         dtype=torch.int32, device=dev), torch.tensor([40, 40], dtype=torch.int32, device=dev),
                         64, case.scale, 0, ws)
    assert pkv.pkv_get_device_error() == 0


def test_kv_write_quantises_to_e4m3_like_the_oracle():
    """f16/bf16 rows into an e4m3 cache: x / scale in fp32, then round-to-nearest-even."""
    import paged_kv_cache_160_gb300 as pkv
    from oracle.formats import encode_e4m3
    g = torch.Generator().manual_seed(82)
    T, H, D, NB = 64, 4, 128, 16
    for src_dt in (torch.bfloat16, torch.float16):
        x_k = (torch.randn((T, H, D), generator=g) * 3).to(src_dt)
        x_v = (torch.randn((T, H, D), generator=g) * 100).to(src_dt)
        x_k[0, 0, :4] = torch.tensor([1e4, -1e4, 0.0, -0.0]).to(src_dt)
        ks = torch.empty(H).uniform_(0.5, 2.0, generator=g)
        vs = torch.empty(H).uniform_(0.5, 2.0, generator=g)
        slots = torch.randperm(NB * 16, generator=g)[:T].to(torch.int64)
        dev = torch.device("cuda")
        kc = torch.zeros((NB, H, 16, D), dtype=torch.uint8, device=dev)
        vc = torch.zeros_like(kc)
        desc = pkv.cache_desc(kc, ks.to(dev), vs.to(dev))
        pkv.pkv_kv_write(x_k.to(dev), x_v.to(dev), slots.to(dev), kc, vc, desc)
        assert pkv.pkv_get_device_error() == 0
        for x, sc, cache in ((x_k, ks, kc), (x_v, vs, vc)):
            q32 = (x.to(torch.float32) / sc.view(1, H, 1)).numpy()     # fp32 quotient, as the kernel
            want = encode_e4m3(q32.astype(np.float64))
            got = cache.cpu().numpy()
            for t, s in enumerate(slots.tolist()):
                assert np.array_equal(got[s // 16, :, s % 16, :], want[t])
