"""GPU parity of paged_prefill_chunk (tcgen05 path) against the fp64 oracle.

Each case builds a paged pool holding, per chunk, a cached prefix followed by the chunk's
own K/V (written on the host by plain indexing), runs the chunks in one launch (varlen
via cu_q_lens) and compares every output row with the oracle's causal chunk attention.
"""
import math

import numpy as np
import pytest
import torch

from tests.harness import TOL, codes, q_f64

pytestmark = pytest.mark.gpu

DT = {"bf16": torch.bfloat16, "f16": torch.float16}


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")


def _case(seed, chunks, hq, hkv, dtype, nan_fill=False, D=128, bs=16):
    g = torch.Generator().manual_seed(seed)
    need = [-(-(p + n) // bs) for p, n in chunks]
    nb = sum(need) + 5
    perm = torch.randperm(nb, generator=g).tolist()
    tables, pos = [], 0
    for k in need:
        tables.append(perm[pos:pos + k]); pos += k
    mb = max(need)
    k_pool = torch.randn((nb, hkv, bs, D), generator=g).to(DT[dtype])
    v_pool = torch.randn((nb, hkv, bs, D), generator=g).to(DT[dtype])
    if nan_fill:
        valid = torch.zeros((nb, bs), dtype=torch.bool)
        for t, (p, n) in zip(tables, chunks):
            for j in range(p + n):
                valid[t[j // bs], j % bs] = True
        m = (~valid).view(nb, 1, bs, 1).expand_as(k_pool)
        k_pool[m] = float("nan")
        v_pool[m] = float("nan")
    total = sum(n for _, n in chunks)
    q = torch.randn((total, hq, D), generator=g).to(DT[dtype])
    cu = [0]
    for _, n in chunks:
        cu.append(cu[-1] + n)
    tab = [t + [-1] * (mb - len(t)) for t in tables]
    return dict(k=k_pool, v=v_pool, q=q, cu=cu, starts=[p for p, _ in chunks], tables=tab, dtype=dtype,
                hq=hq, hkv=hkv, max_q=max(n for _, n in chunks), chunks=chunks)


def _run(c):
    import paged_kv_cache_160_gb300 as pkv
    dev = torch.device("cuda")
    kc, vc = c["k"].to(dev), c["v"].to(dev)
    desc = pkv.cache_desc(kc)
    q = c["q"].to(dev)
    out = torch.full_like(q, float("nan"))
    pkv.pkv_get_device_error()
    pkv.pkv_paged_prefill_chunk(out, q, torch.tensor(c["cu"], dtype=torch.int32, device=dev),
                                torch.tensor(c["starts"], dtype=torch.int32, device=dev), c["max_q"], kc, vc, desc,
                                torch.tensor(c["tables"], dtype=torch.int32, device=dev), 1 / math.sqrt(128))
    err = pkv.pkv_get_device_error()
    return out.cpu(), err


def _check(c, rows_per_chunk=None):
    from oracle.paged_attention import prefill_chunk_attention
    out, err = _run(c)
    assert err == 0, f"device error {err:#x}"
    kcodes, vcodes = codes(c["k"]), codes(c["v"])
    worst = 0.0
    for i, (p, n) in enumerate(c["chunks"]):
        lo, hi = c["cu"][i], c["cu"][i + 1]
        rows = None if rows_per_chunk is None else [r for r in rows_per_chunk if r < n]
        ref = prefill_chunk_attention(q_f64(c["q"][lo:hi]), kcodes, vcodes, c["dtype"], c["tables"][i], p,
                                      1 / math.sqrt(128), rows=rows)
        got = out[lo:hi].to(torch.float64).numpy()
        mask = ~np.isnan(ref)
        d = np.abs(got[mask] - ref[mask])
        assert not np.isnan(d).any(), f"NaN in chunk {i}"
        worst = max(worst, float(d.max()))
    assert worst <= TOL[c["dtype"]], f"max abs err {worst:.3e}"
    return worst


def test_single_chunk_no_prefix_bf16():
    _check(_case(1, [(0, 128)], 4, 4, "bf16"))


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_varlen_chunks_ragged(dtype):
    # prefixes not aligned to 128 or 16, q_len not multiples of 128, one chunk of 1 token
    _check(_case(2, [(37, 200), (0, 5), (300, 129), (1000, 1), (128, 256)], 8, 2, dtype))


def test_block_size_32_chunks():
    """32-token blocks: the kernel gathers each 128-key tile as eight 16-row halves of blocks."""
    _check(_case(5, [(37, 200), (0, 5), (300, 129), (1000, 1)], 8, 2, "bf16", nan_fill=True, bs=32))


def test_single_row_chunks_after_long_prefixes_repeat_exactly():
    """One query row whose keys end inside the last tile: the epilogue must see every PV
    product of the row (the last ones finish after the softmax is done), on every run."""
    c = _case(6, [(600, 1), (1000, 1), (77, 1), (3000, 1)], 8, 2, "bf16")
    first = _check(c)
    for _ in range(4):
        out, err = _run(c)
        assert err == 0
        again, _ = _run(c)
        assert torch.equal(out, again)
    assert first <= TOL["bf16"]


@pytest.mark.parametrize("seed", range(6))
def test_random_chunks(seed):
    """Random chunk counts, prefixes, lengths, head groups and block sizes, NaN in unused rows."""
    rng = np.random.default_rng(seed)
    chunks = [(int(rng.integers(0, 1200)), int(rng.integers(1, 300))) for _ in range(int(rng.integers(1, 5)))]
    hkv = int(rng.integers(1, 3))
    hq = hkv * int(rng.integers(1, 9))
    dtype = ["bf16", "f16"][seed % 2]
    bs = [16, 32][(seed // 2) % 2]
    _check(_case(10 + seed, chunks, hq, hkv, dtype, nan_fill=True, bs=bs), rows_per_chunk=list(range(0, 300, 7)))


@pytest.mark.parametrize("bs", [16, 32])
def test_mha_pairs_of_query_tiles(bs):
    # one query head per kv head: a CTA takes two adjacent q-tiles of a head.  Chunks of 3, 2
    # and 3 q-tiles (the last pair's second tile lies past the chunk), ragged tails, prefixes
    # not aligned to 16 or 128.
    _check(_case(8, [(0, 300), (77, 129), (500, 257), (3, 1)], 4, 4, "bf16", nan_fill=True, bs=bs))


@pytest.mark.parametrize("hq,hkv", [(8, 2), (32, 2), (4, 4)])
def test_multi_tile_chunks_repeat_exactly(hq, hkv):
    """Several key tiles per CTA and both halves of the key range: every run gives the same
    bits.  (The wait for the last PV product once read O while products were still landing,
    by a few ulps, differently from run to run.)"""
    c = _case(11, [(37, 200), (300, 129), (128, 256)], hq, hkv, "bf16")
    first, err = _run(c)
    assert err == 0
    for _ in range(4):
        again, err = _run(c)
        assert err == 0
        assert torch.equal(first, again)


@pytest.mark.parametrize("hq,hkv", [(6, 2), (32, 2)])
def test_group_sizes_3_and_16(hq, hkv):
    # an odd group (its last head pair repeats a head) and a group wider than the decode's 8
    _check(_case(9, [(100, 200), (0, 130)], hq, hkv, "bf16"))


def test_gqa7_long_prefix():
    _check(_case(3, [(3584, 512)], 28, 4, "bf16"), rows_per_chunk=[0, 1, 63, 127, 128, 300, 511])


def test_max_q_len_below_a_chunk_length_is_flagged():
    """max_q_len sizes the grid; a chunk longer than it is reported, not silently cut."""
    import paged_kv_cache_160_gb300 as pkv
    from paged_kv_cache_160_gb300._binding import DEVERR
    for hq, hkv in ((8, 2), (4, 4)):
        c = _case(12, [(10, 300)], hq, hkv, "bf16")
        dev = torch.device("cuda")
        kc, vc = c["k"].to(dev), c["v"].to(dev)
        out = torch.zeros_like(c["q"]).to(dev)
        pkv.pkv_get_device_error()
        pkv.pkv_paged_prefill_chunk(out, c["q"].to(dev), torch.tensor(c["cu"], dtype=torch.int32, device=dev),
                                    torch.tensor(c["starts"], dtype=torch.int32, device=dev), 100, kc, vc,
                                    pkv.cache_desc(kc), torch.tensor(c["tables"], dtype=torch.int32, device=dev),
                                    1 / math.sqrt(128))
        assert pkv.pkv_get_device_error() & DEVERR["chunk"]


def test_nan_in_unused_rows_never_reaches_output():
    _check(_case(4, [(5, 40), (77, 100)], 4, 1, "bf16", nan_fill=True))


def test_mixed_workload_chunk():
    """The mixed step's 512-token chunk at positions 3584..4095, after kv_write, via the harness."""
    import synth
    from tests.harness import device_run, max_abs_err, oracle_plan, oracle_run, product_plan
    case = synth.mixed_config()
    pp = product_plan(case)
    assert pp == oracle_plan(case)
    dev = device_run(case, pp, keep_intermediate=False)
    assert dev.device_error == 0
    ref = oracle_run(case, pp, decode_rows=[(0, 0)], prefill_rows=[0, 1, 100, 255, 256, 400, 511],
                     prefill_heads=[0, 6, 7, 20, 27])
    err = max_abs_err(dev.prefill, ref.prefill)
    assert err <= TOL["bf16"], err


def test_refuses_q_or_caches_that_are_not_memory_of_this_gpu():
    """The prefill kernel multicasts its K/V tiles across a cluster, so the call takes q and the
    caches only in device memory of the current GPU: a pinned host k_cache, v_cache or q is
    refused with PKV_ERR_INVALID_ARG before anything is enqueued (out stays untouched)."""
    import ctypes
    import paged_kv_cache_160_gb300 as pkv
    from paged_kv_cache_160_gb300._binding import pkv_dtype_of
    c = _case(7, [(20, 30)], 4, 2, "bf16")
    dev = torch.device("cuda")
    kc, vc, q = c["k"].to(dev), c["v"].to(dev), c["q"].to(dev)
    hk, hv, hq = c["k"].pin_memory(), c["v"].pin_memory(), c["q"].pin_memory()
    desc = pkv.cache_desc(kc)
    out = torch.full_like(q, float("nan"))
    cu = torch.tensor(c["cu"], dtype=torch.int32, device=dev)
    st = torch.tensor(c["starts"], dtype=torch.int32, device=dev)
    tab = torch.tensor(c["tables"], dtype=torch.int32, device=dev)

    def call(qq, kk, vv):
        return pkv.lib.pkv_paged_prefill_chunk(out.data_ptr(), qq.data_ptr(), pkv_dtype_of(q), cu.data_ptr(),
                                               st.data_ptr(), 1, q.shape[0], c["max_q"], q.shape[1], kk.data_ptr(),
                                               vv.data_ptr(), ctypes.byref(desc), tab.data_ptr(), tab.shape[1],
                                               1 / math.sqrt(128), torch.cuda.current_stream().cuda_stream)

    assert call(q, hk, vc) == 1
    assert call(q, kc, hv) == 1
    assert call(hq, kc, vc) == 1
    torch.cuda.synchronize()
    assert torch.isnan(out).all()
    assert call(q, kc, vc) == 0                    # the same call on device memory runs
    torch.cuda.synchronize()
    assert not torch.isnan(out).any()
    assert pkv.pkv_get_device_error() == 0
