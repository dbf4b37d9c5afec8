"""Pins for the oracle's paged attention (CPU only).

Each pin checks the oracle against something other than itself:

* the address-translation worked example the pages print (token 37 -> block 142, slot 5);
* torch's scaled_dot_product_attention in float64 on the same K/V laid out contiguously
  (the textbook definition that paged attention must equal);
* invariance to a random relabelling of physical block ids;
* identical outputs for sequences that share prefix blocks;
* closed forms (one key; zero query; one dominant key);
* the exact log-sum-exp identity of split-KV partials;
* causal chunked prefill against SDPA with a causal (bottom-right aligned) mask;
* the per-sequence waste bound of at most one partial block.

``test_planted_mistakes_are_caught`` plants plausible bugs into the oracle (on the CPU)
and checks that these pins fail for each of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import paged_attention as pa
from oracle.formats import to_f64


# ---------------------------------------------------------------------------------------
# helpers: contiguous K/V scattered into a paged pool by a random table (test side)
# ---------------------------------------------------------------------------------------

def _paged_case(seed, lens, hq, hkv, d, bs=16, spare=7, dtype="f16"):
    rng = np.random.default_rng(seed)
    nblk = [-(-L // bs) for L in lens]
    nb = sum(nblk) + spare
    perm = rng.permutation(nb)
    tables, k_contig, v_contig = [], [], []
    np_dt = np.float16
    k_pool = rng.standard_normal((nb, hkv, bs, d)).astype(np_dt)
    v_pool = rng.standard_normal((nb, hkv, bs, d)).astype(np_dt)
    pos = 0
    for L, n in zip(lens, nblk):
        t = [int(x) for x in perm[pos:pos + n]]
        pos += n
        tables.append(t)
        kc = rng.standard_normal((L, hkv, d)).astype(np_dt)
        vc = rng.standard_normal((L, hkv, d)).astype(np_dt)
        for j in range(L):                       # scatter token j by plain indexing
            k_pool[t[j // bs], :, j % bs, :] = kc[j]
            v_pool[t[j // bs], :, j % bs, :] = vc[j]
        k_contig.append(kc.astype(np.float64))
        v_contig.append(vc.astype(np.float64))
    q = rng.standard_normal((len(lens), hq, d)).astype(np_dt).astype(np.float64)
    return dict(q=q, k_pool=k_pool.view(np.uint16), v_pool=v_pool.view(np.uint16), tables=tables,
                k_contig=k_contig, v_contig=v_contig, lens=lens, hq=hq, hkv=hkv, d=d, bs=bs)


def _sdpa(q, k, v, scale, mask=None):
    """torch SDPA in float64; q [Hq, n, D], k/v [Hq, L, D]."""
    return torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v),
        attn_mask=None if mask is None else torch.from_numpy(mask), scale=scale).numpy()


def _sdpa_decode(c, i, scale):
    group = c["hq"] // c["hkv"]
    k = np.repeat(c["k_contig"][i].transpose(1, 0, 2), group, axis=0)    # [Hq, L, D]
    v = np.repeat(c["v_contig"][i].transpose(1, 0, 2), group, axis=0)
    return _sdpa(c["q"][i][:, None, :], k, v, scale)[:, 0, :]


# ---------------------------------------------------------------------------------------

def test_address_translation_worked_example(golden_dir):
    ex = json.load(open(os.path.join(golden_dir, "address_translation.json")))
    table = [3, 9, ex["physical_block"], 4]
    slot = pa.slot_of_position(table, ex["token"], ex["block_size"])
    assert slot == ex["slot"]
    assert (slot // ex["block_size"], slot % ex["block_size"]) == (ex["physical_block"], ex["offset"])
    assert ex["token"] // ex["block_size"] == ex["logical_block"]
    # logical_rows must fetch exactly pool[142, h, 5] for token 37
    pool = np.zeros((150, 1, 16, 4), dtype=np.uint16)
    pool[142, 0, 5, :] = np.array([1.5, -2.0, 3.25, 0.5], dtype=np.float16).view(np.uint16)
    rows = pa.logical_rows(pool, "f16", table, 38, 0)
    assert np.array_equal(rows[37], [1.5, -2.0, 3.25, 0.5])


@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 2), (7, 1), (12, 4)])
def test_decode_equals_sdpa_on_contiguous(hq, hkv):
    c = _paged_case(11 + hq, [1, 5, 16, 17, 40, 100], hq, hkv, 32)
    scale = 1 / math.sqrt(32)
    out = pa.decode_attention(c["q"], c["k_pool"], c["v_pool"], "f16", c["tables"], c["lens"], scale)
    for i in range(len(c["lens"])):
        np.testing.assert_allclose(out[i], _sdpa_decode(c, i, scale), rtol=0, atol=1e-12)


def test_decode_invariant_to_block_relabelling():
    c = _paged_case(3, [9, 33, 64, 70], 8, 2, 16, spare=20)
    scale = 0.25
    base = pa.decode_attention(c["q"], c["k_pool"], c["v_pool"], "f16", c["tables"], c["lens"], scale)
    nb = c["k_pool"].shape[0]
    perm = np.random.default_rng(5).permutation(nb)          # old id b -> new id perm[b]
    k2 = np.empty_like(c["k_pool"]); v2 = np.empty_like(c["v_pool"])
    k2[perm] = c["k_pool"]; v2[perm] = c["v_pool"]
    tables2 = [[int(perm[b]) for b in t] for t in c["tables"]]
    out = pa.decode_attention(c["q"], k2, v2, "f16", tables2, c["lens"], scale)
    assert np.array_equal(out, base)


def test_shared_prefix_blocks_give_identical_outputs():
    c = _paged_case(4, [48, 48], 4, 4, 16)
    tables = [c["tables"][0], list(c["tables"][0])]            # second sequence shares all blocks
    q = c["q"].copy(); q[1] = q[0]
    out = pa.decode_attention(q, c["k_pool"], c["v_pool"], "f16", tables, [48, 48], 0.3)
    assert np.array_equal(out[0], out[1])
    # sharing only the first two blocks, identical query, same length -> identical too when
    # the private third blocks hold identical bytes
    k = c["k_pool"].copy(); v = c["v_pool"].copy()
    spare = c["k_pool"].shape[0] - 1
    k[spare] = k[c["tables"][0][2]]; v[spare] = v[c["tables"][0][2]]
    tables = [c["tables"][0], c["tables"][0][:2] + [spare]]
    out = pa.decode_attention(q, k, v, "f16", tables, [48, 48], 0.3)
    assert np.array_equal(out[0], out[1])


def test_closed_forms():
    c = _paged_case(6, [1, 50, 50], 2, 2, 8)
    scale = 0.5
    # one key: out == v_0 exactly
    out = pa.decode_attention(c["q"], c["k_pool"], c["v_pool"], "f16", c["tables"], c["lens"], scale)
    np.testing.assert_array_equal(out[0], c["v_contig"][0][0].reshape(2, 8))
    # zero query: uniform weights -> mean of V
    q0 = np.zeros_like(c["q"])
    out = pa.decode_attention(q0, c["k_pool"], c["v_pool"], "f16", c["tables"], c["lens"], scale)
    np.testing.assert_allclose(out[1], c["v_contig"][1].mean(axis=0), rtol=0, atol=1e-12)
    # one dominant key (k_j = 50 q) -> output is that key's value row
    k = c["k_pool"].copy()
    j = 17
    t = c["tables"][2]
    qd = np.zeros_like(c["q"]); qd[2, :, 0] = 1.0
    row = np.zeros(8, dtype=np.float16); row[0] = 50.0
    k[t[j // 16], :, j % 16, :] = row.view(np.uint16)
    out = pa.decode_attention(qd, k, c["v_pool"], "f16", c["tables"], c["lens"], 1.0)
    np.testing.assert_allclose(out[2], c["v_contig"][2][j], rtol=0, atol=1e-12 + 60 * math.exp(-40))


def test_empty_sequence_gives_zeros():
    c = _paged_case(8, [0, 20], 2, 2, 8)
    out = pa.decode_attention(c["q"], c["k_pool"], c["v_pool"], "f16", c["tables"], c["lens"], 0.3)
    assert np.array_equal(out[0], np.zeros((2, 8)))


@pytest.mark.parametrize("part", [16, 48, 512])
def test_split_kv_partials_merge_to_unsplit(part):
    c = _paged_case(9, [1000, 17], 6, 2, 16)
    scale = 0.25
    full = pa.decode_attention(c["q"], c["k_pool"], c["v_pool"], "f16", c["tables"], c["lens"], scale)
    for i, L in enumerate(c["lens"]):
        for h in range(6):
            parts = pa.decode_partials(c["q"][i], c["k_pool"], c["v_pool"], "f16", c["tables"][i], L,
                                       scale, h, part)
            assert len(parts) == -(-L // part)
            np.testing.assert_allclose(pa.merge_partials(parts), full[i, h], rtol=0, atol=1e-12)


def test_e4m3_cache_uses_per_head_scales():
    rng = np.random.default_rng(12)
    pool_k = rng.integers(0, 0x7E, size=(4, 2, 16, 8), dtype=np.uint8)    # finite codes only
    pool_v = rng.integers(0, 0x7E, size=(4, 2, 16, 8), dtype=np.uint8)
    ks, vs = np.array([0.5, 2.0]), np.array([1.25, 0.75])
    q = rng.standard_normal((1, 4, 8))
    table, L = [2, 0], 20
    out = pa.decode_attention(q, pool_k, pool_v, "e4m3", [table], [L], 0.1, ks, vs)
    for h in range(4):
        g = h // 2
        K = np.concatenate([to_f64(pool_k[2, g], "e4m3"), to_f64(pool_k[0, g], "e4m3")])[:L] * ks[g]
        V = np.concatenate([to_f64(pool_v[2, g], "e4m3"), to_f64(pool_v[0, g], "e4m3")])[:L] * vs[g]
        ref = _sdpa(q[0, h][None, None, :], K[None], V[None], 0.1)[0, 0]
        np.testing.assert_allclose(out[0, h], ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("prefix,n", [(0, 37), (48, 20), (5, 64)])
def test_prefill_chunk_equals_causal_sdpa(prefix, n):
    total = prefix + n
    c = _paged_case(20 + prefix, [total], 4, 2, 16)
    scale = 0.25
    rng = np.random.default_rng(prefix)
    q = rng.standard_normal((n, 4, 16)).astype(np.float16).astype(np.float64)
    out = pa.prefill_chunk_attention(q, c["k_pool"], c["v_pool"], "f16", c["tables"][0], prefix, scale)
    k = np.repeat(c["k_contig"][0].transpose(1, 0, 2), 2, axis=0)
    v = np.repeat(c["v_contig"][0].transpose(1, 0, 2), 2, axis=0)
    if prefix == 0:
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q.transpose(1, 0, 2).copy()), torch.from_numpy(k), torch.from_numpy(v),
            is_causal=True, scale=scale).numpy()
    else:
        mask = np.tril(np.ones((n, total), dtype=bool), k=prefix)        # row r sees keys <= prefix + r
        ref = _sdpa(q.transpose(1, 0, 2).copy(), k, v, scale, mask)
    np.testing.assert_allclose(out, ref.transpose(1, 0, 2), rtol=0, atol=1e-12)


def test_waste_is_at_most_one_partial_block_per_sequence():
    """"PagedAttention: manage the KV cache like virtual memory" §3.1: only a sequence's last
    block can be partly empty.  Grow 200 sequences of random lengths token by token on the
    oracle's block manager and count, for each, the reserved slots it does not use."""
    from oracle.block_manager import BlockManagerModel
    rng = np.random.default_rng(1)
    bs = 16
    lens = [int(x) for x in rng.integers(1, 600, size=200)]
    bm = BlockManagerModel(sum(-(-L // bs) for L in lens), bs)
    for i, L in enumerate(lens):
        bm.allocate(i, 1)
        for _ in range(L - 1):
            bm.append_slot(i)
    tables, got = bm.export(list(range(len(lens))), max(-(-L // bs) for L in lens))
    assert got == lens
    assert bm.num_free() == 0                                   # every block is in some table
    for t, L in zip(tables, lens):
        reserved = bs * sum(1 for b in t if b >= 0)
        assert 0 <= reserved - L <= bs - 1


# ---------------------------------------------------------------------------------------
# planted mistakes: each variant of the oracle must fail at least one pin above
# ---------------------------------------------------------------------------------------

def _bad_rows_offset(cache, kv_dtype, table, n, g, scale=None):
    out = _orig_rows(cache, kv_dtype, table, n + 1, g, scale)
    return out[1:]                                               # off-by-one token


def _bad_rows_head(cache, kv_dtype, table, n, g, scale=None):
    return _orig_rows(cache, kv_dtype, table, n, (g + 1) % cache.shape[1], scale)   # wrong kv head


def _bad_rows_block(cache, kv_dtype, table, n, g, scale=None):
    bs = cache.shape[2]
    t = list(table) + [table[0]]
    shifted = [t[(b + 1) % (len(table))] for b in range(len(table))]           # wrong block order
    return _orig_rows(cache, kv_dtype, shifted, n, g, scale)


def _bad_softmax_no_max(q, k, v, scale):
    if k.shape[0] == 0:
        return np.zeros(v.shape[1])
    s = scale * (k @ q)
    p = np.exp(s)
    return (p @ v) / (p.sum() + 1e-3)                             # wrong normaliser


def _bad_softmax_transposed_scale(q, k, v, scale):
    if k.shape[0] == 0:
        return np.zeros(v.shape[1])
    s = (k @ q) / scale                                           # scale applied inversely
    p = np.exp(s - s.max())
    return (p @ v) / p.sum()


_orig_rows = pa.logical_rows


@pytest.mark.parametrize("name,target,bad", [
    ("token offset", "logical_rows", _bad_rows_offset),
    ("kv head", "logical_rows", _bad_rows_head),
    ("block order", "logical_rows", _bad_rows_block),
    ("normaliser", "softmax_attention", _bad_softmax_no_max),
    ("scale", "softmax_attention", _bad_softmax_transposed_scale),
])
def test_planted_mistakes_are_caught(monkeypatch, name, target, bad):
    monkeypatch.setattr(pa, target, bad)
    c = _paged_case(31, [40, 70], 4, 2, 16)
    scale = 0.25
    out = pa.decode_attention(c["q"], c["k_pool"], c["v_pool"], "f16", c["tables"], c["lens"], scale)
    worst = max(np.abs(out[i] - _sdpa_decode(c, i, scale)).max() for i in range(2))
    assert worst > 1e-6, f"planted mistake '{name}' not caught"
