"""GPU end to end of prefix caching: a second request re-uses the cached blocks of a shared
system prompt ("PagedAttention: manage the KV cache like virtual memory" §3.4: equal prefixes
give equal block hashes, so the table points at the computed blocks; the K/V bytes are the
same, so the output does not change).

K/V rows are a fixed function of (token id, position), as a model's would be.  Request B
writes only its uncached tokens and runs paged_prefill_chunk from its first uncached
position; the result must equal the oracle's causal attention over B's own K/V computed
from scratch in a separate pool.
"""
import math

import numpy as np
import pytest
import torch

from oracle.paged_attention import prefill_chunk_attention
from tests.harness import TOL, codes, max_abs_err, q_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")


def test_second_request_reuses_the_cached_system_prompt():
    import paged_kv_cache_160_gb300 as pkv
    dev = torch.device("cuda")
    hq, hkv, d, bs, nb, vocab = 28, 4, 128, 16, 128, 1000
    g = torch.Generator().manual_seed(21)
    tok_k, tok_v = torch.randn(vocab, hkv, d, generator=g), torch.randn(vocab, hkv, d, generator=g)
    pos_k, pos_v = torch.randn(1024, hkv, d, generator=g), torch.randn(1024, hkv, d, generator=g)

    def kv_rows(tokens, start):
        t = torch.tensor(tokens)
        p = torch.arange(start, start + len(tokens))
        return ((tok_k[t] + 0.25 * pos_k[p]).to(torch.bfloat16), (tok_v[t] + 0.25 * pos_v[p]).to(torch.bfloat16))

    rng = np.random.default_rng(3)
    system = [int(x) for x in rng.integers(0, vocab, 200)]
    a = system + [int(x) for x in rng.integers(0, vocab, 37)]
    b = system + [int(x) for x in rng.integers(0, vocab, 50)]

    kc = torch.full((nb, hkv, bs, d), float("nan"), dtype=torch.bfloat16, device=dev)
    vc = torch.full_like(kc, float("nan"))
    desc = pkv.cache_desc(kc)
    bm = pkv.BlockManager(nb, bs)

    def write(seq, tokens, start):
        tab, _ = bm.export([seq], 32)
        slots = [tab[0][p // bs] * bs + p % bs for p in range(start, len(tokens))]
        kn, vn = kv_rows(tokens[start:], start)
        pkv.pkv_kv_write(kn.to(dev), vn.to(dev), torch.tensor(slots, dtype=torch.int64, device=dev), kc, vc, desc)

    assert bm.allocate_cached(1, a) == 0
    write(1, a, 0)
    cached = bm.allocate_cached(2, b)
    assert cached == (200 // bs) * bs                    # 12 shared blocks, 192 tokens
    write(2, b, cached)                                  # only B's uncached tokens are written
    tab_b, _ = bm.export([2], 32)
    assert tab_b[0][:12] == bm.export([1], 32)[0][0][:12]

    n_new = len(b) - cached
    q = torch.randn(n_new, hq, d, generator=g).to(torch.bfloat16)
    out = torch.full((n_new, hq, d), float("nan"), dtype=torch.bfloat16, device=dev)
    scale = 1 / math.sqrt(d)
    pkv.pkv_get_device_error()
    pkv.pkv_paged_prefill_chunk(out, q.to(dev), torch.tensor([0, n_new], dtype=torch.int32, device=dev),
                                torch.tensor([cached], dtype=torch.int32, device=dev), n_new, kc, vc, desc,
                                torch.tensor(tab_b, dtype=torch.int32, device=dev), scale)
    assert pkv.pkv_get_device_error() == 0

    # from scratch: B's own K/V for every position, in a contiguous pool of its own
    kb, vb = kv_rows(b, 0)
    nbb = -(-len(b) // bs)
    pad = nbb * bs - len(b)
    kpool = torch.cat([kb, torch.zeros(pad, hkv, d, dtype=torch.bfloat16)]).view(nbb, bs, hkv, d).transpose(1, 2)
    vpool = torch.cat([vb, torch.zeros(pad, hkv, d, dtype=torch.bfloat16)]).view(nbb, bs, hkv, d).transpose(1, 2)
    ref = prefill_chunk_attention(q_f64(q), codes(kpool.contiguous()), codes(vpool.contiguous()), "bf16",
                                  list(range(nbb)), cached, scale)
    assert max_abs_err(out.cpu(), ref) <= TOL["bf16"]
