"""Seeded synthetic workloads for paged-KV decode, chunked prefill and CoW.

Shapes follow the five workloads the library is measured on:

* tiny paged decode (4 sequences, MHA 4 heads, head_dim 64, fp16, one shared block);
* a Qwen2.5-7B-shaped GQA decode batch (28/4 heads, head_dim 128, bf16, 64 sequences);
* a 13B-shaped MHA continuous batch (40 heads, fp16, 256 lognormal-length sequences,
  a quarter of them sharing a 1024-token prefix);
* a long-context split-KV decode (32/8 heads, e4m3 KV with per-kv-head scales,
  8 sequences of 32k..128k tokens, 512-token partitions);
* a mixed step (one 512-token causal prefill chunk over a 3584-token paged prefix,
  128 decode sequences, 64 copy-on-write block pairs).

Every random draw comes from one ``torch.Generator`` seeded with ``1600 + n``
(n = workload number), in a fixed order, on the CPU, so the oracle and the GPU
receive identical bytes.  Nothing here computes attention, slots or tables: the
block lists describe which physical blocks hold each sequence's cached tokens
*before* the step; appending the step's new token is the block manager's job.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, List, Optional, Tuple

import torch

TORCH_DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16, "e4m3": torch.uint8}
E4M3_MAX = 448.0


@dataclass
class PrefillChunk:
    """A causal query chunk of ``q_len`` tokens appended after ``prefix_len`` cached tokens."""
    prefix_len: int
    q_len: int
    blocks: List[int]            # physical blocks holding the prefix (logical order)
    q: torch.Tensor              # [q_len, Hq, D]
    k_new: torch.Tensor          # [q_len, Hkv, D]
    v_new: torch.Tensor          # [q_len, Hkv, D]


@dataclass
class DecodeCase:
    name: str
    seed: int
    block_size: int
    num_blocks: int
    num_heads: int
    num_kv_heads: int
    head_dim: int
    q_dtype: str                 # "f16" | "bf16"
    kv_dtype: str                # "f16" | "bf16" | "e4m3"
    scale: float
    context_lens: List[int]      # tokens cached per decode sequence before the step
    seq_blocks: List[List[int]]  # physical blocks holding those tokens, logical order
    q: torch.Tensor              # [S, Hq, D]
    k_cache: torch.Tensor        # [NB, Hkv, BS, D]
    v_cache: torch.Tensor
    k_scale: Optional[torch.Tensor] = None   # [Hkv] float32 (e4m3 caches only)
    v_scale: Optional[torch.Tensor] = None
    k_new: Optional[torch.Tensor] = None     # [S, Hkv, D]: one new token per sequence
    v_new: Optional[torch.Tensor] = None
    partition_size: int = 0      # tokens per split-KV partition; 0 = library's choice
    chunk: Optional[PrefillChunk] = None
    copy_pairs: int = 0          # number of copy-on-write block pairs in the step
    meta: Dict[str, object] = field(default_factory=dict)

    @property
    def num_seqs(self) -> int:
        return len(self.context_lens)

    @property
    def writes(self) -> bool:
        return self.k_new is not None


def _randn(g: torch.Generator, shape, dtype: str, scale: Optional[torch.Tensor] = None,
           head_axis: int = -2) -> torch.Tensor:
    """N(0,1) draws stored in ``dtype``; e4m3 stores round(x / scale[h]) as raw bytes."""
    x = torch.randn(shape, generator=g, dtype=torch.float32)
    if dtype == "e4m3":
        assert scale is not None
        view = [1] * len(shape)
        view[head_axis] = scale.numel()
        x = (x / scale.view(view)).clamp(-E4M3_MAX, E4M3_MAX)
        return x.to(torch.float8_e4m3fn).view(torch.uint8)
    return x.to(TORCH_DTYPES[dtype])


def _pool(g: torch.Generator, nb: int, hkv: int, bs: int, d: int, dtype: str,
          scale: Optional[torch.Tensor], chunk_blocks: int = 4096) -> torch.Tensor:
    """Draw the whole physical pool, in chunks of blocks to bound host memory."""
    parts = []
    for b0 in range(0, nb, chunk_blocks):
        n = min(chunk_blocks, nb - b0)
        parts.append(_randn(g, (n, hkv, bs, d), dtype, scale, head_axis=1))
    return torch.cat(parts, 0) if parts else torch.empty((0, hkv, bs, d), dtype=TORCH_DTYPES[dtype])


def _ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def make_decode_case(name: str, seed: int, lens: List[int], num_heads: int, num_kv_heads: int,
                     head_dim: int, q_dtype: str, kv_dtype: str, *, block_size: int = 16,
                     num_blocks: Optional[int] = None, share: Optional[Dict[int, Tuple[int, int]]] = None,
                     write: bool = True, partition_size: int = 0, scale: Optional[float] = None,
                     chunk: Optional[Tuple[int, int]] = None, copy_pairs: int = 0,
                     pool_slack: float = 1.1, unused_fill: str = "noise",
                     g: Optional[torch.Generator] = None) -> DecodeCase:
    """Build a decode (optionally + prefill chunk) case.

    ``share[i] = (j, n)`` makes sequence i reuse sequence j's first n physical blocks
    (j < i).  ``chunk = (prefix_len, q_len)`` adds a prefill-chunk sequence after the
    decode sequences.  ``unused_fill="nan"`` fills every pool row that holds no valid
    token with NaN (f16/bf16) or the e4m3 NaN byte, to expose reads past a sequence end.
    """
    if g is None:
        g = torch.Generator().manual_seed(seed)
    bs = block_size
    share = share or {}
    S = len(lens)
    # Blocks each sequence holds before the step.
    n_before = [_ceil_div(L, bs) for L in lens]
    n_after_total = sum(_ceil_div(L + (1 if write else 0), bs) for L in lens)
    shared_dups = sum(n for (_, n) in share.values())
    chunk_blocks_before = _ceil_div(chunk[0], bs) if chunk else 0
    chunk_blocks_after = _ceil_div(chunk[0] + chunk[1], bs) if chunk else 0
    unique_before = sum(n_before) - shared_dups + chunk_blocks_before
    needed_after = n_after_total - shared_dups + chunk_blocks_after + copy_pairs
    if num_blocks is None:
        num_blocks = max(1, int(math.ceil(pool_slack * needed_after)))
    assert num_blocks >= needed_after, "pool too small for the step"
    perm = torch.randperm(num_blocks, generator=g).tolist()
    nxt = 0
    seq_blocks: List[List[int]] = []
    for i in range(S):
        blocks: List[int] = []
        src = share.get(i)
        if src is not None:
            j, n = src
            assert j < i and n <= n_before[j] and n <= n_before[i]
            blocks.extend(seq_blocks[j][:n])
        while len(blocks) < n_before[i]:
            blocks.append(perm[nxt]); nxt += 1
        seq_blocks.append(blocks)
    chunk_blk: List[int] = []
    for _ in range(chunk_blocks_before):
        chunk_blk.append(perm[nxt]); nxt += 1
    assert nxt == unique_before

    k_scale = v_scale = None
    if kv_dtype == "e4m3":
        k_scale = torch.empty(num_kv_heads).uniform_(0.5, 2.0, generator=g)
        v_scale = torch.empty(num_kv_heads).uniform_(0.5, 2.0, generator=g)
    q = _randn(g, (S, num_heads, head_dim), q_dtype)
    k_cache = _pool(g, num_blocks, num_kv_heads, bs, head_dim, kv_dtype, k_scale)
    v_cache = _pool(g, num_blocks, num_kv_heads, bs, head_dim, kv_dtype, v_scale)
    k_new = v_new = None
    if write:
        k_new = _randn(g, (S, num_kv_heads, head_dim), kv_dtype, k_scale)
        v_new = _randn(g, (S, num_kv_heads, head_dim), kv_dtype, v_scale)
    pchunk = None
    if chunk:
        prefix_len, q_len = chunk
        pchunk = PrefillChunk(prefix_len=prefix_len, q_len=q_len, blocks=chunk_blk,
                              q=_randn(g, (q_len, num_heads, head_dim), q_dtype),
                              k_new=_randn(g, (q_len, num_kv_heads, head_dim), kv_dtype, k_scale),
                              v_new=_randn(g, (q_len, num_kv_heads, head_dim), kv_dtype, v_scale))
    if unused_fill == "nan":
        _fill_unused(k_cache, v_cache, seq_blocks, lens, chunk_blk, chunk[0] if chunk else 0, bs, kv_dtype)
    if scale is None:
        scale = 1.0 / math.sqrt(head_dim)
    return DecodeCase(name=name, seed=seed, block_size=bs, num_blocks=num_blocks,
                      num_heads=num_heads, num_kv_heads=num_kv_heads, head_dim=head_dim,
                      q_dtype=q_dtype, kv_dtype=kv_dtype, scale=scale, context_lens=list(lens),
                      seq_blocks=seq_blocks, q=q, k_cache=k_cache, v_cache=v_cache,
                      k_scale=k_scale, v_scale=v_scale, k_new=k_new, v_new=v_new,
                      partition_size=partition_size, chunk=pchunk, copy_pairs=copy_pairs)


def _fill_unused(k_cache, v_cache, seq_blocks, lens, chunk_blk, chunk_len, bs, kv_dtype):
    """Overwrite every pool row that holds no cached token with a NaN pattern."""
    valid = torch.zeros(k_cache.shape[0], dtype=torch.int64)
    for blocks, L in list(zip(seq_blocks, lens)) + [(chunk_blk, chunk_len)]:
        for b, pb in enumerate(blocks):
            valid[pb] = max(int(valid[pb]), min(bs, L - b * bs))
    rows = torch.arange(bs).view(1, bs)
    dead = rows >= valid.view(-1, 1)                       # [NB, BS]
    for cache in (k_cache, v_cache):
        m = dead.view(-1, 1, bs, 1).expand_as(cache)
        if kv_dtype == "e4m3":
            cache[m] = 0x7F                                 # e4m3 NaN byte
        else:
            cache[m] = float("nan")


# ----------------------------------------------------------------------------------------
# The five workloads.
# ----------------------------------------------------------------------------------------

def tiny_config() -> DecodeCase:
    """4 sequences {10, 6, 37, 16}, pool of 64 blocks, sequences 0 and 3 share logical block 0."""
    return make_decode_case("tiny", 1601, [10, 6, 37, 16], 4, 4, 64, "f16", "f16",
                            num_blocks=64, share={3: (0, 1)}, scale=1.0 / math.sqrt(64))


def qwen7b_gqa_config() -> DecodeCase:
    """Qwen2.5-7B-shaped GQA decode: 64 sequences, lengths uniform in [128, 2048]."""
    g = torch.Generator().manual_seed(1602)
    lens = torch.randint(128, 2048 + 1, (64,), generator=g).tolist()
    return make_decode_case("qwen7b_gqa", 1602, lens, 28, 4, 128, "bf16", "bf16", g=g)


def _lognormal_len(g: torch.Generator, median: float, sigma: float, lo: int, hi: int) -> int:
    z = float(torch.randn((), generator=g))
    return int(min(hi, max(lo, round(math.exp(math.log(median) + sigma * z)))))


def mha13b_config() -> DecodeCase:
    """13B-shaped MHA batch: 256 lognormal lengths, 64 sequences share a 1024-token prefix."""
    g = torch.Generator().manual_seed(1603)
    lens = [_lognormal_len(g, 512.0, 1.0, 16, 8192) for _ in range(256)]
    sharers = sorted(torch.randperm(256, generator=g)[:64].tolist())
    for i in sharers:                     # redraw conditioned on L > 1024 ("then diverge")
        L = _lognormal_len(g, 512.0, 1.0, 16, 8192)
        while L <= 1024:
            L = _lognormal_len(g, 512.0, 1.0, 16, 8192)
        lens[i] = L
    share = {i: (sharers[0], 64) for i in sharers[1:]}
    case = make_decode_case("mha13b", 1603, lens, 40, 40, 128, "f16", "f16", share=share, g=g)
    case.meta["sharers"] = sharers
    return case


LONG_LENS = [32768, 49152, 65536, 81920, 98304, 114688, 131072, 131072]


def long_splitkv_config() -> DecodeCase:
    """Long-context split-KV decode over an e4m3 cache, 512-token partitions, no write."""
    return make_decode_case("long_splitkv", 1604, LONG_LENS, 32, 8, 128, "bf16", "e4m3",
                            write=False, partition_size=512)


def mixed_config() -> DecodeCase:
    """512-token chunk at positions 3584..4095 + 128 decode sequences + 64 CoW pairs."""
    g = torch.Generator().manual_seed(1605)
    lens = torch.randint(256, 4096 + 1, (128,), generator=g).tolist()
    return make_decode_case("mixed", 1605, lens, 28, 4, 128, "bf16", "bf16",
                            chunk=(3584, 512), copy_pairs=64, g=g)


CONFIG_BUILDERS = {
    1: tiny_config,
    2: qwen7b_gqa_config,
    3: mha13b_config,
    4: long_splitkv_config,
    5: mixed_config,
}
