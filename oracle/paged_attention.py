"""Paged-KV attention in float64, by its plain definition — test infrastructure only.

Sources (page titles and sections):

* "Lecture 33 — KV Cache management: PagedAttention, Continuous Batching, Chunked
  Prefill", §2.2 (block table address translation: token t lives in physical block
  ``block_table[t // block_size]`` at slot ``t % block_size``; the pool is one tensor
  indexed by physical block then kv head), §2.3 (decode: per sequence and head, walk
  the sequence's blocks, QK^T, softmax, weighted sum of V; no gather copy), §4.2
  (a prefill chunk attends the cached earlier chunks as history plus itself, masked
  causally), §8.1 row 1 (paging changes addressing only; the arithmetic is exactly
  standard attention).
* "PagedAttention: manage the KV cache like virtual memory", §6 (the attention
  result with paging is the same as with contiguous KV) and §9 (GQA shrinks the
  per-token KV: query heads share kv heads).

Readings where the pages are silent:

* GQA grouping: query head ``h`` reads kv head ``h // (num_heads // num_kv_heads)``.
* fp8 caches dequantise as ``e4m3_value * scale[kv_head]`` (one fp32 scale per kv head,
  separate for K and V).
* ``context_len == 0`` gives an all-zero output (and a -inf log-sum-exp).

The cache arrays are the stored codes (uint16 for fp16/bf16, uint8 for e4m3) with
layout ``[num_blocks, num_kv_heads, block_size, head_dim]``; only the rows a
sequence owns are decoded.  No online softmax, no partitions, no blocking: the
score vector of a whole sequence is formed and normalised at once.
"""
from __future__ import annotations

import math
from typing import Iterable, List, Optional, Sequence, Tuple

import numpy as np

from .formats import to_f64


def slot_of_position(block_table: Sequence[int], position: int, block_size: int) -> int:
    """Slot of logical token ``position``: ``block_table[position // B] * B + position % B``."""
    return int(block_table[position // block_size]) * block_size + position % block_size


def logical_rows(cache: np.ndarray, kv_dtype: str, block_table: Sequence[int], n_tokens: int,
                 kv_head: int, scale: Optional[float] = None) -> np.ndarray:
    """Materialise a sequence's first ``n_tokens`` K (or V) rows for one kv head, in float64.

    Walks the block table one logical block at a time and copies the valid rows of
    the physical block it names.
    """
    block_size, head_dim = cache.shape[2], cache.shape[3]
    out = np.empty((n_tokens, head_dim), dtype=np.float64)
    n_blocks = -(-n_tokens // block_size)
    for b in range(n_blocks):
        phys = int(block_table[b])
        lo = b * block_size
        hi = min(n_tokens, lo + block_size)
        out[lo:hi] = to_f64(cache[phys, kv_head, : hi - lo, :], kv_dtype)
    if scale is not None:
        out *= scale
    return out


def softmax_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float) -> np.ndarray:
    """softmax(scale * q k^T) v for one query vector over n keys; zeros if n == 0."""
    if k.shape[0] == 0:
        return np.zeros(v.shape[1], dtype=np.float64)
    s = scale * (k @ q)
    p = np.exp(s - s.max())
    return (p @ v) / p.sum()


def _kv_scales(kv_dtype, k_scale, v_scale, g):
    if kv_dtype == "e4m3":
        return float(k_scale[g]), float(v_scale[g])
    return None, None


def decode_attention(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray, kv_dtype: str,
                     block_tables: Sequence[Sequence[int]], context_lens: Sequence[int], scale: float,
                     k_scale=None, v_scale=None,
                     rows: Optional[Iterable[Tuple[int, int]]] = None) -> np.ndarray:
    """One query token per sequence over its paged K/V; returns float64 ``[S, Hq, D]``.

    ``q`` is float64 ``[S, Hq, D]``.  ``rows`` restricts the work to the listed
    (sequence, query head) pairs; other outputs are left as NaN.
    """
    S, Hq, D = q.shape
    Hkv = k_cache.shape[1]
    group = Hq // Hkv
    out = np.full((S, Hq, D), np.nan)
    wanted = None if rows is None else {}
    if rows is not None:
        for (i, h) in rows:
            wanted.setdefault(i, set()).add(h)
    for i in range(S):
        if wanted is not None and i not in wanted:
            continue
        L = int(context_lens[i])
        for g in range(Hkv):
            heads = [h for h in range(g * group, (g + 1) * group)
                     if wanted is None or h in wanted[i]]
            if not heads:
                continue
            ks, vs = _kv_scales(kv_dtype, k_scale, v_scale, g)
            K = logical_rows(k_cache, kv_dtype, block_tables[i], L, g, ks)
            V = logical_rows(v_cache, kv_dtype, block_tables[i], L, g, vs)
            for h in heads:
                out[i, h] = softmax_attention(q[i, h], K, V, scale)
    return out


def decode_partials(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray, kv_dtype: str,
                    block_table: Sequence[int], context_len: int, scale: float, head: int,
                    partition_size: int, k_scale=None, v_scale=None) -> List[Tuple[float, float, np.ndarray]]:
    """Split-KV partials for one (sequence, head): per partition of ``partition_size`` tokens,
    ``m = max s``, ``l = sum exp(s - m)``, ``o = sum exp(s - m) v`` (unnormalised).

    ``q`` is the sequence's float64 query ``[Hq, D]``.
    """
    Hkv = k_cache.shape[1]
    group = q.shape[0] // Hkv
    g = head // group
    ks, vs = _kv_scales(kv_dtype, k_scale, v_scale, g)
    K = logical_rows(k_cache, kv_dtype, block_table, context_len, g, ks)
    V = logical_rows(v_cache, kv_dtype, block_table, context_len, g, vs)
    parts = []
    for lo in range(0, context_len, partition_size):
        hi = min(context_len, lo + partition_size)
        s = scale * (K[lo:hi] @ q[head])
        m = s.max()
        p = np.exp(s - m)
        parts.append((float(m), float(p.sum()), p @ V[lo:hi]))
    return parts


def merge_partials(parts: Sequence[Tuple[float, float, np.ndarray]]) -> np.ndarray:
    """Log-sum-exp merge: ``M = max m_p``; ``out = sum e^(m_p-M) o_p / sum e^(m_p-M) l_p``."""
    M = max(m for (m, _, _) in parts)
    w = [math.exp(m - M) for (m, _, _) in parts]
    num = sum(wi * o for wi, (_, _, o) in zip(w, parts))
    den = sum(wi * l for wi, (_, l, _) in zip(w, parts))
    return num / den


def prefill_chunk_attention(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray, kv_dtype: str,
                            block_table: Sequence[int], q_start: int, scale: float,
                            k_scale=None, v_scale=None,
                            rows: Optional[Iterable[int]] = None,
                            heads: Optional[Iterable[int]] = None) -> np.ndarray:
    """Causal chunk attention: query row r sits at position ``q_start + r`` and attends
    keys ``0 .. q_start + r`` (its cached history and itself); returns float64 ``[n, Hq, D]``.

    The chunk's own K/V must already be in the cache.  ``rows``/``heads`` restrict the
    work; skipped outputs are NaN.
    """
    n, Hq, D = q.shape
    Hkv = k_cache.shape[1]
    group = Hq // Hkv
    out = np.full((n, Hq, D), np.nan)
    rows = list(range(n)) if rows is None else list(rows)
    heads = list(range(Hq)) if heads is None else list(heads)
    total = q_start + (max(rows) + 1 if rows else 0)
    for g in sorted({h // group for h in heads}):
        ks, vs = _kv_scales(kv_dtype, k_scale, v_scale, g)
        K = logical_rows(k_cache, kv_dtype, block_table, total, g, ks)
        V = logical_rows(v_cache, kv_dtype, block_table, total, g, vs)
        for h in heads:
            if h // group != g:
                continue
            for r in rows:
                p = q_start + r
                out[r, h] = softmax_attention(q[r, h], K[: p + 1], V[: p + 1], scale)
    return out
