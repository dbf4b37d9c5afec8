"""KV write and copy-on-write block copy as plain array assignments — test infrastructure only.

Sources:

* "PagedAttention: manage the KV cache like virtual memory", §3.3: in a decode step
  each new token fills the current last block of its sequence; a prefill chunk's
  tokens are written to the cache as well ("Lecture 33", §4.2).
* "Lecture 33 — KV Cache management", §2.2 (slot = physical block * block_size +
  offset) and §2.4 (copy-on-write: the writer gets a new block holding a copy of the
  shared block's contents); §5.2 (swapping: a preempted sequence's blocks are copied to
  host memory and later copied back).

Reading where the pages are silent: a negative slot marks a padding token and is
skipped.  Caches are the stored codes, layout ``[num_blocks, num_kv_heads,
block_size, head_dim]``; the functions return modified copies.
"""
from __future__ import annotations

from typing import Sequence, Tuple

import numpy as np


def kv_write(k_cache: np.ndarray, v_cache: np.ndarray, k_new: np.ndarray, v_new: np.ndarray,
             slot_mapping: Sequence[int]) -> Tuple[np.ndarray, np.ndarray]:
    """Token t's rows ``k_new[t, h, :]`` go to ``cache[slot // B, h, slot % B, :]`` for every kv head."""
    k_out, v_out = k_cache.copy(), v_cache.copy()
    block_size = k_cache.shape[2]
    for t, slot in enumerate(slot_mapping):
        slot = int(slot)
        if slot < 0:
            continue
        blk, off = slot // block_size, slot % block_size
        k_out[blk, :, off, :] = k_new[t]
        v_out[blk, :, off, :] = v_new[t]
    return k_out, v_out


def copy_blocks(k_cache: np.ndarray, v_cache: np.ndarray,
                pairs: Sequence[Tuple[int, int]]) -> Tuple[np.ndarray, np.ndarray]:
    """For each (src, dst): the whole physical block ``dst`` becomes a copy of block ``src``.

    The pairs must not chain (no dst is also a src), so the order does not matter.
    """
    srcs = {int(s) for s, _ in pairs}
    assert not any(int(d) in srcs for _, d in pairs), "a dst block is also a src"
    k_out, v_out = k_cache.copy(), v_cache.copy()
    for src, dst in pairs:
        k_out[int(dst)] = k_cache[int(src)]
        v_out[int(dst)] = v_cache[int(src)]
    return k_out, v_out


def swap_blocks(dst_k: np.ndarray, dst_v: np.ndarray, src_k: np.ndarray, src_v: np.ndarray,
                pairs: Sequence[Tuple[int, int]]) -> Tuple[np.ndarray, np.ndarray]:
    """For each (src, dst): block ``dst`` of the destination pool becomes a copy of block
    ``src`` of the source pool (the two pools share the block layout; one of them is the
    host swap space).  No dst may repeat."""
    dsts = [int(d) for _, d in pairs]
    assert len(set(dsts)) == len(dsts), "a dst block repeats"
    k_out, v_out = dst_k.copy(), dst_v.copy()
    for src, dst in pairs:
        k_out[int(dst)] = src_k[int(src)]
        v_out[int(dst)] = src_v[int(src)]
    return k_out, v_out
