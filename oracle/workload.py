"""The oracle's side of one synthetic step — TEST INFRASTRUCTURE ONLY.

Plans a ``synth`` workload's step on the oracle's own block-manager model and runs the
oracle's KV write and decode attention on a chosen subset of its sequences.  It reads the
synthetic tensors' stored codes directly and imports nothing from the library; the
library plans the same step with its native block manager, and the tests compare the two.

Step order (as the pages describe a decode step: "PagedAttention: manage the KV cache like
virtual memory" §3.3, each new token fills the sequence's last block; "Lecture 33 — KV
Cache management" §2.4, a shared block is copied before it is written): decode sequences
0..S-1 append one slot each, in order; then the prefill chunk appends its rows; then the
mixed step's shared-prefix copy pairs take blocks popped for a scratch sequence.
"""
from __future__ import annotations

from typing import Dict, List

import numpy as np
import torch

SCRATCH_SEQ = 1 << 40


def codes(t: torch.Tensor) -> np.ndarray:
    """Stored codes of a host tensor (uint16 for f16/bf16, uint8 for e4m3 bytes)."""
    t = t.contiguous()
    if t.dtype in (torch.float16, torch.bfloat16):
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.view(torch.uint8).numpy()


def q_f64(t: torch.Tensor) -> np.ndarray:
    """Exact float64 values of an f16/bf16 host tensor."""
    from .formats import to_f64
    return to_f64(codes(t), "bf16" if t.dtype == torch.bfloat16 else "f16")


def table_width(case) -> int:
    """Blocks a table row needs to hold every sequence after the step."""
    need = [(L + 1 + case.block_size - 1) // case.block_size for L in case.context_lens] + [1]
    if case.chunk is not None:
        need.append((case.chunk.prefix_len + case.chunk.q_len + case.block_size - 1) // case.block_size)
    return max(need)


def plan_step(case) -> Dict[str, object]:
    """Tables, lengths (after the step), slots, copy-on-write pairs and the mixed step's chunk
    table, chunk slots and shared-prefix pairs, from the oracle's block-manager model."""
    from .block_manager import BlockManagerModel
    bm = BlockManagerModel(case.num_blocks, case.block_size)
    for i, (blocks, L) in enumerate(zip(case.seq_blocks, case.context_lens)):
        bm.import_seq(i, blocks, L)
    if case.chunk is not None:
        bm.import_seq(case.num_seqs, case.chunk.blocks, case.chunk.prefix_len)
    mb = table_width(case)
    slots: List[int] = []
    cows = []
    if case.writes:
        for i in range(case.num_seqs):
            s, c = bm.append_slot(i)
            slots.append(s)
            if c is not None:
                cows.append(c)
    tables, lens = bm.export(list(range(case.num_seqs)), mb)
    step = {"tables": tables, "lens": lens, "slots": slots, "cows": cows, "chunk_table": None, "chunk_slots": [],
            "share_pairs": []}
    if case.chunk is not None:
        step["chunk_slots"], ccows = bm.append_slots(case.num_seqs, case.chunk.q_len)
        step["cows"] = cows + list(ccows)
        step["chunk_table"] = bm.export([case.num_seqs], mb)[0][0]
        if case.copy_pairs:
            bm.allocate(SCRATCH_SEQ, case.copy_pairs * case.block_size)
            step["share_pairs"] = list(zip(step["chunk_table"][:case.copy_pairs], bm.tables[SCRATCH_SEQ]))
    return step


def decode_sample(case, tables, lens, slots, seqs) -> np.ndarray:
    """The step's KV write and decode attention for the sequences in ``seqs`` only.  Their
    blocks are first gathered into a pool of their own (tables and slots renumbered), so the
    write copies only that pool.  Returns the float64 outputs [len(seqs), Hq, D]."""
    from . import cache_ops, paged_attention as pa
    bs = case.block_size
    used = sorted({b for i in seqs for b in tables[i] if b >= 0})
    new_id = {b: n for n, b in enumerate(used)}
    k, v = codes(case.k_cache)[used], codes(case.v_cache)[used]
    sub_tables = [[new_id[b] for b in tables[i] if b >= 0] for i in seqs]
    if case.writes:
        sub_slots = [new_id[slots[i] // bs] * bs + slots[i] % bs for i in seqs]
        k, v = cache_ops.kv_write(k, v, codes(case.k_new)[seqs], codes(case.v_new)[seqs], sub_slots)
    ks = case.k_scale.numpy().astype(np.float64) if case.k_scale is not None else None
    vs = case.v_scale.numpy().astype(np.float64) if case.v_scale is not None else None
    return pa.decode_attention(q_f64(case.q)[seqs], k, v, case.kv_dtype, sub_tables, [lens[i] for i in seqs],
                               case.scale, ks, vs)
