"""Host-side planning of one decode step for a batch held by the native block manager.

A caller (or the benchmark) that starts from a set of sequences whose cached tokens sit
in known physical blocks imports them into ``BlockManager`` (``pkv_bm_*``), lets it append
each sequence's new token (copy-on-write included) and exports the block tables, context
lengths and slot mapping the device calls take.  Everything here drives the C++ block
manager; no table or slot is computed in Python.

Address translation and appending follow "Lecture 33 — KV Cache management" §2.2 (logical
block -> physical block via the block table) and "PagedAttention: manage the KV cache like
virtual memory" §3.3 (each new token fills the last block, a new block is popped when it
is full).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional, Tuple

# A sequence id outside any batch, used to pop blocks for copy-on-write destinations.
SCRATCH_SEQ = 1 << 40


@dataclass
class Plan:
    """What one step gives the device calls: tables/lengths after the step, the slot of
    every new decode token, copy-on-write pairs, and (mixed steps) the prefill chunk's
    table and slots and the shared-prefix copy pairs."""
    tables: List[List[int]]
    lens: List[int]
    slots: List[int]
    cows: List[Tuple[int, int]]
    chunk_table: Optional[List[int]] = None
    chunk_slots: List[int] = field(default_factory=list)
    share_pairs: List[Tuple[int, int]] = field(default_factory=list)


def max_blocks_of(case) -> int:
    """Table width that holds every sequence after the step (and the prefill chunk)."""
    mb = max([-(-(L + 1) // case.block_size) for L in case.context_lens] + [1])
    if case.chunk is not None:
        mb = max(mb, -(-(case.chunk.prefix_len + case.chunk.q_len) // case.block_size))
    return mb


def import_all(bm, case) -> None:
    """Hands every sequence's cached blocks to the block manager (sequence ids 0..S-1; the
    prefill chunk's sequence is S)."""
    for i, (blocks, L) in enumerate(zip(case.seq_blocks, case.context_lens)):
        bm.import_seq(i, blocks, L)
    if case.chunk is not None:
        bm.import_seq(case.num_seqs, case.chunk.blocks, case.chunk.prefix_len)


def product_plan(case) -> Plan:
    """Plans the step on the native block manager: decode sequences 0..S-1 append one slot
    each (in order), then the prefill chunk appends its rows, then (mixed steps) the
    shared-prefix copy pairs take blocks popped for a scratch sequence."""
    from ._binding import BlockManager
    bm = BlockManager(case.num_blocks, case.block_size)
    import_all(bm, case)
    mb = max_blocks_of(case)
    seqs = list(range(case.num_seqs))
    if case.writes:
        slots, cows, tables, lens = bm.step_decode(seqs, mb)
    else:
        slots, cows = [], []
        tables, lens = bm.export(seqs, mb)
    plan = Plan(tables, lens, slots, list(cows))
    if case.chunk is not None:
        plan.chunk_slots, ccows = bm.append_slots(case.num_seqs, case.chunk.q_len)
        plan.cows += ccows
        plan.chunk_table = bm.export([case.num_seqs], mb)[0][0]
        if case.copy_pairs:
            bm.allocate(SCRATCH_SEQ, case.copy_pairs * case.block_size)
            tab = bm.export([SCRATCH_SEQ], case.copy_pairs)[0][0]
            plan.share_pairs = list(zip(plan.chunk_table[:case.copy_pairs], tab))
    return plan


def append_slots(case, plan: Plan) -> List[int]:
    """Slot of position L - 1 of each decode sequence (L = its length after the step): the
    slots the fused append call writes."""
    bs = case.block_size
    return [plan.tables[i][(L - 1) // bs] * bs + (L - 1) % bs if L >= 1 else -1 for i, L in enumerate(plan.lens)]


def decode_tile_rows(case, plan: Plan) -> List[int]:
    """First pool row of every 16-row tile a decode call reads, in its order: sequence, kv
    head, tile.  A block of B tokens holds B / 16 tiles at rows (block * Hkv + h) * B + 16 * i."""
    bs, hkv = case.block_size, case.num_kv_heads
    rows = []
    for t, L in zip(plan.tables, plan.lens):
        ntiles = -(-L // 16)
        for h in range(hkv):
            for i in range(ntiles):
                blk = t[(16 * i) // bs]
                rows.append((blk * hkv + h) * bs + (16 * i) % bs)
    return rows
