"""Runs one paged-KV step of a synthetic case on both sides and compares them.

Product side: the C++ block manager (``pkv_bm_*``) plans the step, then the CUDA calls
run it: copy_blocks for copy-on-write pairs, kv_write of the new tokens, paged_decode,
paged_prefill_chunk, and (mixed workload) a second copy_blocks of shared-prefix blocks.

Oracle side: ``oracle.block_manager`` plans the same step, ``oracle.cache_ops`` applies
it to host copies of the pool and ``oracle.paged_attention`` computes the attention in
float64.  Both sides start from the same ``synth`` tensors; nothing flows from the
product side into the oracle.

Step order (both sides): decode sequences 0..S-1 append one slot each (in order), then
the prefill chunk appends its q_len slots; copy-on-write copies; one kv_write of the
decode tokens followed by the chunk tokens; decode and chunk attention; finally the
shared-prefix copies (pairs = chunk blocks 0..n-1 -> n blocks popped for a scratch
sequence).
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Dict, List, Optional, Tuple

import numpy as np
import torch

from oracle.workload import codes, q_f64  # noqa: F401  (re-exported for the tests)
from paged_kv_cache_160_gb300.planner import (  # noqa: F401  (re-exported for the tests)
    Plan, append_slots, import_all, max_blocks_of, product_plan)

TOL = {"f16": 2e-3, "bf16": 1e-2, "e4m3": 3e-2}


def oracle_plan(case) -> Plan:
    """The same step planned on the oracle's block-manager model (oracle.workload)."""
    from oracle.workload import plan_step
    st = plan_step(case)
    return Plan(st["tables"], st["lens"], st["slots"], st["cows"], st["chunk_table"], st["chunk_slots"],
                st["share_pairs"])


# ---------------------------------------------------------------------------------------
# oracle execution
# ---------------------------------------------------------------------------------------

@dataclass
class OracleResult:
    k_cache: np.ndarray
    v_cache: np.ndarray
    k_final: np.ndarray           # after the shared-prefix copies
    v_final: np.ndarray
    decode: np.ndarray            # float64 [S, Hq, D] (NaN where not computed)
    prefill: Optional[np.ndarray]


def oracle_run(case, plan: Plan, decode_rows=None, prefill_rows=None, prefill_heads=None) -> OracleResult:
    from oracle import cache_ops, paged_attention as pa
    k = codes(case.k_cache)
    v = codes(case.v_cache)
    ks = case.k_scale.numpy().astype(np.float64) if case.k_scale is not None else None
    vs = case.v_scale.numpy().astype(np.float64) if case.v_scale is not None else None
    if plan.cows:
        k, v = cache_ops.copy_blocks(k, v, plan.cows)
    slots = list(plan.slots) + list(plan.chunk_slots)
    if slots:
        kn = [codes(case.k_new)] if case.writes else []
        vn = [codes(case.v_new)] if case.writes else []
        if case.chunk is not None:
            kn.append(codes(case.chunk.k_new)); vn.append(codes(case.chunk.v_new))
        k, v = cache_ops.kv_write(k, v, np.concatenate(kn), np.concatenate(vn), slots)
    dec = pa.decode_attention(q_f64(case.q), k, v, case.kv_dtype, plan.tables, plan.lens, case.scale, ks, vs,
                              rows=decode_rows)
    pre = None
    if case.chunk is not None:
        pre = pa.prefill_chunk_attention(q_f64(case.chunk.q), k, v, case.kv_dtype, plan.chunk_table,
                                         case.chunk.prefix_len, case.scale, ks, vs, rows=prefill_rows,
                                         heads=prefill_heads)
    kf, vf = (cache_ops.copy_blocks(k, v, plan.share_pairs) if plan.share_pairs else (k, v))
    return OracleResult(k, v, kf, vf, dec, pre)


# ---------------------------------------------------------------------------------------
# product execution
# ---------------------------------------------------------------------------------------

@dataclass
class DeviceResult:
    k_cache: torch.Tensor         # after kv_write (before the shared-prefix copies), host copy
    v_cache: torch.Tensor
    k_final: torch.Tensor
    v_final: torch.Tensor
    decode: torch.Tensor          # [S, Hq, D] host, q dtype
    prefill: Optional[torch.Tensor]
    device_error: int


def device_run(case, plan: Plan, partition_size: Optional[int] = None, keep_intermediate: bool = True,
               device: str = "cuda", run_prefill: bool = True, fused_append: bool = False,
               append_inputs: Optional[Tuple[torch.Tensor, torch.Tensor]] = None) -> DeviceResult:
    """fused_append: the decode tokens' K/V go through pkv_paged_decode_append instead of
    pkv_kv_write + pkv_paged_decode (each decode token's slot must be its sequence's last
    position).  append_inputs: the (k_new, v_new) the fused call gets, when they differ from the
    case's stored codes (f16/bf16 rows that an e4m3 cache quantises)."""
    import paged_kv_cache_160_gb300 as pkv
    if fused_append:
        assert case.writes and append_slots(case, plan) == list(plan.slots), "slots are not the last positions"
    dev = torch.device(device)
    kc = case.k_cache.to(dev)
    vc = case.v_cache.to(dev)
    ks = case.k_scale.to(dev) if case.k_scale is not None else None
    vs = case.v_scale.to(dev) if case.v_scale is not None else None
    desc = pkv.cache_desc(kc, ks, vs)
    if plan.cows:
        pkv.pkv_copy_blocks(kc, vc, desc, torch.tensor(plan.cows, dtype=torch.int32, device=dev))
    dec_writes = case.writes and not fused_append
    slots = (list(plan.slots) if dec_writes else []) + list(plan.chunk_slots)
    if slots:
        kn = [case.k_new] if dec_writes else []
        vn = [case.v_new] if dec_writes else []
        if case.chunk is not None:
            kn.append(case.chunk.k_new); vn.append(case.chunk.v_new)
        pkv.pkv_kv_write(torch.cat(kn).to(dev), torch.cat(vn).to(dev),
                         torch.tensor(slots, dtype=torch.int64, device=dev), kc, vc, desc)
    q = case.q.to(dev)
    out = torch.empty_like(q)
    tables = torch.tensor(plan.tables, dtype=torch.int32, device=dev)
    lens = torch.tensor(plan.lens, dtype=torch.int32, device=dev)
    part = case.partition_size if partition_size is None else partition_size
    max_len = max(plan.lens) if plan.lens else 0
    ws_bytes = pkv.pkv_decode_workspace_bytes(case.num_seqs, case.num_heads, case.num_kv_heads, case.head_dim,
                                              case.block_size, max_len, part)
    ws = torch.zeros(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    if fused_append:
        kn_, vn_ = append_inputs if append_inputs is not None else (case.k_new, case.v_new)
        pkv.pkv_paged_decode_append(out, q, kn_.to(dev), vn_.to(dev), kc, vc, desc, tables, lens,
                                    max_len, case.scale, part, ws)
    else:
        pkv.pkv_paged_decode(out, q, kc, vc, desc, tables, lens, max_len, case.scale, part, ws)
    pre = None
    if case.chunk is not None and run_prefill:
        cq = case.chunk.q.to(dev)
        pout = torch.empty_like(cq)
        pkv.pkv_paged_prefill_chunk(pout, cq, torch.tensor([0, case.chunk.q_len], dtype=torch.int32, device=dev),
                                    torch.tensor([case.chunk.prefix_len], dtype=torch.int32, device=dev),
                                    case.chunk.q_len, kc, vc, desc,
                                    torch.tensor([plan.chunk_table], dtype=torch.int32, device=dev), case.scale)
        pre = pout
    torch.cuda.synchronize()
    k_mid = kc.cpu() if keep_intermediate else None
    v_mid = vc.cpu() if keep_intermediate else None
    if plan.share_pairs:
        pkv.pkv_copy_blocks(kc, vc, desc, torch.tensor(plan.share_pairs, dtype=torch.int32, device=dev))
    err = pkv.pkv_get_device_error()
    return DeviceResult(k_mid, v_mid, kc.cpu(), vc.cpu(), out.cpu(), pre.cpu() if pre is not None else None, err)


def out_f64(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.float64).numpy()


def max_abs_err(got: torch.Tensor, ref: np.ndarray) -> float:
    g = out_f64(got)
    m = ~np.isnan(ref)
    if not m.any():
        return 0.0
    d = np.abs(g[m] - ref[m])
    if np.isnan(d).any():
        return math.inf
    return float(d.max())
