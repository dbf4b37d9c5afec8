"""Benchmark of the paged-KV decode step on one GB300: effective HBM GB/s and seq-tokens/s.

Headline workload: the Qwen2.5-7B-shaped GQA decode batch — 64 running sequences with
context lengths uniform in [128, 2048], 28 query heads / 4 kv heads, head_dim 128, bf16
Q/K/V, 16-token blocks in a shuffled pool ([num_blocks, 4, 16, 128], pool = blocks needed +
10%).  One step = the write of the 64 new tokens' K/V, then paged_decode over every
sequence's L + 1 tokens.  Every new token belongs at its sequence's last position, so the
write is fused into the decode call (pkv_paged_decode_append: two launches, the split-KV
decode and the log-sum-exp merge of split segments as its programmatic dependent);
kv_write + decode is timed beside it.  The step is planned once on the native block manager
(its cost is reported separately).

Timing: CUDA events on the launching stream around one CUDA graph of K steps.  Every step
uses the next of R pool copies whose combined size is above 3x the L2 size, so no step
finds its K/V in L2.  `value` is device-resident throughput.  `e2e` passes HOST buffers to
the call: every step's inputs (q, new K/V, tables, lengths) are read in place from pinned
host memory and its output is written to pinned host memory by the kernels, across
NVLink-C2C; the same steps with staged H2D/D2H copies on copy streams are reported beside it.

The same line also reports, each timed the same way:
  roofline.copy_same_size_gbs  a plain device copy moving the decode call's bytes (half read,
                               half written), rotating over the same number of buffers;
  workloads                    the decode call on the 13B MHA batch and the long-context
                               e4m3 batch;
  mixed_step                   the mixed chunked-prefill + decode step as one graph per step:
                               the 128 decodes (fused append, on 66 SMs) beside the 512 chunk
                               rows' kv_write and prefill on another stream, then copy_blocks
                               of 64 pairs (and the same work in one stream on every SM);
  prefill_chunk, cache_ops, swap_blocks, host_step: single calls;
  cpu_baseline                 the float64 oracle on the host cores, one core and all cores.

    python bench.py [--gpus 1] [--steps K] [--warmup W] [--impl reference] [--workload 2|3|4|5]

--workload picks another decode workload for the headline fields (3: 13B MHA, 4: long-context
e4m3, 5: the mixed step's decode part); the default, 2, is the headline.  The library runs on
one GPU: --gpus N > 1 (or a torchrun launch with more than one rank) prints a one-line refusal.
"""
from __future__ import annotations

import os

# The CPU baseline times the oracle with one BLAS thread per process; pin numpy's BLAS
# before it loads (spawned worker processes re-run this module's top level).
for _var in ("OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS", "OMP_NUM_THREADS"):
    os.environ.setdefault(_var, "1")

import argparse
import hashlib
import json
import math
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged-decode effective HBM GB/s (% of GB300 peak); seq-tokens attended/s"
WORKLOADS = {
    2: "qwen2.5-7b-gqa paged decode step: 64 seqs, context_lens U[128,2048] (seed 1602), "
       "28 q heads / 4 kv heads, head_dim 128, bf16, block_size 16, kv_write 64 tokens + paged_decode",
    3: "13b-mha paged decode step: 256 seqs, lognormal context_lens (median 512, clipped to [16,8192], "
       "seed 1603), 64 sharing a 1024-token prefix, 40/40 heads, head_dim 128, fp16, kv_write 256 tokens "
       "+ paged_decode",
    4: "long-context split-KV decode: 8 seqs of 32K..128K tokens (704,512 in all), 32 q heads / 8 kv heads, "
       "head_dim 128, bf16 q, e4m3 KV with per-head scales, 512-token partitions, paged_decode only",
    5: "mixed step's decode part: 128 seqs, context_lens U[256,4096] (seed 1605), 28/4 heads, head_dim 128, "
       "bf16, kv_write 128 tokens + paged_decode (its 512-row chunk is the prefill_chunk line)",
}
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0

# DRAM bytes per decode call on the headline workload (paged_decode_kernel +
# split_kv_merge_kernel, dram__bytes_read.sum + dram__bytes_write.sum of one call in one ncu
# capture; ncu flushes the caches before each kernel, so the merge's reads of the
# partials count as DRAM reads), valid only for the kernel source with this hash; when the
# source changes, traffic is reported as null until re-measured.
TRAFFIC = {"source_sha1": "99b29df5523fdb6f246d2e32cb6d75fc16dafa77", "bytes_per_launch": 161419264}


def _src_hash() -> str:
    h = hashlib.sha1()
    for f in ("paged_decode.cu", "pkv_device.cuh"):
        h.update(open(os.path.join(ROOT, "paged_kv_cache_160_gb300", "csrc", f), "rb").read())
    return h.hexdigest()


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def _bf16_peak():
    """Measured dense bf16 TFLOP/s (burst: the prefill kernel is timed alone)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        return float(json.load(open(path))["bf16_tflops"]), "measured"
    return FALLBACK_BF16_TFLOPS, "fallback"


def _world():
    return int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0"))


def refuse_multi_gpu(args) -> bool:
    """The library and its benchmark run on one GPU.  Under --gpus N > 1 or a multi-rank
    launch, rank 0 prints one refusal line; every rank exits without GPU work."""
    world, rank = _world()
    if args.gpus == 1 and world == 1:
        return False
    if rank == 0:
        print(json.dumps({"metric": METRIC, "impl": args.impl, "n_gpus": max(args.gpus, world),
                          "unavailable": "single-GPU library: the decode path runs on one GPU and has no "
                                         "multi-GPU mode; run with --gpus 1"}))
    return True


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.25)
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        mhz, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                mhz.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not mhz:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(mhz)}


# ---------------------------------------------------------------------------------------
# algorithmic work
# ---------------------------------------------------------------------------------------

def workload_bytes(case, plan):
    """Algorithmic bytes of one decode step: each unique attended K/V row once (K and V), q
    and out, one table entry per 16-token tile and one length per sequence; and the step's
    write (new rows read and written, plus their slots).  Returns (decode, write, tokens)."""
    Hkv, D, Hq, bs = case.num_kv_heads, case.head_dim, case.num_heads, case.block_size
    kv_elt = 1 if case.kv_dtype == "e4m3" else 2
    q_elt = 2
    unique_rows = set()
    for t, L in zip(plan.tables, plan.lens):
        for j in range(L):
            unique_rows.add(t[j // bs] * bs + j % bs)
    n_rows = len(unique_rows)
    ntiles = sum(-(-L // 16) for L in plan.lens)
    S = case.num_seqs
    decode = 2 * n_rows * Hkv * D * kv_elt + 2 * S * Hq * D * q_elt + 4 * ntiles + 4 * S
    T = len(plan.slots)
    write = 2 * 2 * T * Hkv * D * kv_elt + 8 * T
    return decode, write, sum(plan.lens)


def prefill_work(case, plan):
    """The mixed step's prefill chunk: FLOPs = 4 * head_dim * (attended query-key pairs) * heads;
    bytes = the chunk sequence's K/V rows once, its q and out, its table row."""
    ch = case.chunk
    Hkv, D, Hq = case.num_kv_heads, case.head_dim, case.num_heads
    pairs = sum(ch.prefix_len + r + 1 for r in range(ch.q_len))
    flops = 4 * D * pairs * Hq
    rows = ch.prefix_len + ch.q_len
    nbytes = 2 * rows * Hkv * D * 2 + 2 * ch.q_len * Hq * D * 2 + 4 * len(plan.chunk_table)
    return flops, nbytes


# SMs the mixed step's decodes run on, beside the prefill chunk on the others.  Measured on
# this step (decodes alone / the two-stream step, us): every SM 92 / 131; 88: 91 / 119;
# 72: 93 / 110; 64: 100 / 107; 56: 112 / 116; and the two-stream step alone at 60-70 SMs:
# 60: 110; 62: 108-109; 64: 107; 66: 105.6; 68: 106-107; 70: 107.  Below 72 SMs the decodes
# no longer saturate HBM; above about 66 the prefill's 128 CTAs get too few SMs.
MIXED_DECODE_SMS = 66


def mixed_step_work(case, plan):
    """Bytes and FLOPs of the whole mixed step: the kv_write of every new row (decode tokens
    and chunk rows), the decode attention, the prefill chunk and the copy-on-write pairs."""
    Hkv, D = case.num_kv_heads, case.head_dim
    decode, _, tokens = workload_bytes(case, plan)
    T = len(plan.slots) + len(plan.chunk_slots)
    write = 2 * 2 * T * Hkv * D * 2 + 8 * T
    pf_flops, pf_bytes = prefill_work(case, plan)
    block_bytes = Hkv * case.block_size * D * 2
    copy = 2 * 2 * len(plan.share_pairs) * block_bytes + 8 * len(plan.share_pairs)
    dec_flops = 4 * D * tokens * case.num_heads
    return {"decode_bytes": decode, "write_bytes": write, "prefill_bytes": pf_bytes, "copy_bytes": copy,
            "bytes": decode + write + pf_bytes + copy, "prefill_flops": pf_flops, "decode_flops": dec_flops,
            "flops": pf_flops + dec_flops, "tokens": tokens}


# ---------------------------------------------------------------------------------------
# timing helpers
# ---------------------------------------------------------------------------------------

def graph_ms(stream, fn, n_calls: int, warm_calls: int) -> float:
    """Average ms per call of fn(k) for k = 0..n_calls-1, captured as one CUDA graph and
    replayed between two events.  Before that: warm_calls eager calls (the library's
    per-device state exists before capture) and one untimed replay of the same graph (a
    graph's first launch also uploads it to the device)."""
    import torch
    with torch.cuda.stream(stream):
        for k in range(max(2, warm_calls)):
            fn(k)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
        for k in range(n_calls):
            fn(warm_calls + k)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        g.replay()
        a.record(stream)
        g.replay()
        b.record(stream)
    stream.synchronize()
    return a.elapsed_time(b) / n_calls


def rotation(case, l2: int) -> int:
    """Pool copies to rotate over so that their combined size exceeds 3x L2."""
    pool_bytes = 2 * case.k_cache.numel() * case.k_cache.element_size()
    return max(1, math.ceil(3 * l2 / pool_bytes) + 1) if pool_bytes < 3 * l2 else 1


def device_case(pkv, case, dev, R):
    import torch
    kcs = [case.k_cache.to(dev) for _ in range(R)]
    vcs = [case.v_cache.to(dev) for _ in range(R)]
    ks = case.k_scale.to(dev) if case.k_scale is not None else None   # e4m3 caches: per-head scales
    vs = case.v_scale.to(dev) if case.v_scale is not None else None
    descs = [pkv.cache_desc(k, ks, vs) for k in kcs]
    return kcs, vcs, descs


# ---------------------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------------------

def run_gpu(args):
    import torch

    import paged_kv_cache_160_gb300 as pkv
    import synth
    from paged_kv_cache_160_gb300.planner import append_slots, decode_tile_rows, product_plan

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)

    case = synth.CONFIG_BUILDERS[args.workload]()
    t0 = time.perf_counter()
    plan = product_plan(case)
    host_plan_us = (time.perf_counter() - t0) * 1e6
    decode_bytes, write_bytes, tokens = workload_bytes(case, plan)
    step_bytes = decode_bytes + write_bytes

    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 0) or 132 * 1024 * 1024
    pool_bytes = 2 * case.k_cache.numel() * case.k_cache.element_size()
    R = max(2, math.ceil(3 * l2 / pool_bytes) + 1)
    kcs, vcs, descs = device_case(pkv, case, dev, R)
    q = case.q.to(dev)
    k_new = case.k_new.to(dev) if case.writes else None
    v_new = case.v_new.to(dev) if case.writes else None
    slots = torch.tensor(plan.slots, dtype=torch.int64, device=dev)
    tables = torch.tensor(plan.tables, dtype=torch.int32, device=dev)
    lens = torch.tensor(plan.lens, dtype=torch.int32, device=dev)
    out = torch.empty_like(q)
    max_len = max(plan.lens)
    part = case.partition_size
    wsb = pkv.pkv_decode_workspace_bytes(case.num_seqs, case.num_heads, case.num_kv_heads, case.head_dim,
                                         case.block_size, max_len, part)
    ws = torch.zeros(wsb, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)

    # Every decode token goes to its sequence's last position, so the step's write is fused
    # into the decode call (pkv_paged_decode_append); the unfused pair is timed beside it.
    fused = case.writes and append_slots(case, plan) == list(plan.slots)

    def write(r):
        if case.writes:
            pkv.pkv_kv_write(k_new, v_new, slots, kcs[r], vcs[r], descs[r], stream)

    def decode(r):
        pkv.pkv_paged_decode(out, q, kcs[r], vcs[r], descs[r], tables, lens, max_len, case.scale, part, ws, stream)

    def step(r, fuse=fused):
        if fuse:
            pkv.pkv_paged_decode_append(out, q, k_new, v_new, kcs[r], vcs[r], descs[r], tables, lens, max_len,
                                        case.scale, part, ws, stream)
        else:
            write(r)
            decode(r)

    # eager warm-up (also initialises the library's per-device state before capture)
    with torch.cuda.stream(stream):
        for r in range(R):
            step(r, False)
            step(r)
    stream.synchronize()
    assert pkv.pkv_get_device_error(stream) == 0
    K, W = args.steps, args.warmup

    # The timed loop is one CUDA graph of K steps (each: the fused append + decode -> split-KV
    # merge, or kv_write -> decode -> merge, launched as programmatic dependents), rotating over
    # the pool copies.
    def capture(n_steps, first, kind="step"):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
            for k in range(n_steps):
                r = (first + k) % R
                if kind == "step":
                    step(r)
                elif kind == "unfused":
                    step(r, False)
                else:
                    decode(r)
        return g

    g_warm = capture(W, 0)
    g_timed = capture(K, W)
    g_unf = capture(K, W, kind="unfused") if fused else None
    torch.cuda.synchronize(dev)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    # W warm-up steps, then one untimed replay of the timed graph itself (a graph's first
    # launch also uploads it to the device), then the timed replay.
    with torch.cuda.stream(stream):
        g_warm.replay()
        g_timed.replay()
    stream.synchronize()
    with ClockSampler(0) as clk:
        with torch.cuda.stream(stream):
            start.record(stream)
            g_timed.replay()
            end.record(stream)
        stream.synchronize()
        # The decode call alone, for its roofline: the step's call when the write is fused
        # (it is the whole step), else decode + merge without the write.
        if fused:
            dec_avg_ms = None
        else:
            dec_avg_ms = graph_ms(stream, lambda k: decode(k % R), K, W)
        unfused_ms = None
        if g_unf is not None:
            u_start, u_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                g_unf.replay()
                u_start.record(stream)
                g_unf.replay()
                u_end.record(stream)
            stream.synchronize()
            unfused_ms = u_start.elapsed_time(u_end) / K
    elapsed_ms = start.elapsed_time(end)
    if dec_avg_ms is None:
        dec_avg_ms = elapsed_ms / K
    assert pkv.pkv_get_device_error(stream) == 0

    # The same-size ceiling: a plain device copy moving the decode call's bytes (half read,
    # half written), rotating over R buffer pairs, one graph of K copies.
    roof_bytes = step_bytes if fused else decode_bytes        # the fused call also moves the new rows
    half = (roof_bytes // 2) & ~4095                          # whole 4 KiB pages: the copy's fast path
    src = [torch.empty(half, dtype=torch.uint8, device=dev).fill_(1) for _ in range(R)]
    dst = [torch.empty(half, dtype=torch.uint8, device=dev) for _ in range(R)]
    copy_ms = graph_ms(stream, lambda k: dst[k % R].copy_(src[k % R]), K, W)
    copy_gbs = 2 * half / (copy_ms * 1e-3) / 1e9
    del src, dst
    # The decode's own memory ceiling: the same K/V tiles read by the same kind of pipeline
    # (pkv_stream_tiles: persistent grid, 12 warps x 2 bulk-copy stages per SM), no compute.
    tile_rows = decode_tile_rows(case, plan)
    rows_t = torch.tensor(tile_rows, dtype=torch.int32, device=dev)
    csum = torch.zeros(1, dtype=torch.int32, device=dev)
    stream_ms = graph_ms(stream, lambda k: pkv.pkv_stream_tiles(kcs[k % R], vcs[k % R], descs[k % R], rows_t, csum,
                                                                stream), K, W)
    tile_read_bytes = 2 * len(tile_rows) * 16 * case.head_dim * (1 if case.kv_dtype == "e4m3" else 2)
    assert pkv.pkv_get_device_error(stream) == 0

    # ---- end to end, staged: explicit copies on copy streams --------------------------------
    host_parts = [case.q, torch.tensor(plan.tables, dtype=torch.int32), torch.tensor(plan.lens, dtype=torch.int32)]
    if case.writes:
        host_parts += [case.k_new, case.v_new]
        if not fused:
            host_parts.append(torch.tensor(plan.slots, dtype=torch.int64))
    offs, pos = [], 0
    for t in host_parts:
        offs.append(pos)
        pos += -(-t.numel() * t.element_size() // 256) * 256
    h_in = torch.zeros(pos, dtype=torch.uint8).pin_memory()
    for t, o in zip(host_parts, offs):
        h_in[o:o + t.numel() * t.element_size()] = t.contiguous().view(-1).view(torch.uint8)
    d_in = [torch.empty(pos, dtype=torch.uint8, device=dev) for _ in range(2)]

    def views(buf):
        return [buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape) for t, o in zip(host_parts, offs)]

    dv = [views(d_in[i]) for i in range(2)]
    outs = [torch.empty_like(out) for _ in range(2)]
    h_outs = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host_parts)
    d2h = h_outs[0].numel() * h_outs[0].element_size()
    up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def e2e_graph(n_steps, first):
        """n_steps serving steps captured in one graph: per step, the H2D of the staged
        inputs (upload stream), the step's kernels, and the D2H of its output (download
        stream), with events giving the double-buffer order."""
        g = torch.cuda.CUDAGraph()
        evs = []
        with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
            fork = torch.cuda.Event()
            fork.record(stream)
            up.wait_event(fork)
            down.wait_event(fork)
            for k in range(n_steps):
                i, r = k % 2, (first + k) % R
                in_ready, step_done, out_copied = torch.cuda.Event(), torch.cuda.Event(), torch.cuda.Event()
                if k >= 2:
                    up.wait_event(evs[k - 2][1])             # step k-2 no longer reads buffer i
                with torch.cuda.stream(up):
                    d_in[i].copy_(h_in, non_blocking=True)
                    in_ready.record(up)
                stream.wait_event(in_ready)
                if k >= 2:
                    stream.wait_event(evs[k - 2][2])         # step k-2's output has been read back
                qi, tbi, lni = dv[i][:3]
                if fused:
                    kni, vni = dv[i][3:5]
                    pkv.pkv_paged_decode_append(outs[i], qi, kni, vni, kcs[r], vcs[r], descs[r], tbi, lni, max_len,
                                                case.scale, part, ws, stream)
                else:
                    if case.writes:
                        kni, vni, sli = dv[i][3:]
                        pkv.pkv_kv_write(kni, vni, sli, kcs[r], vcs[r], descs[r], stream)
                    pkv.pkv_paged_decode(outs[i], qi, kcs[r], vcs[r], descs[r], tbi, lni, max_len, case.scale,
                                         part, ws, stream)
                step_done.record(stream)
                down.wait_event(step_done)
                with torch.cuda.stream(down):
                    h_outs[i].copy_(outs[i], non_blocking=True)
                    out_copied.record(down)
                evs.append((in_ready, step_done, out_copied))
            for ev in evs[-2:]:
                stream.wait_event(ev[2])
            join = torch.cuda.Event()
            join.record(up)
            stream.wait_event(join)
        return g

    g_e2e_warm = e2e_graph(W, 0)
    g_e2e = e2e_graph(K, W)
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        g_e2e_warm.replay()
        g_e2e.replay()
        e_start.record(stream)
        g_e2e.replay()
        e_end.record(stream)
    stream.synchronize()
    staged_ms = e_start.elapsed_time(e_end)
    for i in range(2):
        assert torch.equal(h_outs[i], out.cpu())

    # Zero-copy (the headline e2e): the step's inputs sit in pinned host buffers that are
    # passed to the call itself, and the kernels write the output straight into pinned host
    # memory; Grace reaches both over NVLink-C2C, so every step still moves its input and
    # output bytes across the host link, with no copy node breaking the programmatic launches.
    # Two buffer sets alternate, as a serving loop's host would fill one while the other is read.
    zero_copy = fused or not case.writes
    if zero_copy:
        hsets = []
        for _ in range(2):
            hs = {"q": case.q.clone().pin_memory(), "tb": torch.tensor(plan.tables, dtype=torch.int32).pin_memory(),
                  "ln": torch.tensor(plan.lens, dtype=torch.int32).pin_memory(),
                  "out": torch.empty(out.shape, dtype=out.dtype).pin_memory()}
            if case.writes:
                hs["kn"], hs["vn"] = case.k_new.clone().pin_memory(), case.v_new.clone().pin_memory()
            hsets.append(hs)

        def zc_call(k):
            hs, r = hsets[k % 2], k % R
            if fused:
                pkv.pkv_paged_decode_append(hs["out"], hs["q"], hs["kn"], hs["vn"], kcs[r], vcs[r], descs[r],
                                            hs["tb"], hs["ln"], max_len, case.scale, part, ws, stream)
            else:
                pkv.pkv_paged_decode(hs["out"], hs["q"], kcs[r], vcs[r], descs[r], hs["tb"], hs["ln"],
                                     max_len, case.scale, part, ws, stream)

        e2e_ms = graph_ms(stream, zc_call, K, W) * K
        for hs in hsets:
            assert torch.equal(hs["out"], out.cpu())
    else:
        e2e_ms = staged_ms
    del d_in, outs, h_outs
    pf_ms, pf_flops = prefill_measure(dev)
    cache_ops = cache_ops_measure(pkv, case, plan, kcs[0], vcs[0], descs[0], k_new, v_new, slots, write_bytes,
                                  stream) if case.writes else None
    sw_out, sw_in, sw_bytes, sw_link = swap_measure(dev)
    host_step = host_step_measure(case) if case.writes else None
    del kcs, vcs, descs
    torch.cuda.empty_cache()

    peak, peak_kind = _peaks()
    bf16_peak, bf16_kind = _bf16_peak()
    others = {}
    mixed = None
    if args.workload == 2 and not args.headline_only:
        for n in (3, 4):
            others[str(n)] = decode_call_measure(n, dev, l2, stream, peak, K, W)
        mixed = mixed_step_measure(dev, l2, stream, K, W, peak, bf16_peak)

    ms_per_step = elapsed_ms / K
    value = step_bytes / (ms_per_step * 1e-3) / 1e9
    achieved = roof_bytes / (dec_avg_ms * 1e-3) / 1e9
    traffic = (TRAFFIC["bytes_per_launch"] if args.workload == 2 and TRAFFIC["source_sha1"] == _src_hash()
               else None)
    launches_per_step = 3 if case.writes and not fused else 2      # (kv_write,) decode, merge
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": 1,
        "steps": K,
        "warmup": W,
        "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3-kv/bf16" if case.kv_dtype == "e4m3" else case.kv_dtype,
        "data": "synthetic (seeded N(0,1) Q/K/V, shuffled physical block ids)",
        "config": {"workload": WORKLOADS[args.workload], "num_seqs": case.num_seqs, "attended_tokens": tokens,
                   "step_bytes": step_bytes, "decode_bytes": decode_bytes, "kv_write_bytes": write_bytes,
                   "pool_copies": R, "l2": f"rotating {R} pool copies ({R * pool_bytes / 1e6:.0f} MB > 3x L2)",
                   "launch": ("one CUDA graph of K steps (fused kv write + decode, then merge, per step; "
                              "programmatic dependent launches)" if fused else
                              "one CUDA graph of K steps (kv_write, decode, merge per step; programmatic "
                              "dependent launches)"),
                   "step_kind": "pkv_paged_decode_append + merge" if fused else
                                ("pkv_kv_write + pkv_paged_decode + merge" if case.writes else
                                 "pkv_paged_decode + merge"),
                   "partition_size": part,
                   "untimed_graph_replays": "the timed K-step graph is replayed once untimed after the W warm-up "
                                            "steps (a graph's first launch also uploads it)",
                   "parallelism": "single GPU"},
        "seq_tokens_per_s": round(tokens / (ms_per_step * 1e-3), 1),
        "pct_of_nominal_8tbs": round(100 * value / NOMINAL_HBM_GBS, 2),
        "pct_of_measured_copy": round(100 * value / peak, 2),
        "roofline": {"kernel": "paged_decode_append (decode + merge)" if fused else "paged_decode (decode + merge)",
                     "bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "peak_kind": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_kind == "measured" else "fallback 6.8 TB/s",
                     "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                     "algorithmic_bytes_per_launch": roof_bytes, "avg_launch_ms": round(dec_avg_ms, 5),
                     "frac_of_nominal_8tbs": round(achieved / NOMINAL_HBM_GBS, 4),
                     "copy_same_size_gbs": round(copy_gbs, 1),
                     "copy_same_size_ms": round(copy_ms, 5),
                     "frac_of_copy_same_size": round(achieved / copy_gbs, 4),
                     "copy_same_size_what": f"device copy of {half} B into {half} B (the call's bytes, half read "
                                            f"and half written, rounded down to 4 KiB), rotating over {R} buffer "
                                            "pairs, one graph of K copies",
                     "tile_stream_ms": round(stream_ms, 5),
                     "tile_stream_gbs": round(tile_read_bytes / (stream_ms * 1e-3) / 1e9, 1),
                     "frac_of_tile_stream": round(stream_ms / dec_avg_ms, 4),
                     "tile_stream_what": f"pkv_stream_tiles over the call's {len(tile_rows)} K/V tiles "
                                         f"({tile_read_bytes} B): the decode's memory pipeline with no compute, "
                                         "same rotation, one graph of K calls"},
        "e2e": {"value": round(step_bytes / (e2e_ms / K * 1e-3) / 1e9, 1), "unit": "GB/s",
                "ms_per_step": round(e2e_ms / K, 5), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "copies": ("the call gets HOST buffers: each step's inputs (q, new K/V, tables, lengths) are "
                           "read in place from pinned host memory and its output is written to pinned host "
                           "memory by the kernels (NVLink-C2C); two buffer sets alternate; the K steps are "
                           "one CUDA graph") if zero_copy else
                          ("per step one H2D of the pinned staged inputs and one D2H of the output, on two copy "
                           "streams ordered by events; double-buffered; the K steps are one CUDA graph"),
                "staged_copies": {"value": round(step_bytes / (staged_ms / K * 1e-3) / 1e9, 1),
                                  "ms_per_step": round(staged_ms / K, 5),
                                  "what": "the same steps with explicit H2D/D2H copies on two copy streams, "
                                          "ordered by events (double-buffered), in one CUDA graph"}},
        "workloads": others or None,
        "mixed_step": mixed,
        "prefill_chunk": {"workload": "mixed-step chunk: 512 causal rows at 3584..4095, 28/4 heads, bf16",
                          "bound": "tensor", "achieved": round(pf_flops / (pf_ms * 1e-3) / 1e12, 1),
                          "peak": bf16_peak, "peak_kind": f"{bf16_kind} bf16 burst (MEASURED_PEAKS.json)",
                          "unit": "TFLOP/s",
                          "frac": round(pf_flops / (pf_ms * 1e-3) / 1e12 / bf16_peak, 4),
                          "avg_launch_ms": round(pf_ms, 5), "flops_per_launch": pf_flops},
        "swap_blocks": {"workload": "4096 scattered blocks of the 7B layout (K and V), device <-> pinned host",
                        "bytes_per_call": sw_bytes, "device_to_host_gbs": round(sw_out, 1),
                        "host_to_device_gbs": round(sw_in, 1),
                        "contiguous_copy_gbs": {"device_to_host": round(sw_link[0], 1),
                                                "host_to_device": round(sw_link[1], 1)}},
        "cache_ops": cache_ops,
        "host_plan_us": round(host_plan_us, 1),
        "host_step": host_step,
        "gpu_launches": launches_per_step * K,
        "unfused_step": None if unfused_ms is None else {
            "ms_per_step": round(unfused_ms, 5), "value": round(step_bytes / (unfused_ms * 1e-3) / 1e9, 1),
            "what": "the same step as pkv_kv_write + pkv_paged_decode (3 launches), one graph of K steps"},
        "clocks": clk.summary(),
    }
    line["cpu_baseline"] = cpu_baseline(args.workload, case, plan, args.cpu_budget)
    print(json.dumps(line))


def decode_call_measure(n, dev, l2, stream, peak, K, W):
    """The decode call (the step's call: fused append when the step writes, else decode +
    merge) on workload n, rotating pool copies when the pool is smaller than 3x L2."""
    import torch
    import paged_kv_cache_160_gb300 as pkv
    import synth
    from paged_kv_cache_160_gb300.planner import append_slots, product_plan
    case = synth.CONFIG_BUILDERS[n]()
    plan = product_plan(case)
    decode_bytes, write_bytes, tokens = workload_bytes(case, plan)
    R = rotation(case, l2)
    kcs, vcs, descs = device_case(pkv, case, dev, R)
    del case.k_cache, case.v_cache
    q = case.q.to(dev)
    out = torch.empty_like(q)
    tables = torch.tensor(plan.tables, dtype=torch.int32, device=dev)
    lens = torch.tensor(plan.lens, dtype=torch.int32, device=dev)
    max_len = max(plan.lens)
    part = case.partition_size
    ws = torch.zeros(pkv.pkv_decode_workspace_bytes(case.num_seqs, case.num_heads, case.num_kv_heads,
                                                    case.head_dim, case.block_size, max_len, part),
                     dtype=torch.uint8, device=dev)
    fused = case.writes and append_slots(case, plan) == list(plan.slots)
    k_new = case.k_new.to(dev) if fused else None
    v_new = case.v_new.to(dev) if fused else None

    def call(k):
        r = k % R
        if fused:
            pkv.pkv_paged_decode_append(out, q, k_new, v_new, kcs[r], vcs[r], descs[r], tables, lens, max_len,
                                        case.scale, part, ws, stream)
        else:
            pkv.pkv_paged_decode(out, q, kcs[r], vcs[r], descs[r], tables, lens, max_len, case.scale, part, ws,
                                 stream)

    n_calls = max(5, min(K, 40)) if decode_bytes > 1e9 else K
    ms = graph_ms(stream, call, n_calls, max(3, min(W, 5)))
    assert pkv.pkv_get_device_error(stream) == 0
    nbytes = decode_bytes + (write_bytes if fused else 0)
    res = {"workload": WORKLOADS[n], "call": "pkv_paged_decode_append + merge" if fused else
           "pkv_paged_decode + merge", "bytes_per_call": nbytes, "attended_tokens": tokens,
           "ms_per_call": round(ms, 5), "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1),
           "frac": round(nbytes / (ms * 1e-3) / 1e9 / peak, 4),
           "seq_tokens_per_s": round(tokens / (ms * 1e-3), 1), "calls_timed": n_calls,
           "l2": f"rotating {R} pool copies" if R > 1 else "one pool copy larger than 3x L2"}
    del kcs, vcs, descs
    torch.cuda.empty_cache()
    return res


def mixed_step_measure(dev, l2, stream, K, W, peak, bf16_peak):
    """The mixed chunked-prefill + decode step: 128 decode tokens and a 512-row chunk at
    positions 3584..4095 (640 new rows), then copy_blocks of the 64 shared-prefix pairs.
    The decodes are HBM-bound and the chunk's prefill tensor-bound, and neither reads what the
    other writes, so they run side by side:
    - this stream: pkv_paged_decode_append of the 128 sequences (their new rows written in the
      same call) under an SM budget of MIXED_DECODE_SMS, then its merge;
    - a second stream: pkv_kv_write of the chunk's 512 rows, then pkv_paged_prefill_chunk,
      whose 128 CTAs take the other SMs;
    - joined, then copy_blocks.
    K steps in one graph, rotating pool copies.  serial_ms_per_step times the same work in one
    stream on every SM: kv_write of the 640 rows, prefill, decode, copy_blocks."""
    import torch
    import paged_kv_cache_160_gb300 as pkv
    import synth
    from paged_kv_cache_160_gb300.planner import append_slots, product_plan
    case = synth.mixed_config()
    plan = product_plan(case)
    assert not plan.cows, "the mixed step's decode tokens need no copy-on-write"
    assert append_slots(case, plan) == list(plan.slots), "each decode token goes to its sequence's last position"
    work = mixed_step_work(case, plan)
    R = rotation(case, l2)
    kcs, vcs, descs = device_case(pkv, case, dev, R)
    ch = case.chunk
    q = case.q.to(dev)
    out = torch.empty_like(q)
    k_all = torch.cat([case.k_new, ch.k_new]).to(dev)
    v_all = torch.cat([case.v_new, ch.v_new]).to(dev)
    slots = torch.tensor(list(plan.slots) + list(plan.chunk_slots), dtype=torch.int64, device=dev)
    k_dec, v_dec = case.k_new.to(dev), case.v_new.to(dev)
    k_ch, v_ch = ch.k_new.to(dev), ch.v_new.to(dev)
    ch_slots = torch.tensor(list(plan.chunk_slots), dtype=torch.int64, device=dev)
    tables = torch.tensor(plan.tables, dtype=torch.int32, device=dev)
    lens = torch.tensor(plan.lens, dtype=torch.int32, device=dev)
    max_len = max(plan.lens)
    ws = torch.zeros(pkv.pkv_decode_workspace_bytes(case.num_seqs, case.num_heads, case.num_kv_heads,
                                                    case.head_dim, case.block_size, max_len, 0),
                     dtype=torch.uint8, device=dev)
    cq = ch.q.to(dev)
    cout = torch.empty_like(cq)
    cu = torch.tensor([0, ch.q_len], dtype=torch.int32, device=dev)
    st0 = torch.tensor([ch.prefix_len], dtype=torch.int32, device=dev)
    ctab = torch.tensor([plan.chunk_table], dtype=torch.int32, device=dev)
    pairs = torch.tensor(plan.share_pairs, dtype=torch.int32, device=dev)

    s2 = torch.cuda.Stream(dev)
    forked, joined = torch.cuda.Event(), torch.cuda.Event()

    def split_step(k):
        r = k % R
        forked.record(stream)
        s2.wait_event(forked)                  # after the previous step's copy_blocks
        pkv.pkv_paged_decode_append(out, q, k_dec, v_dec, kcs[r], vcs[r], descs[r], tables, lens, max_len,
                                    case.scale, 0, ws, stream)
        pkv.pkv_kv_write(k_ch, v_ch, ch_slots, kcs[r], vcs[r], descs[r], s2)
        pkv.pkv_paged_prefill_chunk(cout, cq, cu, st0, ch.q_len, kcs[r], vcs[r], descs[r], ctab, case.scale, s2)
        joined.record(s2)
        stream.wait_event(joined)
        pkv.pkv_copy_blocks(kcs[r], vcs[r], descs[r], pairs, stream)

    def serial_step(k):
        r = k % R
        pkv.pkv_kv_write(k_all, v_all, slots, kcs[r], vcs[r], descs[r], stream)
        pkv.pkv_paged_prefill_chunk(cout, cq, cu, st0, ch.q_len, kcs[r], vcs[r], descs[r], ctab, case.scale, stream)
        pkv.pkv_paged_decode(out, q, kcs[r], vcs[r], descs[r], tables, lens, max_len, case.scale, 0, ws, stream)
        pkv.pkv_copy_blocks(kcs[r], vcs[r], descs[r], pairs, stream)

    pkv.pkv_set_decode_sm_budget(MIXED_DECODE_SMS)
    try:
        ms = graph_ms(stream, split_step, K, W)   # the budget is fixed in the graph at capture
    finally:
        pkv.pkv_set_decode_sm_budget(0)
    ms_serial = graph_ms(stream, serial_step, K, W)
    assert pkv.pkv_get_device_error(stream) == 0
    res = {"workload": "mixed chunked-prefill + decode step: 512-row causal chunk at 3584..4095 over its paged "
                       "prefix, 128 decode seqs with context_lens U[256,4096] (seed 1605), 28/4 heads, head_dim 128, "
                       "bf16; kv_write 640 rows, then prefill chunk and paged_decode, then copy_blocks 64 pairs",
           "ms_per_step": round(ms, 5), "serial_ms_per_step": round(ms_serial, 5), "launches_per_step": 5,
           "decode_sm_budget": MIXED_DECODE_SMS,
           "what": "one CUDA graph of K steps: pkv_paged_decode_append (decode + merge) under the SM budget on the "
                   "bench stream, beside pkv_kv_write of the chunk rows then pkv_paged_prefill_chunk on a second "
                   "stream; pkv_copy_blocks after both. serial_ms_per_step: kv_write, prefill, decode, copy_blocks "
                   "in one stream on every SM",
           "bytes_per_step": work["bytes"], "flops_per_step": work["flops"],
           "gbs": round(work["bytes"] / (ms * 1e-3) / 1e9, 1),
           "tflops": round(work["flops"] / (ms * 1e-3) / 1e12, 1),
           "seq_tokens_per_s": round(work["tokens"] / (ms * 1e-3), 1),
           "parts": {k: work[k] for k in ("decode_bytes", "write_bytes", "prefill_bytes", "copy_bytes",
                                          "prefill_flops", "decode_flops")},
           "l2": f"rotating {R} pool copies" if R > 1 else "one pool copy larger than 3x L2"}
    del kcs, vcs, descs
    torch.cuda.empty_cache()
    return res


def host_step_measure(case, n_steps: int = 20) -> dict:
    """The native block-manager step (pkv_bm_step_decode: one slot per sequence, copy-on-write
    pairs, exported tables and lengths) on the workload's pool, timed over n_steps consecutive
    steps after an untimed set-up."""
    import ctypes
    from paged_kv_cache_160_gb300 import BlockManager
    from paged_kv_cache_160_gb300._binding import lib
    from paged_kv_cache_160_gb300.planner import import_all, max_blocks_of
    bm = BlockManager(case.num_blocks, case.block_size)
    import_all(bm, case)
    n = case.num_seqs
    mb = max_blocks_of(case) + -(-n_steps // case.block_size) + 1
    seqs = (ctypes.c_int64 * n)(*range(n))
    slots = (ctypes.c_int64 * n)()
    pairs = (ctypes.c_int32 * (2 * n))()
    tables = (ctypes.c_int32 * (n * mb))()
    lens = (ctypes.c_int32 * n)()
    nc = ctypes.c_int()
    t0 = time.perf_counter()
    for _ in range(n_steps):
        assert lib.pkv_bm_step_decode(bm._h, seqs, n, mb, slots, pairs, ctypes.byref(nc), tables, lens) == 0
    dt = (time.perf_counter() - t0) / n_steps
    return {"us_per_step": round(dt * 1e6, 2), "seqs": n, "steps": n_steps,
            "what": "pkv_bm_step_decode through ctypes: append one slot per sequence, export tables and lengths"}


def cache_ops_measure(pkv, case, plan, kc, vc, desc, k_new, v_new, slots, write_bytes, stream,
                      iters: int = 50, pairs: int = 64):
    """kv_write of the step's tokens and copy_blocks of `pairs` used blocks into free ones, each
    timed alone: one CUDA graph of `iters` calls between two events.  Both are latency-bound
    at these sizes (a few MB at most)."""
    import torch
    bs = case.block_size
    used = set()
    for row, L in zip(plan.tables, plan.lens):
        used.update(row[:-(-L // bs)])
    free = [b for b in range(case.num_blocks) if b not in used]
    n = min(pairs, len(free))
    src = sorted(used)[:n]
    pr = torch.tensor(list(zip(src, free[:n])), dtype=torch.int32, device=kc.device)
    block_bytes = kc[0].numel() * kc.element_size()
    kw_ms = graph_ms(stream, lambda k: pkv.pkv_kv_write(k_new, v_new, slots, kc, vc, desc, stream), iters, 3)
    cb_ms = graph_ms(stream, lambda k: pkv.pkv_copy_blocks(kc, vc, desc, pr, stream), iters, 3)
    assert pkv.pkv_get_device_error(stream) == 0
    cb_bytes = 2 * 2 * n * block_bytes                    # K and V blocks, read and written
    return {"kv_write": {"tokens": len(plan.slots), "bytes": write_bytes, "avg_launch_ms": round(kw_ms, 5),
                         "gbs": round(write_bytes / (kw_ms * 1e-3) / 1e9, 1)},
            "copy_blocks": {"pairs": n, "bytes": cb_bytes, "avg_launch_ms": round(cb_ms, 5),
                            "gbs": round(cb_bytes / (cb_ms * 1e-3) / 1e9, 1)},
            "timing": f"one CUDA graph of {iters} back-to-back calls between events, per-call average"}


def prefill_measure(dev, iters: int = 30, reps: int = 10):
    """paged_prefill_chunk on the mixed workload's chunk: 512 causal rows at positions
    3584..4095 over the sequence's paged cache, 28/4 heads, bf16.  One CUDA graph of `reps`
    back-to-back calls, replayed `iters` times between events: the time per call without the
    graph's launch; FLOPs = 4 * head_dim * (attended query-key pairs) * heads."""
    import torch
    import paged_kv_cache_160_gb300 as pkv
    import synth
    from paged_kv_cache_160_gb300.planner import product_plan
    case = synth.mixed_config()
    plan = product_plan(case)
    ch = case.chunk
    kc, vc = case.k_cache.to(dev), case.v_cache.to(dev)
    desc = pkv.cache_desc(kc)
    pkv.pkv_kv_write(ch.k_new.to(dev), ch.v_new.to(dev), torch.tensor(plan.chunk_slots, dtype=torch.int64, device=dev),
                     kc, vc, desc)
    q = ch.q.to(dev)
    out = torch.empty_like(q)
    cu = torch.tensor([0, ch.q_len], dtype=torch.int32, device=dev)
    st0 = torch.tensor([ch.prefix_len], dtype=torch.int32, device=dev)
    tab = torch.tensor([plan.chunk_table], dtype=torch.int32, device=dev)
    s = torch.cuda.Stream(device=dev)

    def run():
        pkv.pkv_paged_prefill_chunk(out, q, cu, st0, ch.q_len, kc, vc, desc, tab, case.scale, s)

    with torch.cuda.stream(s):
        run()
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s, capture_error_mode="thread_local"):
        for _ in range(reps):
            run()
    ea = [torch.cuda.Event(enable_timing=True) for _ in range(iters)]
    eb = [torch.cuda.Event(enable_timing=True) for _ in range(iters)]
    with torch.cuda.stream(s):
        for _ in range(3):
            g.replay()
        for k in range(iters):
            ea[k].record(s)
            g.replay()
            eb[k].record(s)
    s.synchronize()
    assert pkv.pkv_get_device_error(s) == 0
    ms = sum(a.elapsed_time(b) for a, b in zip(ea, eb)) / (iters * reps)
    flops, _ = prefill_work(case, plan)
    return ms, flops


def swap_measure(dev, n_blocks: int = 4096, iters: int = 10):
    """pkv_swap_blocks between the device pool and a pinned host pool, 7B-workload block layout
    ([blocks, 4 kv heads, 16, 128] bf16: 16 KiB per K or V block), blocks scattered by a
    permutation.  Returns (device->host GB/s, host->device GB/s, bytes per call)."""
    import torch
    import paged_kv_cache_160_gb300 as pkv
    g = torch.Generator(device=dev).manual_seed(7)
    shape = (n_blocks, 4, 16, 128)
    kc = torch.randn(shape, device=dev, generator=g).to(torch.bfloat16)
    vc = torch.randn(shape, device=dev, generator=g).to(torch.bfloat16)
    hk = torch.empty(shape, dtype=torch.bfloat16).pin_memory()
    hv = torch.empty(shape, dtype=torch.bfloat16).pin_memory()
    desc = pkv.cache_desc(kc)
    perm = torch.randperm(n_blocks, generator=torch.Generator().manual_seed(8))
    out_pairs = torch.stack([torch.arange(n_blocks), perm], 1).to(torch.int32).to(dev)
    in_pairs = torch.stack([perm, torch.arange(n_blocks)], 1).to(torch.int32).to(dev)
    s = torch.cuda.Stream(device=dev)
    res = []
    for dst_k, dst_v, src_k, src_v, pairs in ((hk, hv, kc, vc, out_pairs), (kc, vc, hk, hv, in_pairs)):
        with torch.cuda.stream(s):
            for _ in range(2):
                pkv.pkv_swap_blocks(dst_k, dst_v, src_k, src_v, desc, pairs, s)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(s)
            for _ in range(iters):
                pkv.pkv_swap_blocks(dst_k, dst_v, src_k, src_v, desc, pairs, s)
            b.record(s)
        s.synchronize()
        res.append(a.elapsed_time(b) / iters)
    assert pkv.pkv_get_device_error(s) == 0
    nbytes = 2 * kc.numel() * kc.element_size()
    # The host link's reference: the same bytes as one contiguous copy each way (copy engines).
    flat_d = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    flat_h = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    link = []
    for dst, src in ((flat_h, flat_d), (flat_d, flat_h)):
        with torch.cuda.stream(s):
            dst.copy_(src, non_blocking=True)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(s)
            for _ in range(iters):
                dst.copy_(src, non_blocking=True)
            b.record(s)
        s.synchronize()
        link.append(nbytes / (a.elapsed_time(b) / iters * 1e-3) / 1e9)
    return nbytes / (res[0] * 1e-3) / 1e9, nbytes / (res[1] * 1e-3) / 1e9, nbytes, link


# ---------------------------------------------------------------------------------------
# the oracle on the host cores (cpu_baseline and the reference arm)
# ---------------------------------------------------------------------------------------

def _sample_bytes(case, plan, seqs):
    """Algorithmic bytes of the sampled sequences' share of the step (their rows counted per
    sequence, as the oracle reads them)."""
    Hkv, D = case.num_kv_heads, case.head_dim
    kv_elt = 1 if case.kv_dtype == "e4m3" else 2
    rows = sum(plan["lens"][i] for i in seqs)
    n_w = len(seqs) if case.writes else 0
    return (2 * rows * Hkv * D * kv_elt + 2 * len(seqs) * case.num_heads * D * 2 + 4 * len(seqs)
            + 2 * 2 * n_w * Hkv * D * kv_elt + 8 * n_w), rows


_W_CASE = None
_W_PLAN = None


def _oracle_worker_init(workload: int) -> None:
    """Each worker process builds the (seeded, identical) workload and plans it with the
    oracle's own block manager, so no pool crosses a process boundary."""
    global _W_CASE, _W_PLAN
    import synth
    from oracle.workload import plan_step
    _W_CASE = synth.CONFIG_BUILDERS[workload]()
    _W_PLAN = plan_step(_W_CASE)


def _oracle_task(seqs):
    from oracle.workload import decode_sample
    decode_sample(_W_CASE, _W_PLAN["tables"], _W_PLAN["lens"], _W_PLAN["slots"], list(seqs))
    return _sample_bytes(_W_CASE, _W_PLAN, seqs)


def _groups(case, plan, per: int):
    return [list(range(i, min(i + per, case.num_seqs))) for i in range(0, case.num_seqs, per)]


def cpu_baseline(workload: int, case, plan_unused, budget_s: float) -> dict:
    """Times the fp64 oracle (kv_write + decode, as it stands) on the host cores: once in this
    process on one core, once over a spawned pool of one process per core (each with one BLAS
    thread), each for about budget_s seconds of whole-batch passes."""
    import multiprocessing as mp
    from oracle.workload import plan_step
    global _W_CASE, _W_PLAN
    _W_CASE, _W_PLAN = case, plan_step(case)
    per = 8 if max(_W_PLAN["lens"]) <= 8192 else 1
    groups = _groups(case, _W_PLAN, per)
    # one core
    done_b = done_rows = n_seq = 0
    t0 = time.perf_counter()
    i = 0
    while time.perf_counter() - t0 < budget_s:
        seqs = groups[i % len(groups)]
        b, rows = _oracle_task(seqs)
        done_b += b
        done_rows += rows
        n_seq += len(seqs)
        i += 1
    dt1 = time.perf_counter() - t0
    one = {"value": round(done_b / dt1 / 1e9, 4), "unit": "GB/s", "cores": 1,
           "seq_tokens_per_s": round(done_rows / dt1, 1),
           "sample": f"{n_seq} sequence-steps of the workload, {per} sequences per oracle call, {dt1:.1f} s wall"}
    # all cores: whole-batch passes until the budget is spent
    cores = os.cpu_count() or 1
    ctx = mp.get_context("spawn")
    with ctx.Pool(cores, initializer=_oracle_worker_init, initargs=(workload,)) as pool:
        pool.map(_oracle_task, [[0]] * cores, chunksize=1)          # every worker built its case
        fine = [[s] for s in range(case.num_seqs)] if per > 1 else groups
        done_b = done_rows = n_seq = passes = 0
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < budget_s or passes == 0:
            for b, rows in pool.imap_unordered(_oracle_task, fine, chunksize=1):
                done_b += b
                done_rows += rows
            n_seq += case.num_seqs
            passes += 1
        dtn = time.perf_counter() - t0
    alln = {"value": round(done_b / dtn / 1e9, 4), "unit": "GB/s", "cores": cores,
            "seq_tokens_per_s": round(done_rows / dtn, 1),
            "sample": f"{passes} whole-batch passes ({n_seq} sequence-steps), one sequence per task over "
                      f"{cores} spawned processes with one BLAS thread each, {dtn:.1f} s wall"}
    return {"value": alln["value"], "unit": "GB/s", "cores": cores, "kind": "oracle",
            "seq_tokens_per_s": alln["seq_tokens_per_s"],
            "sample": "fp64 numpy oracle (kv_write + decode) on the same workload; " + alln["sample"],
            "single_core": one, "all_cores": alln}


def run_reference(args):
    """The oracle as the reference arm: every step is the whole batch's kv_write + decode, as
    the oracle stands, over a spawned pool of one process per host core."""
    import multiprocessing as mp
    import synth
    from oracle.workload import plan_step
    case = synth.CONFIG_BUILDERS[args.workload]()
    plan = plan_step(case)
    cores = os.cpu_count() or 1
    per = 1
    tasks = _groups(case, plan, per)
    ctx = mp.get_context("spawn")
    with ctx.Pool(cores, initializer=_oracle_worker_init, initargs=(args.workload,)) as pool:
        pool.map(_oracle_task, [[0]] * cores, chunksize=1)
        for _ in range(args.warmup):
            list(pool.imap_unordered(_oracle_task, tasks, chunksize=1))
        tot_b = tot_rows = 0
        t0 = time.perf_counter()
        for _ in range(args.steps):
            for b, rows in pool.imap_unordered(_oracle_task, tasks, chunksize=1):
                tot_b += b
                tot_rows += rows
        dt = time.perf_counter() - t0
    value = tot_b / dt / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * dt / args.steps, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": WORKLOADS[args.workload], "sample_per_step": "the whole batch"},
            "seq_tokens_per_s": round(tot_rows / dt, 1),
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": f"every step is the whole batch's kv_write + decode, one sequence per task "
                                       f"over {cores} spawned processes with one BLAS thread each (fp64 numpy)"},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="pkv", choices=["pkv", "reference"])
    ap.add_argument("--workload", type=int, default=2, choices=sorted(WORKLOADS),
                    help="2: the 7B GQA decode step (default, the headline); 3-5: the other decode workloads")
    ap.add_argument("--headline-only", action="store_true",
                    help="skip the other workloads and the mixed step (quicker runs)")
    ap.add_argument("--cpu-budget", type=float, default=10.0, help="seconds of oracle work per CPU-baseline leg")
    ap.add_argument("--part", choices=["prefill"],
                    help="time one call alone and print its line (a small command to profile): "
                         "prefill = paged_prefill_chunk on the mixed-step chunk")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if refuse_multi_gpu(args):
        return
    if args.part == "prefill":
        run_part_prefill(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


def run_part_prefill(args):
    """Only the prefill chunk of the mixed step, `args.steps` graph replays of 10 calls."""
    import torch
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    ms, flops = prefill_measure(dev, iters=max(1, args.steps))
    peak, _ = _bf16_peak()
    tf = flops / (ms * 1e-3) / 1e12
    print(json.dumps({"part": "prefill_chunk", "workload": "mixed-step chunk: 512 causal rows at 3584..4095, 28/4 heads, bf16",
                      "avg_launch_ms": round(ms, 5), "tflops": round(tf, 1), "frac_of_bf16_peak": round(tf / peak, 4),
                      "flops_per_launch": flops}))


if __name__ == "__main__":
    main()
