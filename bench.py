"""Benchmark of the paged-KV decode step on GB300: effective HBM GB/s and seq-tokens/s.

Workload: the Qwen2.5-7B-shaped GQA decode batch — 64 running sequences with context
lengths uniform in [128, 2048], 28 query heads / 4 kv heads, head_dim 128, bf16 Q/K/V,
16-token blocks in a shuffled pool ([num_blocks, 4, 16, 128], pool = blocks needed + 10%).
One step = plan the step on the host block manager (done once; its cost is reported
separately), the write of the 64 new tokens' K/V, then paged_decode over every sequence's
L + 1 tokens.  Every new token belongs at its sequence's last position, so the write is
fused into the decode call (pkv_paged_decode_append: two launches, the split-KV decode and
the log-sum-exp merge of split segments as its programmatic dependent); kv_write + decode
is timed beside it.

Timing: CUDA events on the launching stream.  The K timed steps are captured into one
CUDA graph and replayed once between two events.  The decode call's own average duration
(decode + merge, for its roofline) comes from a second graph of K calls timed the same way.
Every step uses the next of R pool copies whose combined size is above 3x the L2 size, so
no step finds its K/V in L2.  `value` is device-resident throughput.  `e2e` passes HOST
buffers to the call: every step's inputs (q, new K/V, tables, lengths) are read in place
from pinned host memory and its output is written to pinned host memory by the kernels,
across NVLink-C2C.  The same steps with explicit staged H2D/D2H copies on copy streams are
reported beside it.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference] [--workload 2|3|4|5]

--workload picks another decode workload (3: 13B MHA, 4: long-context e4m3, 5: the mixed
step's decode part); the default, 2, is the headline.
"""
from __future__ import annotations

import os

# The CPU baseline times the oracle with one BLAS thread; pin numpy's BLAS before it loads.
for _var in ("OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
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

# DRAM bytes per decode call on this workload (paged_decode_kernel + split_kv_merge_kernel,
# dram__bytes_read.sum + dram__bytes_write.sum from one ncu capture each), valid only for the
# kernel source with this hash; when the source changes, traffic is reported as null until
# re-measured.
TRAFFIC = {"source_sha1": "aabb1d5dca5ecc7a6f5daf1ee59b2bd12bc1de7c", "bytes_per_launch": 161774592}


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


def _bf16_peak() -> float:
    """Measured dense bf16 TFLOP/s (burst: the prefill kernel is timed alone)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        return float(json.load(open(path))["bf16_tflops"])
    return 1900.0


def max_over_ranks(x: float, device) -> float:
    """The largest value of x over all ranks (the slowest rank defines the timed region)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_gbs(bytes_per_rank: int, ms_per_step: float, world: int) -> float:
    """Whole-job GB/s: every rank runs its own replica of the step (weak scaling)."""
    return world * bytes_per_rank / (ms_per_step * 1e-3) / 1e9


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


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


def workload_bytes(case, plan):
    """Algorithmic bytes of one step (each unique attended K/V row once)."""
    Hkv, D, Hq = case.num_kv_heads, case.head_dim, case.num_heads
    kv_elt = 1 if case.kv_dtype == "e4m3" else 2
    q_elt = 2
    unique_rows = set()
    for t, L in zip(plan.tables, plan.lens):
        for j in range(L):
            unique_rows.add(t[j // 16] * 16 + j % 16)
    n_rows = len(unique_rows)
    nblocks = sum(-(-L // 16) for L in plan.lens)
    S = case.num_seqs
    decode = 2 * n_rows * Hkv * D * kv_elt + 2 * S * Hq * D * q_elt + 4 * nblocks + 4 * S
    T = len(plan.slots)
    write = 2 * 2 * T * Hkv * D * kv_elt + 8 * T
    return decode, write, sum(plan.lens)


def run_gpu(args):
    import numpy as np
    import torch

    import paged_kv_cache_160_gb300 as pkv
    import synth
    from tests.harness import append_slots, product_plan

    ws_n, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws_n > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

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
    kcs = [case.k_cache.to(dev) for _ in range(R)]
    vcs = [case.v_cache.to(dev) for _ in range(R)]
    k_scale = case.k_scale.to(dev) if case.k_scale is not None else None   # e4m3 caches: per-head scales
    v_scale = case.v_scale.to(dev) if case.v_scale is not None else None
    descs = [pkv.cache_desc(k, k_scale, v_scale) for k in kcs]
    q = case.q.to(dev)
    k_new = case.k_new.to(dev) if case.writes else None
    v_new = case.v_new.to(dev) if case.writes else None
    slots = torch.tensor(plan.slots, dtype=torch.int64, device=dev)
    tables = torch.tensor(plan.tables, dtype=torch.int32, device=dev)
    lens = torch.tensor(plan.lens, dtype=torch.int32, device=dev)
    out = torch.empty_like(q)
    max_len = max(plan.lens)
    part = case.partition_size
    wsb = pkv.pkv_decode_workspace_bytes(case.num_seqs, case.num_heads, case.num_kv_heads, case.head_dim, 16,
                                         max_len, part)
    ws = torch.zeros(wsb, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)

    # Every decode token goes to its sequence's last position, so the step's write is fused
    # into the decode call (pkv_paged_decode_append); the unfused pair is timed beside it.
    fused = case.writes and append_slots(case, plan) == list(plan.slots)

    def write(r):
        if case.writes:
            pkv.pkv_kv_write(k_new, v_new, slots, kcs[r], vcs[r], descs[r])

    def decode(r):
        pkv.pkv_paged_decode(out, q, kcs[r], vcs[r], descs[r], tables, lens, max_len, case.scale, part, ws)

    def step(r, fuse=fused):
        if fuse:
            pkv.pkv_paged_decode_append(out, q, k_new, v_new, kcs[r], vcs[r], descs[r], tables, lens, max_len,
                                        case.scale, part, ws)
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

    def barrier():
        if ws_n > 1:
            import torch.distributed as dist
            dist.barrier()

    # The timed loop is one CUDA graph of K steps (each: the fused append + decode -> split-KV
    # merge, or kv_write -> decode -> merge, launched as programmatic dependents), rotating over
    # the pool copies.  The decode kernel's own average duration (decode + merge, without the
    # write, for its roofline) is timed the same way on a graph of K decodes alone; event nodes
    # between kernels would break the programmatic launches and inflate it.
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
    g_dec_warm = capture(W, 0, kind="step" if fused else "decode")   # the step's decode call alone
    g_dec = capture(K, W, kind="step" if fused else "decode")
    g_unf = capture(K, W, kind="unfused") if fused else None
    torch.cuda.synchronize(dev)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    d_start, d_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    with torch.cuda.stream(stream):
        g_warm.replay()
    stream.synchronize()
    barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        with torch.cuda.stream(stream):
            start.record(stream)
            g_timed.replay()
            end.record(stream)
        stream.synchronize()
        barrier()
        torch.cuda.synchronize(dev)
        with torch.cuda.stream(stream):
            g_dec_warm.replay()
            d_start.record(stream)
            g_dec.replay()
            d_end.record(stream)
        stream.synchronize()
        unfused_ms = None
        if g_unf is not None:
            u_start, u_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                g_warm.replay()
                u_start.record(stream)
                g_unf.replay()
                u_end.record(stream)
            stream.synchronize()
            unfused_ms = u_start.elapsed_time(u_end) / K
    elapsed_ms = max_over_ranks(start.elapsed_time(end), dev)
    dec_avg_ms = d_start.elapsed_time(d_end) / K
    assert pkv.pkv_get_device_error(stream) == 0

    # ---- end to end, staged: explicit copies on copy streams --------------------------------
    # A serving loop's shape: each step's inputs (q, new K/V, slots, tables, lengths) sit in one
    # pinned staging buffer and go up in one copy; device inputs and outputs are double-
    # buffered; uploads run on one copy stream and output downloads on another, ordered by
    # events, so step k+1's upload and step k's download overlap step k's kernels.  Every step
    # still moves its full input and output bytes across the host link.
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
                                                case.scale, part, ws)
                else:
                    if case.writes:
                        kni, vni, sli = dv[i][3:]
                        pkv.pkv_kv_write(kni, vni, sli, kcs[r], vcs[r], descs[r])
                    pkv.pkv_paged_decode(outs[i], qi, kcs[r], vcs[r], descs[r], tbi, lni, max_len, case.scale,
                                         part, ws)
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
    barrier()
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        g_e2e_warm.replay()
        e_start.record(stream)
        g_e2e.replay()
        e_end.record(stream)
    stream.synchronize()
    barrier()
    staged_ms = max_over_ranks(e_start.elapsed_time(e_end), dev)
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

        def zc_graph(n_steps, first):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
                for k in range(n_steps):
                    hs, r = hsets[k % 2], (first + k) % R
                    if fused:
                        pkv.pkv_paged_decode_append(hs["out"], hs["q"], hs["kn"], hs["vn"], kcs[r], vcs[r], descs[r],
                                                    hs["tb"], hs["ln"], max_len, case.scale, part, ws)
                    else:
                        pkv.pkv_paged_decode(hs["out"], hs["q"], kcs[r], vcs[r], descs[r], hs["tb"], hs["ln"],
                                             max_len, case.scale, part, ws)
            return g

        gz_warm, gz = zc_graph(W, 0), zc_graph(K, W)
        z_start, z_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        torch.cuda.synchronize(dev)
        with torch.cuda.stream(stream):
            gz_warm.replay()
            z_start.record(stream)
            gz.replay()
            z_end.record(stream)
        stream.synchronize()
        barrier()
        e2e_ms = max_over_ranks(z_start.elapsed_time(z_end), dev)
        for hs in hsets:
            assert torch.equal(hs["out"], out.cpu())
    else:
        e2e_ms = staged_ms
    pf_ms, pf_flops = prefill_measure(dev)
    cache_ops = cache_ops_measure(pkv, case, plan, kcs[0], vcs[0], descs[0], k_new, v_new, slots, write_bytes,
                                  stream) if case.writes else None
    sw_out, sw_in, sw_bytes, sw_link = swap_measure(dev)

    peak, peak_kind = _peaks()
    ms_per_step = elapsed_ms / K
    value = aggregate_gbs(step_bytes, ms_per_step, ws_n)
    roof_bytes = step_bytes if fused else decode_bytes        # the fused call also moves the new rows
    achieved = roof_bytes / (dec_avg_ms * 1e-3) / 1e9
    traffic = (TRAFFIC["bytes_per_launch"] if args.workload == 2 and TRAFFIC["source_sha1"] == _src_hash()
               else None)
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": ws_n,
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
                   "parallelism": f"replicas x{ws_n}" if ws_n > 1 else "single GPU"},
        "seq_tokens_per_s": round(ws_n * tokens / (ms_per_step * 1e-3), 1),
        "pct_of_nominal_8tbs": round(100 * value / ws_n / NOMINAL_HBM_GBS, 2),
        "pct_of_measured_copy": round(100 * value / ws_n / peak, 2),
        "roofline": {"kernel": "paged_decode_append (decode + merge)" if fused else "paged_decode (decode + merge)",
                     "bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "peak_kind": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_kind == "measured" else "fallback 6.8 TB/s",
                     "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                     "algorithmic_bytes_per_launch": roof_bytes, "avg_launch_ms": round(dec_avg_ms, 5),
                     "frac_of_nominal_8tbs": round(achieved / NOMINAL_HBM_GBS, 4)},
        "e2e": {"value": round(aggregate_gbs(step_bytes, e2e_ms / K, ws_n), 1), "unit": "GB/s",
                "ms_per_step": round(e2e_ms / K, 5), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "copies": ("the call gets HOST buffers: each step's inputs (q, new K/V, tables, lengths) are "
                           "read in place from pinned host memory and its output is written to pinned host "
                           "memory by the kernels (NVLink-C2C); two buffer sets alternate; the K steps are "
                           "one CUDA graph") if zero_copy else
                          ("per step one H2D of the pinned staged inputs and one D2H of the output, on two copy "
                           "streams ordered by events; double-buffered; the K steps are one CUDA graph"),
                "staged_copies": {"value": round(aggregate_gbs(step_bytes, staged_ms / K, ws_n), 1),
                                  "ms_per_step": round(staged_ms / K, 5),
                                  "what": "the same steps with explicit H2D/D2H copies on two copy streams, "
                                          "ordered by events (double-buffered), in one CUDA graph"}},
        "prefill_chunk": {"workload": "mixed-step chunk: 512 causal rows at 3584..4095, 28/4 heads, bf16",
                          "bound": "tensor", "achieved": round(pf_flops / (pf_ms * 1e-3) / 1e12, 1),
                          "peak": _bf16_peak(), "unit": "TFLOP/s",
                          "frac": round(pf_flops / (pf_ms * 1e-3) / 1e12 / _bf16_peak(), 4),
                          "avg_launch_ms": round(pf_ms, 5), "flops_per_launch": pf_flops},
        "swap_blocks": {"workload": "4096 scattered blocks of the 7B layout (K and V), device <-> pinned host",
                        "bytes_per_call": sw_bytes, "device_to_host_gbs": round(sw_out, 1),
                        "host_to_device_gbs": round(sw_in, 1),
                        "contiguous_copy_gbs": {"device_to_host": round(sw_link[0], 1),
                                                "host_to_device": round(sw_link[1], 1)}},
        "cache_ops": cache_ops,
        "host_plan_us": round(host_plan_us, 1),
        "host_step": host_step_measure(case) if case.writes else None,
        "gpu_launches": (3 if case.writes and not fused else 2) * K,   # (kv_write,) decode, merge per step
        "unfused_step": None if unfused_ms is None else {
            "ms_per_step": round(unfused_ms, 5), "value": round(aggregate_gbs(step_bytes, unfused_ms, 1), 1),
            "what": "the same step as pkv_kv_write + pkv_paged_decode (3 launches), one graph of K steps"},
        "clocks": clk.summary(),
    }
    if rank == 0:
        line["cpu_baseline"] = cpu_baseline(case, plan, decode_bytes, write_bytes)
        print(json.dumps(line))
    if ws_n > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def host_step_measure(case, n_steps: int = 20) -> dict:
    """The native block-manager step (pkv_bm_step_decode: one slot per sequence, copy-on-write
    pairs, exported tables and lengths) on the workload's pool, timed over n_steps consecutive
    steps after an untimed set-up."""
    import ctypes
    from paged_kv_cache_160_gb300 import BlockManager
    from paged_kv_cache_160_gb300._binding import lib
    from tests.harness import _import_all, max_blocks_of
    bm = BlockManager(case.num_blocks, case.block_size)
    _import_all(bm, case)
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

    def timed(fn):
        with torch.cuda.stream(stream):
            for _ in range(3):
                fn()
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
            for _ in range(iters):
                fn()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            g.replay()
            a.record(stream)
            g.replay()
            b.record(stream)
        stream.synchronize()
        return a.elapsed_time(b) / iters

    kw_ms = timed(lambda: pkv.pkv_kv_write(k_new, v_new, slots, kc, vc, desc))
    cb_ms = timed(lambda: pkv.pkv_copy_blocks(kc, vc, desc, pr))
    assert pkv.pkv_get_device_error(stream) == 0
    cb_bytes = 2 * 2 * n * block_bytes                    # K and V blocks, read and written
    return {"kv_write": {"tokens": len(plan.slots), "bytes": write_bytes, "avg_launch_ms": round(kw_ms, 5),
                         "gbs": round(write_bytes / (kw_ms * 1e-3) / 1e9, 1)},
            "copy_blocks": {"pairs": n, "bytes": cb_bytes, "avg_launch_ms": round(cb_ms, 5),
                            "gbs": round(cb_bytes / (cb_ms * 1e-3) / 1e9, 1)},
            "timing": f"one CUDA graph of {iters} back-to-back calls between events, per-call average"}


def prefill_measure(dev, iters: int = 30):
    """paged_prefill_chunk on the mixed workload's chunk: 512 causal rows at positions
    3584..4095 over the sequence's paged cache, 28/4 heads, bf16.  CUDA-graph replays timed
    with events; FLOPs = 4 * head_dim * (attended query-key pairs) * heads."""
    import torch
    import paged_kv_cache_160_gb300 as pkv
    import synth
    from tests.harness import append_slots, product_plan
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
        pkv.pkv_paged_prefill_chunk(out, q, cu, st0, ch.q_len, kc, vc, desc, tab, case.scale)

    with torch.cuda.stream(s):
        run()
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s, capture_error_mode="thread_local"):
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
    ms = sum(a.elapsed_time(b) for a, b in zip(ea, eb)) / iters
    pairs = sum(ch.prefix_len + r + 1 for r in range(ch.q_len))
    flops = 4 * case.head_dim * pairs * case.num_heads
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


def _oracle_step(case, plan, seqs):
    """The oracle (as it stands) on a subset of the step: its KV write and decode.  The sampled
    sequences' blocks are gathered into a pool of their own first (tables and slots renumbered),
    so the oracle's copy-on-return KV write copies only that pool."""
    import numpy as np
    from oracle import cache_ops, paged_attention as pa
    from tests.harness import codes, q_f64
    bs = case.block_size
    used = sorted({b for i in seqs for b in plan.tables[i] if b >= 0})
    new_id = {b: n for n, b in enumerate(used)}
    k, v = codes(case.k_cache)[used], codes(case.v_cache)[used]
    tables = [[new_id[b] for b in plan.tables[i] if b >= 0] for i in seqs]
    if case.writes:
        slots = [new_id[plan.slots[i] // bs] * bs + plan.slots[i] % bs for i in seqs]
        k, v = cache_ops.kv_write(k, v, codes(case.k_new)[seqs], codes(case.v_new)[seqs], slots)
    ks = case.k_scale.numpy().astype(np.float64) if case.k_scale is not None else None
    vs = case.v_scale.numpy().astype(np.float64) if case.v_scale is not None else None
    pa.decode_attention(q_f64(case.q)[seqs], k, v, case.kv_dtype, tables, [plan.lens[i] for i in seqs], case.scale,
                        ks, vs)


def _sample_bytes(case, plan, seqs):
    """Algorithmic bytes of the sampled sequences' share of the step (their rows counted per
    sequence, as the oracle reads them)."""
    Hkv, D = case.num_kv_heads, case.head_dim
    kv_elt = 1 if case.kv_dtype == "e4m3" else 2
    rows = sum(plan.lens[i] for i in seqs)
    n_w = len(seqs) if case.writes else 0
    return (2 * rows * Hkv * D * kv_elt + 2 * len(seqs) * case.num_heads * D * 2 + 4 * len(seqs)
            + 2 * 2 * n_w * Hkv * D * kv_elt + 8 * n_w), rows


def cpu_baseline(case, plan, decode_bytes, write_bytes, budget_s: float = 12.0):
    """Times the fp64 oracle on the host cores, single-threaded BLAS, cycling over the batch."""
    seqs_all = list(range(case.num_seqs))
    done_bytes = done_tokens = 0
    n_seq = 0
    per = 8 if max(plan.lens) <= 8192 else 1          # long sequences: one per oracle call
    t0 = time.perf_counter()
    i = 0
    while time.perf_counter() - t0 < budget_s:         # about budget_s of CPU work
        seqs = [seqs_all[(i + j) % case.num_seqs] for j in range(per)]
        _oracle_step(case, plan, seqs)
        b, rows = _sample_bytes(case, plan, seqs)
        done_bytes += b
        done_tokens += rows
        n_seq += len(seqs)
        i += per
    dt = time.perf_counter() - t0
    return {"value": round(done_bytes / dt / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "seq_tokens_per_s": round(done_tokens / dt, 1),
            "sample": f"fp64 numpy oracle (kv_write + decode) on {n_seq} sequence-steps of the same workload, "
                      f"{per} sequences per call, {dt:.1f} s wall, 1 BLAS thread"}


def run_reference(args):
    """The oracle as the reference arm: each step is a bounded sample (4 sequences)."""
    import synth
    from tests.harness import oracle_plan
    ws_n, rank, _ = _dist()
    if rank != 0:
        return
    case = synth.CONFIG_BUILDERS[args.workload]()
    plan = oracle_plan(case)
    per = 4 if max(plan.lens) <= 8192 else 1
    if True:
        for k in range(args.warmup):
            _oracle_step(case, plan, [(k * per + j) % case.num_seqs for j in range(per)])
        tot_b = tot_rows = 0
        t0 = time.perf_counter()
        for k in range(args.steps):
            seqs = [((args.warmup + k) * per + j) % case.num_seqs for j in range(per)]
            _oracle_step(case, plan, seqs)
            b, rows = _sample_bytes(case, plan, seqs)
            tot_b += b
            tot_rows += rows
        dt = time.perf_counter() - t0
    value = tot_b / dt / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": ws_n,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * dt / args.steps, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": WORKLOADS[args.workload], "sample_per_step": f"{per} sequences"},
            "seq_tokens_per_s": round(tot_rows / dt, 1),
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": f"{per} sequences of the workload per step (kv_write + decode), fp64 numpy, "
                                       "1 BLAS thread"},
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
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
