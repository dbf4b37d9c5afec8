"""The bench's algorithmic-byte accounting (the roofline's numerator), pinned to closed forms.

Decode bytes = every unique attended K/V row once (K and V) + q and out + one table entry per
16-token tile + one length per sequence; write bytes = the new rows read and written + their
slots.  A prefix shared through identical block ids is counted once.
"""
import bench
import synth
from tests.harness import product_plan


def _closed_form(lens_after, S, Hq, Hkv, D, elt, shared_rows, T):
    rows = sum(lens_after) - shared_rows
    tiles = sum(-(-L // 16) for L in lens_after)
    decode = 2 * rows * Hkv * D * elt + 2 * S * Hq * D * 2 + 4 * tiles + 4 * S
    write = 2 * 2 * T * Hkv * D * elt + 8 * T
    return decode, write


def test_private_blocks_count_every_row():
    lens = [1, 15, 16, 17, 200]
    case = synth.make_decode_case("acct_private", 11, lens, 8, 2, 64, "f16", "f16")
    plan = product_plan(case)
    after = [L + 1 for L in lens]
    assert plan.lens == after
    assert bench.workload_bytes(case, plan) == (*_closed_form(after, 5, 8, 2, 64, 2, 0, 5), sum(after))


def test_a_shared_prefix_is_counted_once():
    # sequences 1..4 reuse sequence 0's first two (full) blocks: 4 x 32 rows are not re-counted
    lens = [40, 50, 60, 70, 80]
    case = synth.make_decode_case("acct_shared", 5, lens, 8, 2, 64, "f16", "f16",
                                  share={i: (0, 2) for i in range(1, 5)})
    plan = product_plan(case)
    after = [L + 1 for L in lens]
    assert bench.workload_bytes(case, plan) == (*_closed_form(after, 5, 8, 2, 64, 2, 4 * 32, 5), sum(after))


def test_e4m3_rows_are_one_byte_and_no_write():
    lens = [33, 100]
    case = synth.make_decode_case("acct_e4m3", 12, lens, 32, 8, 128, "bf16", "e4m3", write=False)
    plan = product_plan(case)
    decode, write = _closed_form(lens, 2, 32, 8, 128, 1, 0, 0)
    assert bench.workload_bytes(case, plan) == (decode, write, sum(lens))


def test_prefill_and_mixed_step_work_closed_forms():
    # chunk of n rows at positions p0..p0+n-1: sum over rows of (p0 + r + 1) attended keys
    p0, n = 40, 20
    case = synth.make_decode_case("acct_mixed", 13, [30, 17], 8, 2, 64, "bf16", "bf16", chunk=(p0, n),
                                  copy_pairs=2)
    plan = product_plan(case)
    flops, nbytes = bench.prefill_work(case, plan)
    pairs = n * p0 + n * (n + 1) // 2
    assert flops == 4 * 64 * pairs * 8
    assert nbytes == 2 * (p0 + n) * 2 * 64 * 2 + 2 * n * 8 * 64 * 2 + 4 * len(plan.chunk_table)
    w = bench.mixed_step_work(case, plan)
    decode, _, tokens = bench.workload_bytes(case, plan)
    T = 2 + n                                       # one decode token per sequence + the chunk rows
    block = 2 * 16 * 64 * 2
    assert w["write_bytes"] == 2 * 2 * T * 2 * 64 * 2 + 8 * T
    assert w["copy_bytes"] == 2 * 2 * 2 * block + 8 * 2
    assert w["bytes"] == decode + w["write_bytes"] + nbytes + w["copy_bytes"]
    assert w["flops"] == flops + 4 * 64 * tokens * 8


def test_bench_refuses_more_than_one_gpu():
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--gpus", "2", "--steps", "3"],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    lines = [x for x in r.stdout.splitlines() if x.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["n_gpus"] == 2 and "unavailable" in d


def test_decode_tile_rows_follow_the_block_tables():
    """Every tile row is the pool row of logical token 16 * i of its sequence (address
    translation of Lecture 33 §2.2), for 16- and 32-token blocks."""
    from paged_kv_cache_160_gb300.planner import decode_tile_rows
    for bs in (16, 32):
        case = synth.make_decode_case("acct_rows", 21, [5, 40, 33], 4, 2, 64, "f16", "f16", block_size=bs)
        plan = product_plan(case)
        rows = decode_tile_rows(case, plan)
        want = []
        for t, L in zip(plan.tables, plan.lens):
            for h in range(2):
                for j in range(0, L, 16):
                    want.append((t[j // bs] * 2 + h) * bs + j % bs)
        assert rows == want


def test_mixed_step_decode_tokens_are_last_positions():
    """The bench's mixed step writes its decode tokens inside pkv_paged_decode_append, which
    stores each sequence's new row at position context_len - 1; that is the kv_write of the
    serial step only if every decode token's slot is its sequence's last position.  The chunk
    rows go through kv_write on the prefill's stream, and no slot is written twice."""
    from paged_kv_cache_160_gb300.planner import append_slots
    case = synth.mixed_config()
    plan = product_plan(case)
    assert not plan.cows
    assert append_slots(case, plan) == list(plan.slots)
    assert len(plan.slots) == case.num_seqs and len(plan.chunk_slots) == case.chunk.q_len
    assert not set(plan.slots) & set(plan.chunk_slots)
    assert bench.MIXED_DECODE_SMS > 0
