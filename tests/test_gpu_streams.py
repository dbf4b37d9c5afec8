"""The mixed chunked-prefill step with its prefill chunk and its decodes running side by side,
and the decode's SM budget that makes room for the prefill.

"Lecture 33 — KV Cache management", §4.2 batches a prefill chunk with the running decodes in
one step.  The chunk's attention is tensor-bound and the decodes' attention is HBM-bound, so a
serving loop runs them side by side on two streams.  Neither call reads what the other
writes, so the results must equal the serial order bit for bit, eagerly and as one captured
graph.  The serial order itself is checked against the fp64 oracle by the parity tests.  Under
an SM budget the decode splits its tiles over fewer workers: its outputs are checked against
the oracle again, at several budgets, and the fused append still equals kv_write + decode bit
for bit.
"""
import numpy as np
import pytest
import torch

import synth
from tests.harness import device_run, product_plan
from tests.test_gpu_parity import _check_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import paged_kv_cache_160_gb300  # noqa: F401  (fails loudly if the library is missing)


def _setup():
    import paged_kv_cache_160_gb300 as pkv
    from paged_kv_cache_160_gb300.planner import product_plan
    dev = torch.device("cuda")
    case = synth.mixed_config()
    plan = product_plan(case)
    ch = case.chunk
    s = {
        "case": case, "plan": plan, "ch": ch,
        "q": case.q.to(dev), "cq": ch.q.to(dev),
        "k_all": torch.cat([case.k_new, ch.k_new]).to(dev),
        "v_all": torch.cat([case.v_new, ch.v_new]).to(dev),
        "slots": torch.tensor(list(plan.slots) + list(plan.chunk_slots), dtype=torch.int64, device=dev),
        "tables": torch.tensor(plan.tables, dtype=torch.int32, device=dev),
        "lens": torch.tensor(plan.lens, dtype=torch.int32, device=dev),
        "max_len": max(plan.lens),
        "cu": torch.tensor([0, ch.q_len], dtype=torch.int32, device=dev),
        "st0": torch.tensor([ch.prefix_len], dtype=torch.int32, device=dev),
        "ctab": torch.tensor([plan.chunk_table], dtype=torch.int32, device=dev),
        "pairs": torch.tensor(plan.share_pairs, dtype=torch.int32, device=dev),
    }
    s["ws"] = torch.zeros(pkv.pkv_decode_workspace_bytes(case.num_seqs, case.num_heads, case.num_kv_heads,
                                                         case.head_dim, case.block_size, s["max_len"], 0),
                          dtype=torch.uint8, device=dev)
    return s


def _fresh(s):
    """A pool copy, its descriptor and NaN-filled outputs."""
    import paged_kv_cache_160_gb300 as pkv
    dev = torch.device("cuda")
    kc, vc = s["case"].k_cache.to(dev), s["case"].v_cache.to(dev)
    return {"kc": kc, "vc": vc, "desc": pkv.cache_desc(kc),
            "out": torch.full_like(s["q"], float("nan")), "cout": torch.full_like(s["cq"], float("nan"))}


def _step(s, p, stream, s2=None, events=None):
    """kv_write -> prefill chunk and paged_decode -> copy_blocks; on two streams when s2 is given."""
    import paged_kv_cache_160_gb300 as pkv
    case, ch = s["case"], s["ch"]
    pkv.pkv_kv_write(s["k_all"], s["v_all"], s["slots"], p["kc"], p["vc"], p["desc"], stream)
    dstream = stream
    if s2 is not None:
        events[0].record(stream)
        s2.wait_event(events[0])
        dstream = s2
    pkv.pkv_paged_prefill_chunk(p["cout"], s["cq"], s["cu"], s["st0"], ch.q_len, p["kc"], p["vc"], p["desc"],
                                s["ctab"], case.scale, stream)
    pkv.pkv_paged_decode(p["out"], s["q"], p["kc"], p["vc"], p["desc"], s["tables"], s["lens"], s["max_len"],
                         case.scale, 0, s["ws"], dstream)
    if s2 is not None:
        events[1].record(s2)
        stream.wait_event(events[1])
    pkv.pkv_copy_blocks(p["kc"], p["vc"], p["desc"], s["pairs"], stream)


def _same(a, b):
    for key in ("out", "cout", "kc", "vc"):
        assert torch.equal(a[key].view(torch.uint8), b[key].view(torch.uint8)), key


def test_two_streams_equal_the_serial_order_bit_for_bit():
    import paged_kv_cache_160_gb300 as pkv
    s = _setup()
    stream, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    events = (torch.cuda.Event(), torch.cuda.Event())
    serial, forked = _fresh(s), _fresh(s)
    with torch.cuda.stream(stream):
        _step(s, serial, stream)
        _step(s, forked, stream, s2, events)
    stream.synchronize()
    assert pkv.pkv_get_device_error(stream) == 0
    assert not torch.isnan(serial["out"]).any() and not torch.isnan(serial["cout"]).any()
    _same(serial, forked)


def test_two_streams_captured_as_one_graph():
    """Two steps of the fork/join schedule captured in one CUDA graph and replayed twice."""
    import paged_kv_cache_160_gb300 as pkv
    s = _setup()
    stream, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    events = (torch.cuda.Event(), torch.cuda.Event())
    serial, graphed = _fresh(s), _fresh(s)
    with torch.cuda.stream(stream):
        _step(s, serial, stream)
        _step(s, graphed, stream, s2, events)          # eager first: the library's device state exists
    stream.synchronize()
    graphed["out"].fill_(float("nan"))
    graphed["cout"].fill_(float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
        for _ in range(2):
            _step(s, graphed, stream, s2, events)
    with torch.cuda.stream(stream):
        g.replay()
        g.replay()
    stream.synchronize()
    assert pkv.pkv_get_device_error(stream) == 0
    _same(serial, graphed)


# ---------------------------------------------------------------------------------------
# the decode under an SM budget
# ---------------------------------------------------------------------------------------

class _budget:
    def __init__(self, n):
        self.n = n

    def __enter__(self):
        import paged_kv_cache_160_gb300 as pkv
        pkv.pkv_set_decode_sm_budget(self.n)

    def __exit__(self, *exc):
        import paged_kv_cache_160_gb300 as pkv
        pkv.pkv_set_decode_sm_budget(0)


BUDGET_CASES = [
    # name, lens, Hq, Hkv, D, q dtype, kv dtype, partition
    ("gqa7_bf16", [5, 16, 100, 257, 1000], 28, 4, 128, "bf16", "bf16", 0),
    ("e4m3_partitions", [1, 17, 511, 512, 513, 2000], 32, 8, 128, "bf16", "e4m3", 512),
    ("mha_f16_d64_many", [int(x) for x in np.random.default_rng(9).integers(1, 300, size=60)], 4, 4, 64,
     "f16", "f16", 32),
]


@pytest.mark.parametrize("budget", [1, 5, 64, 100000])
@pytest.mark.parametrize("name,lens,hq,hkv,d,qd,kd,part", BUDGET_CASES, ids=[c[0] for c in BUDGET_CASES])
def test_decode_under_an_sm_budget_matches_the_oracle(budget, name, lens, hq, hkv, d, qd, kd, part):
    """1 CTA (12 workers holding many segments each), 5, 64 and a budget above the SM count."""
    case = synth.make_decode_case(name, 91, lens, hq, hkv, d, qd, kd, partition_size=part)
    with _budget(budget):
        _check_case(case)


def test_fused_append_under_an_sm_budget_equals_write_then_decode():
    case = synth.make_decode_case("budget_append", 92, [3, 16, 17, 300, 1200], 28, 4, 128, "bf16", "bf16")
    plan = product_plan(case)
    with _budget(5):
        plain = device_run(case, plan, keep_intermediate=False)
        fused = device_run(case, plan, keep_intermediate=False, fused_append=True)
    assert plain.device_error == 0 and fused.device_error == 0
    assert torch.equal(plain.decode.view(torch.uint8), fused.decode.view(torch.uint8))
    assert torch.equal(plain.k_final.view(torch.uint8), fused.k_final.view(torch.uint8))
    assert torch.equal(plain.v_final.view(torch.uint8), fused.v_final.view(torch.uint8))


def _split_step(s, p, stream, s2, events):
    """The decodes as the fused append under the budget on `stream`; beside them on s2 the
    chunk rows' kv_write, then the prefill chunk; joined before copy_blocks."""
    import paged_kv_cache_160_gb300 as pkv
    case, ch, plan = s["case"], s["ch"], s["plan"]
    events[0].record(stream)
    s2.wait_event(events[0])                       # after the previous step's copy_blocks
    pkv.pkv_paged_decode_append(p["out"], s["q"], s["k_dec"], s["v_dec"], p["kc"], p["vc"], p["desc"],
                                s["tables"], s["lens"], s["max_len"], case.scale, 0, s["ws"], stream)
    pkv.pkv_kv_write(s["k_ch"], s["v_ch"], s["ch_slots"], p["kc"], p["vc"], p["desc"], s2)
    pkv.pkv_paged_prefill_chunk(p["cout"], s["cq"], s["cu"], s["st0"], ch.q_len, p["kc"], p["vc"], p["desc"],
                                s["ctab"], case.scale, s2)
    events[1].record(s2)
    stream.wait_event(events[1])
    pkv.pkv_copy_blocks(p["kc"], p["vc"], p["desc"], s["pairs"], stream)


def _split_setup():
    s = _setup()
    dev = torch.device("cuda")
    case, ch, plan = s["case"], s["ch"], s["plan"]
    from paged_kv_cache_160_gb300.planner import append_slots
    assert append_slots(case, plan) == list(plan.slots), "the decode tokens' slots are not their last positions"
    s.update(k_dec=case.k_new.to(dev), v_dec=case.v_new.to(dev), k_ch=ch.k_new.to(dev), v_ch=ch.v_new.to(dev),
             ch_slots=torch.tensor(list(plan.chunk_slots), dtype=torch.int64, device=dev))
    return s


@pytest.mark.parametrize("budget", [64, 72])
def test_split_step_under_a_budget_equals_the_serial_order(budget):
    """The schedule the bench times: under the same budget, the two-stream step equals the
    one-stream kv_write -> prefill -> decode -> copy_blocks bit for bit, eagerly and as a graph."""
    import paged_kv_cache_160_gb300 as pkv
    s = _split_setup()
    stream, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    events = (torch.cuda.Event(), torch.cuda.Event())
    serial, split, graphed = _fresh(s), _fresh(s), _fresh(s)
    with _budget(budget):
        with torch.cuda.stream(stream):
            _step(s, serial, stream)
            _split_step(s, split, stream, s2, events)
            _split_step(s, graphed, stream, s2, events)
        stream.synchronize()
        graphed["out"].fill_(float("nan"))
        graphed["cout"].fill_(float("nan"))
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
            for _ in range(2):
                _split_step(s, graphed, stream, s2, events)
    with torch.cuda.stream(stream):
        g.replay()
    stream.synchronize()
    assert pkv.pkv_get_device_error(stream) == 0
    assert not torch.isnan(serial["out"]).any() and not torch.isnan(serial["cout"]).any()
    _same(serial, split)
    _same(serial, graphed)
