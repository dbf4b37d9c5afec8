"""The allocation-free decode entry point against the workspace one (GPU).

pkv_paged_decode_noalloc serves callers that cannot allocate device memory at decode
time — a plain C host with no device allocator of its own, or a serving loop that must
not call cudaMalloc on its hot path because it can synchronise the device.  It keeps its
split-KV scratch in one fixed array inside the library.  This test calls it through the
C ABI twice in a row (the second call finds the first call's leftovers in the shared
array) and checks both results against pkv_paged_decode with a caller-owned workspace.
Both calls run the same kernels with the same split of the work, so the outputs must agree
bit for bit: a tolerance could hide a scratch-layout mistake.  It also checks that the
array holds the largest call this device accepts, and that a larger call is refused.

The file name sorts last so that a run stopping at the first failure has already run
every other test.
"""
import ctypes

import pytest
import torch

import synth
from tests.harness import product_plan

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")


@pytest.mark.parametrize("builder,part", [(synth.qwen7b_gqa_config, 0),
                                          (lambda: synth.make_decode_case("noalloc_e4m3", 90, [1, 40, 700, 3000],
                                                                          16, 4, 128, "bf16", "e4m3"), 512)])
def test_noalloc_matches_workspace_entry_point_twice(builder, part):
    import paged_kv_cache_160_gb300 as pkv
    case = builder()
    plan = product_plan(case)
    dev = torch.device("cuda")
    kc, vc = case.k_cache.to(dev), case.v_cache.to(dev)
    ks = case.k_scale.to(dev) if case.k_scale is not None else None
    vs = case.v_scale.to(dev) if case.v_scale is not None else None
    desc = pkv.cache_desc(kc, ks, vs)
    q = case.q.to(dev)
    tables = torch.tensor(plan.tables, dtype=torch.int32, device=dev)
    lens = torch.tensor(plan.lens, dtype=torch.int32, device=dev)
    max_len = max(plan.lens)
    ws_bytes = pkv.pkv_decode_workspace_bytes(case.num_seqs, case.num_heads, case.num_kv_heads, case.head_dim, 16,
                                              max_len, part)
    assert 0 < ws_bytes <= pkv.pkv_noalloc_scratch_bytes()
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
    ref = torch.empty_like(q)
    pkv.pkv_paged_decode(ref, q, kc, vc, desc, tables, lens, max_len, case.scale, part, ws)
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(2):
        out = torch.full_like(q, float("nan"))
        st = pkv.lib.pkv_paged_decode_noalloc(out.data_ptr(), q.data_ptr(), pkv._binding.pkv_dtype_of(q),
                                              case.num_seqs, case.num_heads, kc.data_ptr(), vc.data_ptr(),
                                              ctypes.byref(desc), tables.data_ptr(), tables.shape[1],
                                              lens.data_ptr(), max_len, case.scale, part, stream)
        assert st == 0
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
    assert pkv.pkv_get_device_error() == 0


def _largest_supported_need(pkv):
    """Scratch bytes of the largest call the decode accepts on this device: it depends on
    the SM count, the group size (at most 8) and head_dim (at most 128), not on the number
    of sequences or their lengths."""
    return max(pkv.pkv_decode_workspace_bytes(1, g * 8, 8, d, 16, 4096, 0) for g in (1, 2, 4, 8) for d in (64, 128))


def test_noalloc_scratch_holds_every_supported_call_on_this_gpu():
    import paged_kv_cache_160_gb300 as pkv
    need = _largest_supported_need(pkv)
    assert 0 < need <= pkv.pkv_noalloc_scratch_bytes(), need


def test_noalloc_refuses_more_scratch_than_it_holds():
    """A call needing more scratch than the array holds is refused before anything is
    enqueued.  Such a call exists only on a device with more SMs than the scratch was sized
    for; the call below passes placeholder pointers, so it is made only when the library's
    own size function says the scratch is too small for it."""
    import paged_kv_cache_160_gb300 as pkv
    from paged_kv_cache_160_gb300._binding import CacheDesc
    need = pkv.pkv_decode_workspace_bytes(16, 64, 8, 128, 16, 4096, 0)
    if need <= pkv.pkv_noalloc_scratch_bytes():
        pytest.skip(f"every supported call fits the scratch on this device ({need} bytes at most)")
    desc = CacheDesc(1 << 20, 8, 16, 128, 1, None, None)
    st = pkv.lib.pkv_paged_decode_noalloc(16, 16, 1, 16, 64, 16, 16, ctypes.byref(desc), 16, 256, 16, 4096, 0.1,
                                          0, None)
    assert st == 3                                 # PKV_ERR_WORKSPACE, nothing enqueued
