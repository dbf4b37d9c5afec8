"""ctypes binding of libpkv (``include/pkv.h``): argument marshalling only.

Every function here has the C entry point's name and forwards torch tensors as raw
device pointers; all computation happens in the library's CUDA kernels.  There is no
fallback: if ``libpkv.so`` is missing, importing this module raises, and a call with a
CPU tensor raises.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_float, c_int, c_int32, c_int64, c_size_t, c_void_p
from typing import List, Optional, Sequence, Tuple

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libpkv.so")

PKV_OK = 0
STATUS_NAMES = {0: "PKV_OK", 1: "PKV_ERR_INVALID_ARG", 2: "PKV_ERR_UNSUPPORTED", 3: "PKV_ERR_WORKSPACE",
                4: "PKV_ERR_CUDA", 5: "PKV_ERR_NO_BLOCKS", 6: "PKV_ERR_DEVICE_CHECK"}
PKV_F16, PKV_BF16, PKV_FP8_E4M3 = 0, 1, 2
DEVERR = {"block_id": 1, "context_len": 2, "slot": 4, "copy_pair": 8, "timeout": 16, "chunk": 32}


class PkvError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)}")


class NoBlocksError(PkvError):
    pass


class CacheDesc(ctypes.Structure):
    _fields_ = [("num_blocks", c_int), ("num_kv_heads", c_int), ("block_size", c_int), ("head_dim", c_int),
                ("kv_dtype", c_int), ("k_scale", c_void_p), ("v_scale", c_void_p)]


def _load() -> ctypes.CDLL:
    if not os.path.exists(_LIB_PATH):
        raise ImportError(f"libpkv.so is not built ({_LIB_PATH}); run `python paged_kv_cache_160_gb300/build.py`")
    lib = ctypes.CDLL(_LIB_PATH)
    S = c_int
    lib.pkv_status_string.restype = ctypes.c_char_p
    lib.pkv_status_string.argtypes = [c_int]
    lib.pkv_version.restype = c_int
    lib.pkv_kv_write.restype = S
    lib.pkv_kv_write.argtypes = [c_void_p, c_void_p, c_int, c_int, c_void_p, c_void_p, c_void_p,
                                 POINTER(CacheDesc), c_void_p]
    lib.pkv_copy_blocks.restype = S
    lib.pkv_copy_blocks.argtypes = [c_void_p, c_void_p, POINTER(CacheDesc), c_void_p, c_int, c_void_p]
    lib.pkv_check_bounded_wait.restype = S
    lib.pkv_check_bounded_wait.argtypes = [ctypes.c_uint64, c_void_p]
    lib.pkv_stream_tiles.restype = S
    lib.pkv_stream_tiles.argtypes = [c_void_p, c_void_p, POINTER(CacheDesc), c_void_p, c_int, c_void_p, c_void_p]
    lib.pkv_swap_blocks.restype = S
    lib.pkv_swap_blocks.argtypes = [c_void_p, c_void_p, c_int, c_void_p, c_void_p, c_int, POINTER(CacheDesc),
                                    c_void_p, c_int, c_void_p]
    lib.pkv_decode_workspace_bytes.restype = c_size_t
    lib.pkv_decode_workspace_bytes.argtypes = [c_int] * 7
    lib.pkv_paged_decode.restype = S
    lib.pkv_paged_decode.argtypes = [c_void_p, c_void_p, c_int, c_int, c_int, c_void_p, c_void_p,
                                     POINTER(CacheDesc), c_void_p, c_int, c_void_p, c_int, c_float, c_int,
                                     c_void_p, c_size_t, c_void_p]
    lib.pkv_paged_decode_append.restype = S
    lib.pkv_paged_decode_append.argtypes = [c_void_p, c_void_p, c_int, c_int, c_int, c_void_p, c_void_p, c_void_p,
                                            c_void_p, POINTER(CacheDesc), c_void_p, c_int, c_void_p, c_int, c_float,
                                            c_int, c_void_p, c_size_t, c_void_p]
    lib.pkv_noalloc_scratch_bytes.restype = c_size_t
    lib.pkv_noalloc_scratch_bytes.argtypes = []
    lib.pkv_set_decode_sm_budget.restype = S
    lib.pkv_set_decode_sm_budget.argtypes = [c_int]
    lib.pkv_get_decode_sm_budget.restype = c_int
    lib.pkv_get_decode_sm_budget.argtypes = []
    lib.pkv_paged_decode_noalloc.restype = S
    lib.pkv_paged_decode_noalloc.argtypes = [c_void_p, c_void_p, c_int, c_int, c_int, c_void_p, c_void_p,
                                             POINTER(CacheDesc), c_void_p, c_int, c_void_p, c_int, c_float, c_int,
                                             c_void_p]
    lib.pkv_paged_prefill_chunk.restype = S
    lib.pkv_paged_prefill_chunk.argtypes = [c_void_p, c_void_p, c_int, c_void_p, c_void_p, c_int, c_int, c_int,
                                            c_int, c_void_p, c_void_p, POINTER(CacheDesc), c_void_p, c_int,
                                            c_float, c_void_p]
    lib.pkv_get_device_error.restype = S
    lib.pkv_get_device_error.argtypes = [POINTER(c_int), c_void_p]
    # block manager
    BM = c_void_p
    lib.pkv_bm_create.restype = S
    lib.pkv_bm_create.argtypes = [c_int, c_int, POINTER(c_void_p)]
    lib.pkv_bm_destroy.restype = None
    lib.pkv_bm_destroy.argtypes = [BM]
    lib.pkv_bm_import_seq.restype = S
    lib.pkv_bm_import_seq.argtypes = [BM, c_int64, POINTER(c_int32), c_int, c_int]
    lib.pkv_bm_allocate.restype = S
    lib.pkv_bm_allocate.argtypes = [BM, c_int64, c_int]
    lib.pkv_bm_append_slot.restype = S
    lib.pkv_bm_append_slot.argtypes = [BM, c_int64, POINTER(c_int64), POINTER(c_int32), POINTER(c_int32)]
    lib.pkv_bm_append_slots.restype = S
    lib.pkv_bm_append_slots.argtypes = [BM, c_int64, c_int, POINTER(c_int64), POINTER(c_int32), POINTER(c_int)]
    lib.pkv_bm_step_decode.restype = S
    lib.pkv_bm_step_decode.argtypes = [BM, POINTER(c_int64), c_int, c_int, POINTER(c_int64), POINTER(c_int32),
                                       POINTER(c_int), POINTER(c_int32), POINTER(c_int32)]
    lib.pkv_bm_fork.restype = S
    lib.pkv_bm_fork.argtypes = [BM, c_int64, c_int64]
    lib.pkv_bm_free.restype = S
    lib.pkv_bm_free.argtypes = [BM, c_int64]
    lib.pkv_bm_export.restype = S
    lib.pkv_bm_export.argtypes = [BM, POINTER(c_int64), c_int, c_int, POINTER(c_int32), POINTER(c_int32)]
    lib.pkv_bm_allocate_cached.restype = S
    lib.pkv_bm_allocate_cached.argtypes = [BM, c_int64, POINTER(c_int32), c_int, POINTER(c_int)]
    lib.pkv_bm_block_hash.restype = c_int
    lib.pkv_bm_block_hash.argtypes = [BM, c_int, POINTER(ctypes.c_uint64)]
    lib.pkv_bm_num_cached.restype = c_int
    lib.pkv_bm_num_cached.argtypes = [BM]
    lib.pkv_bm_set_host_pool.restype = S
    lib.pkv_bm_set_host_pool.argtypes = [BM, c_int]
    lib.pkv_bm_swap_out.restype = S
    lib.pkv_bm_swap_out.argtypes = [BM, c_int64, POINTER(c_int32), c_int, POINTER(c_int)]
    lib.pkv_bm_swap_in.restype = S
    lib.pkv_bm_swap_in.argtypes = [BM, c_int64, POINTER(c_int32), c_int, POINTER(c_int)]
    lib.pkv_bm_num_free_host.restype = c_int
    lib.pkv_bm_num_free_host.argtypes = [BM]
    lib.pkv_bm_is_swapped.restype = c_int
    lib.pkv_bm_is_swapped.argtypes = [BM, c_int64]
    lib.pkv_bm_ref_cnt.restype = c_int
    lib.pkv_bm_ref_cnt.argtypes = [BM, c_int]
    lib.pkv_bm_num_free.restype = c_int
    lib.pkv_bm_num_free.argtypes = [BM]
    lib.pkv_bm_free_queue.restype = c_int
    lib.pkv_bm_free_queue.argtypes = [BM, POINTER(c_int32), c_int]
    return lib


lib = _load()


def _check(status: int, what: str) -> None:
    if status == PKV_OK:
        return
    if status == 5:
        raise NoBlocksError(status, what)
    raise PkvError(status, what)


# ---------------------------------------------------------------------------------------
# device calls
# ---------------------------------------------------------------------------------------

_DT = {torch.float16: PKV_F16, torch.bfloat16: PKV_BF16, torch.uint8: PKV_FP8_E4M3,
       torch.float8_e4m3fn: PKV_FP8_E4M3}


def pkv_dtype_of(t: torch.Tensor) -> int:
    try:
        return _DT[t.dtype]
    except KeyError:
        raise TypeError(f"unsupported dtype {t.dtype}") from None


def _dev(t: Optional[torch.Tensor], name: str) -> int:
    if t is None:
        return 0
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (libpkv has no CPU path)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def cache_desc(k_cache: torch.Tensor, k_scale: Optional[torch.Tensor] = None,
               v_scale: Optional[torch.Tensor] = None) -> CacheDesc:
    """Descriptor of a pool tensor shaped [num_blocks, num_kv_heads, block_size, head_dim].

    The descriptor holds raw pointers to the scale tensors, so it keeps references to
    them: the memory stays valid for as long as the descriptor lives.
    """
    nb, hkv, bs, d = k_cache.shape
    desc = CacheDesc(nb, hkv, bs, d, pkv_dtype_of(k_cache), _dev(k_scale, "k_scale") or None,
                     _dev(v_scale, "v_scale") or None)
    desc._keep = (k_scale, v_scale)
    return desc


def pkv_kv_write(k_new: torch.Tensor, v_new: torch.Tensor, slot_mapping: torch.Tensor, k_cache: torch.Tensor,
                 v_cache: torch.Tensor, desc: CacheDesc, stream=None) -> None:
    assert slot_mapping.dtype == torch.int64
    _check(lib.pkv_kv_write(_dev(k_new, "k_new"), _dev(v_new, "v_new"), pkv_dtype_of(k_new), k_new.shape[0],
                            _dev(slot_mapping, "slot_mapping"), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
                            ctypes.byref(desc), _stream(stream)), "pkv_kv_write")


def pkv_copy_blocks(k_cache: torch.Tensor, v_cache: torch.Tensor, desc: CacheDesc, block_pairs: torch.Tensor,
                    stream=None) -> None:
    assert block_pairs.dtype == torch.int32
    _check(lib.pkv_copy_blocks(_dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"), ctypes.byref(desc),
                               _dev(block_pairs, "block_pairs"), block_pairs.shape[0], _stream(stream)),
           "pkv_copy_blocks")


def pkv_check_bounded_wait(limit_ns: int, stream=None) -> None:
    """Run the shared bounded wait on a barrier nothing arrives on; it sets the timeout bit."""
    _check(lib.pkv_check_bounded_wait(int(limit_ns), _stream(stream)), "pkv_check_bounded_wait")


def pkv_stream_tiles(k_cache: torch.Tensor, v_cache: torch.Tensor, desc: CacheDesc, tile_rows: torch.Tensor,
                     checksum: torch.Tensor, stream=None) -> None:
    """Read the listed K/V tiles with the decode's memory pipeline and nothing else (a
    measurement of the decode's memory ceiling); tile_rows holds each tile's first pool row."""
    assert tile_rows.dtype == torch.int32 and checksum.dtype == torch.int32 and checksum.numel() >= 1
    _check(lib.pkv_stream_tiles(_dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"), ctypes.byref(desc),
                                _dev(tile_rows, "tile_rows"), tile_rows.numel(), _dev(checksum, "checksum"),
                                _stream(stream)), "pkv_stream_tiles")


def _dev_or_pinned(t: torch.Tensor, name: str) -> int:
    """Device address of a CUDA tensor, or of a pinned host tensor (unified addressing)."""
    if not (t.is_cuda or t.is_pinned()):
        raise ValueError(f"{name} must be a CUDA tensor or pinned host memory")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def pkv_swap_blocks(dst_k: torch.Tensor, dst_v: torch.Tensor, src_k: torch.Tensor, src_v: torch.Tensor,
                    desc: CacheDesc, block_pairs: torch.Tensor, stream=None) -> None:
    """Block copies between two pools of ``desc``'s layout; either may be pinned host memory."""
    assert block_pairs.dtype == torch.int32
    _check(lib.pkv_swap_blocks(_dev_or_pinned(dst_k, "dst_k"), _dev_or_pinned(dst_v, "dst_v"), dst_k.shape[0],
                               _dev_or_pinned(src_k, "src_k"), _dev_or_pinned(src_v, "src_v"), src_k.shape[0],
                               ctypes.byref(desc), _dev(block_pairs, "block_pairs"), block_pairs.shape[0],
                               _stream(stream)),
           "pkv_swap_blocks")


def pkv_decode_workspace_bytes(num_seqs: int, num_heads: int, num_kv_heads: int, head_dim: int, block_size: int,
                               max_context_len: int, partition_size: int) -> int:
    return int(lib.pkv_decode_workspace_bytes(num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                                              max_context_len, partition_size))


def pkv_paged_decode(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                     desc: CacheDesc, block_tables: torch.Tensor, context_lens: torch.Tensor, max_context_len: int,
                     scale: float, partition_size: int, workspace: torch.Tensor, stream=None) -> None:
    """out, q, block_tables and context_lens may be pinned host memory (read and written in place)."""
    assert block_tables.dtype == torch.int32 and context_lens.dtype == torch.int32
    _check(lib.pkv_paged_decode(_dev_or_pinned(out, "out"), _dev_or_pinned(q, "q"), pkv_dtype_of(q), q.shape[0],
                                q.shape[1], _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"), ctypes.byref(desc),
                                _dev_or_pinned(block_tables, "block_tables"), block_tables.shape[1],
                                _dev_or_pinned(context_lens, "context_lens"), int(max_context_len), float(scale),
                                int(partition_size), _dev(workspace, "workspace"),
                                workspace.numel() * workspace.element_size(), _stream(stream)),
           "pkv_paged_decode")


def pkv_paged_decode_append(out: torch.Tensor, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                            k_cache: torch.Tensor, v_cache: torch.Tensor, desc: CacheDesc, block_tables: torch.Tensor,
                            context_lens: torch.Tensor, max_context_len: int, scale: float, partition_size: int,
                            workspace: torch.Tensor, stream=None) -> None:
    """Writes each sequence's new K/V row (k_new, v_new: [num_seqs, num_kv_heads, head_dim], q's dtype)
    at position context_lens[i] - 1, then decodes as pkv_paged_decode.  out, q, k_new, v_new,
    block_tables and context_lens may be pinned host memory (read and written in place)."""
    assert block_tables.dtype == torch.int32 and context_lens.dtype == torch.int32
    assert k_new.dtype == q.dtype and v_new.dtype == q.dtype and k_new.shape == v_new.shape
    assert k_new.shape[0] == q.shape[0] and k_new.is_contiguous() and v_new.is_contiguous()
    _check(lib.pkv_paged_decode_append(_dev_or_pinned(out, "out"), _dev_or_pinned(q, "q"), pkv_dtype_of(q),
                                       q.shape[0], q.shape[1], _dev_or_pinned(k_new, "k_new"),
                                       _dev_or_pinned(v_new, "v_new"), _dev(k_cache, "k_cache"),
                                       _dev(v_cache, "v_cache"), ctypes.byref(desc),
                                       _dev_or_pinned(block_tables, "block_tables"), block_tables.shape[1],
                                       _dev_or_pinned(context_lens, "context_lens"), int(max_context_len), float(scale),
                                       int(partition_size), _dev(workspace, "workspace"),
                                       workspace.numel() * workspace.element_size(), _stream(stream)),
           "pkv_paged_decode_append")


def pkv_noalloc_scratch_bytes() -> int:
    return int(lib.pkv_noalloc_scratch_bytes())


def pkv_set_decode_sm_budget(num_sms: int) -> None:
    """SMs (persistent CTAs) the decode calls made after this use; 0 = every SM."""
    _check(lib.pkv_set_decode_sm_budget(int(num_sms)), "pkv_set_decode_sm_budget")


def pkv_get_decode_sm_budget() -> int:
    return int(lib.pkv_get_decode_sm_budget())


def pkv_paged_decode_noalloc(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                             desc: CacheDesc, block_tables: torch.Tensor, context_lens: torch.Tensor,
                             max_context_len: int, scale: float, partition_size: int, stream=None) -> None:
    """pkv_paged_decode with the library's own fixed scratch array instead of a workspace."""
    assert block_tables.dtype == torch.int32 and context_lens.dtype == torch.int32
    _check(lib.pkv_paged_decode_noalloc(_dev(out, "out"), _dev(q, "q"), pkv_dtype_of(q), q.shape[0], q.shape[1],
                                        _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"), ctypes.byref(desc),
                                        _dev(block_tables, "block_tables"), block_tables.shape[1],
                                        _dev(context_lens, "context_lens"), int(max_context_len), float(scale),
                                        int(partition_size), _stream(stream)), "pkv_paged_decode_noalloc")


def pkv_paged_prefill_chunk(out: torch.Tensor, q: torch.Tensor, cu_q_lens: torch.Tensor, q_start_pos: torch.Tensor,
                            max_q_len: int, k_cache: torch.Tensor, v_cache: torch.Tensor, desc: CacheDesc,
                            block_tables: torch.Tensor, scale: float, stream=None) -> None:
    assert cu_q_lens.dtype == torch.int32 and q_start_pos.dtype == torch.int32
    _check(lib.pkv_paged_prefill_chunk(_dev(out, "out"), _dev(q, "q"), pkv_dtype_of(q), _dev(cu_q_lens, "cu_q_lens"),
                                       _dev(q_start_pos, "q_start_pos"), q_start_pos.shape[0], q.shape[0],
                                       int(max_q_len), q.shape[1], _dev(k_cache, "k_cache"),
                                       _dev(v_cache, "v_cache"), ctypes.byref(desc),
                                       _dev(block_tables, "block_tables"), block_tables.shape[1], float(scale),
                                       _stream(stream)), "pkv_paged_prefill_chunk")


def pkv_get_device_error(stream=None) -> int:
    code = c_int(0)
    st = lib.pkv_get_device_error(ctypes.byref(code), _stream(stream))
    if st not in (PKV_OK, 6):
        _check(st, "pkv_get_device_error")
    return int(code.value)


# ---------------------------------------------------------------------------------------
# host block manager
# ---------------------------------------------------------------------------------------

def _i32(xs: Sequence[int]):
    return (c_int32 * max(1, len(xs)))(*xs)


class BlockManager:
    """Owner of a ``pkv_block_manager`` handle; methods map 1:1 onto ``pkv_bm_*``."""

    def __init__(self, num_blocks: int, block_size: int):
        h = c_void_p()
        _check(lib.pkv_bm_create(num_blocks, block_size, ctypes.byref(h)), "pkv_bm_create")
        self._h = h
        self.num_blocks = num_blocks
        self.block_size = block_size

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            lib.pkv_bm_destroy(h)
            self._h = None

    def import_seq(self, seq: int, blocks: Sequence[int], n_tokens: int) -> None:
        _check(lib.pkv_bm_import_seq(self._h, seq, _i32(blocks), len(blocks), n_tokens), "pkv_bm_import_seq")

    def allocate(self, seq: int, n_tokens: int) -> None:
        _check(lib.pkv_bm_allocate(self._h, seq, n_tokens), "pkv_bm_allocate")

    def append_slot(self, seq: int) -> Tuple[int, Optional[Tuple[int, int]]]:
        slot, cs, cd = c_int64(), c_int32(), c_int32()
        _check(lib.pkv_bm_append_slot(self._h, seq, ctypes.byref(slot), ctypes.byref(cs), ctypes.byref(cd)),
               "pkv_bm_append_slot")
        return slot.value, (None if cs.value < 0 else (cs.value, cd.value))

    def append_slots(self, seq: int, n: int):
        slots = (c_int64 * max(1, n))()
        pairs = (c_int32 * max(2, 2 * n))()
        nc = c_int()
        _check(lib.pkv_bm_append_slots(self._h, seq, n, slots, pairs, ctypes.byref(nc)), "pkv_bm_append_slots")
        return list(slots[:n]), [(pairs[2 * i], pairs[2 * i + 1]) for i in range(nc.value)]

    def step_decode(self, seqs: Sequence[int], max_blocks: int):
        n = len(seqs)
        s = (c_int64 * max(1, n))(*seqs)
        slots = (c_int64 * max(1, n))()
        pairs = (c_int32 * max(2, 2 * n))()
        tables = (c_int32 * max(1, n * max_blocks))()
        lens = (c_int32 * max(1, n))()
        nc = c_int()
        _check(lib.pkv_bm_step_decode(self._h, s, n, max_blocks, slots, pairs, ctypes.byref(nc), tables, lens),
               "pkv_bm_step_decode")
        tab = [list(tables[i * max_blocks:(i + 1) * max_blocks]) for i in range(n)]
        return list(slots[:n]), [(pairs[2 * i], pairs[2 * i + 1]) for i in range(nc.value)], tab, list(lens[:n])

    def fork(self, parent: int, child: int) -> None:
        _check(lib.pkv_bm_fork(self._h, parent, child), "pkv_bm_fork")

    def free(self, seq: int) -> None:
        _check(lib.pkv_bm_free(self._h, seq), "pkv_bm_free")

    def allocate_cached(self, seq: int, tokens: Sequence[int]) -> int:
        """Admit a prompt reusing its cached full-block prefix; returns the cached token count."""
        n = c_int()
        _check(lib.pkv_bm_allocate_cached(self._h, seq, _i32(tokens), len(tokens), ctypes.byref(n)),
               "pkv_bm_allocate_cached")
        return n.value

    def block_hash(self, block: int) -> Optional[int]:
        h = ctypes.c_uint64()
        r = lib.pkv_bm_block_hash(self._h, block, ctypes.byref(h))
        if r < 0:
            raise PkvError(1, "pkv_bm_block_hash: bad arguments")
        return h.value if r == 1 else None

    def num_cached(self) -> int:
        return lib.pkv_bm_num_cached(self._h)

    def set_host_pool(self, num_host_blocks: int) -> None:
        _check(lib.pkv_bm_set_host_pool(self._h, num_host_blocks), "pkv_bm_set_host_pool")

    def _swap(self, fn, name, seq: int, max_pairs: int):
        pairs = (c_int32 * max(1, 2 * max_pairs))()
        n = c_int()
        _check(fn(self._h, seq, pairs, max_pairs, ctypes.byref(n)), name)
        return [(pairs[2 * i], pairs[2 * i + 1]) for i in range(n.value)]

    def swap_out(self, seq: int, max_pairs: int = 1 << 16) -> List[Tuple[int, int]]:
        """(device block, host block) pairs, in table order."""
        return self._swap(lib.pkv_bm_swap_out, "pkv_bm_swap_out", seq, max_pairs)

    def swap_in(self, seq: int, max_pairs: int = 1 << 16) -> List[Tuple[int, int]]:
        """(host block, device block) pairs, in table order."""
        return self._swap(lib.pkv_bm_swap_in, "pkv_bm_swap_in", seq, max_pairs)

    def num_free_host(self) -> int:
        return lib.pkv_bm_num_free_host(self._h)

    def is_swapped(self, seq: int) -> int:
        return lib.pkv_bm_is_swapped(self._h, seq)

    def export(self, seqs: Sequence[int], max_blocks: int):
        n = len(seqs)
        s = (c_int64 * max(1, n))(*seqs)
        tables = (c_int32 * max(1, n * max_blocks))()
        lens = (c_int32 * max(1, n))()
        _check(lib.pkv_bm_export(self._h, s, n, max_blocks, tables, lens), "pkv_bm_export")
        return [list(tables[i * max_blocks:(i + 1) * max_blocks]) for i in range(n)], list(lens[:n])

    def ref_cnt(self, block: int) -> int:
        return int(lib.pkv_bm_ref_cnt(self._h, block))

    def num_free(self) -> int:
        return int(lib.pkv_bm_num_free(self._h))

    def free_queue(self):
        n = lib.pkv_bm_free_queue(self._h, None, 0)
        buf = (c_int32 * max(1, n))()
        lib.pkv_bm_free_queue(self._h, buf, n)
        return list(buf[:n])
