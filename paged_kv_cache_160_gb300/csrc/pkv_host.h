// Host-side helpers shared by the libpkv entry points (not part of the public ABI).
#pragma once

#include <utility>

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pkv.h"

namespace pkv {

// Device pointer of the library's error word on the current device (nullptr on failure).
unsigned* error_word_ptr();

// Streaming multiprocessors of the current device (0 on failure).
int num_sms();

// Current device ordinal (-1 on failure).
int current_device();

// Encodes a 2-D tiled tensor map (dim0 innermost).  Returns false when the driver entry
// point is unavailable or the driver rejects the arguments.
bool encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t dim0, uint64_t dim1,
                    uint64_t stride1_bytes, uint32_t box0, uint32_t box1, CUtensorMapSwizzle swizzle);

// Encodes a 3-D tiled tensor map (dim0 innermost).
bool encode_tmap_3d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t dim0, uint64_t dim1,
                    uint64_t dim2, uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box0, uint32_t box1,
                    uint32_t box2, CUtensorMapSwizzle swizzle);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// True when p points into memory allocated on the current device (cudaMalloc or a pool
// allocation), false for host, managed, unregistered or another device's memory, or when the
// query fails.  The runtime's error state is left clear.
bool on_current_device(const void* p);

inline int dtype_bytes(pkv_dtype d) { return d == PKV_FP8_E4M3 ? 1 : 2; }

// Shared checks of a cache descriptor; returns PKV_OK or the failing status.
pkv_status check_cache_desc(const pkv_cache_desc* c);

// The argument checks of the paged-decode entry points (no CUDA work is enqueued).  On
// PKV_OK, *need holds the workspace bytes the call needs (0 when num_seqs == 0).
pkv_status decode_check(const void* out, const void* q, pkv_dtype q_dtype, int num_seqs, int num_heads,
                        const void* k_cache, const void* v_cache, const pkv_cache_desc* cache,
                        const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                        int max_context_len, int partition_size, size_t* need);

#ifdef __CUDACC__
// Launch with programmatic stream serialization: the kernel may be scheduled while the
// previous kernel on the stream still runs, and must call griddep_wait() before it touches
// memory that kernel may write.
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kern)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}
#endif

}  // namespace pkv
