// Host-side helpers shared by the libpkv entry points (not part of the public ABI).
#pragma once

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

inline int dtype_bytes(pkv_dtype d) { return d == PKV_FP8_E4M3 ? 1 : 2; }

// Shared checks of a cache descriptor; returns PKV_OK or the failing status.
pkv_status check_cache_desc(const pkv_cache_desc* c);

}  // namespace pkv
