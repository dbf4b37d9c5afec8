// kv_write (scatter of the step's new K/V rows into their slots) and copy_blocks (the copy
// step of copy-on-write).  Both move bytes with 16-byte vector loads/stores; both are
// bound by HBM traffic and, at serving sizes, by launch latency.
//
// Sources: "PagedAttention: manage the KV cache like virtual memory" §3.3 (each new token
// fills its sequence's last block); "Lecture 33 — KV Cache management" §2.2 (slot =
// block * block_size + offset) and §2.4 (copy-on-write copies the shared block).
#include "pkv_device.cuh"
#include "pkv_host.h"

namespace pkv {
namespace {

constexpr int kThreads = 256;

// Same dtype in and out: every (token, kv head) row is `chunks` 16-byte vectors.
__global__ void __launch_bounds__(kThreads) kv_write_copy_kernel(const uint4* __restrict__ k_new,
                                                                 const uint4* __restrict__ v_new,
                                                                 const int64_t* __restrict__ slots,
                                                                 uint4* __restrict__ k_cache,
                                                                 uint4* __restrict__ v_cache, int num_tokens,
                                                                 int num_kv_heads, int chunks, int block_size,
                                                                 int64_t num_slots, unsigned* err) {
  griddep_launch_dependents();   // a following decode may start its length-only prologue
  griddep_wait();                // the previous kernel (which may read this cache) is done
  const int64_t total = int64_t(num_tokens) * num_kv_heads * chunks;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < total; i += int64_t(gridDim.x) * blockDim.x) {
    const int c = int(i % chunks);
    const int64_t r = i / chunks;
    const int h = int(r % num_kv_heads);
    const int64_t t = r / num_kv_heads;
    const int64_t slot = slots[t];
    if (slot < 0) continue;                       // padding token
    if (slot >= num_slots) {
      if (c == 0 && h == 0) set_error(err, PKV_DEVERR_SLOT);
      continue;
    }
    const int64_t blk = slot / block_size, off = slot % block_size;
    const int64_t dst = ((blk * num_kv_heads + h) * block_size + off) * chunks + c;
    k_cache[dst] = __ldg(k_new + i);
    v_cache[dst] = __ldg(v_new + i);
  }
}

template <bool kBF16>
__device__ __forceinline__ float2 load2(const void* p) {
  if constexpr (kBF16) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
  } else {
    return __half22float2(*reinterpret_cast<const __half2*>(p));
  }
}

// f16/bf16 rows into an e4m3 cache: code = e4m3(x / scale[h]); 16 codes per thread.
template <bool kBF16>
__global__ void __launch_bounds__(kThreads) kv_write_quant_kernel(
    const uint8_t* __restrict__ k_new, const uint8_t* __restrict__ v_new, const int64_t* __restrict__ slots,
    uint4* __restrict__ k_cache, uint4* __restrict__ v_cache, const float* __restrict__ k_scale,
    const float* __restrict__ v_scale, int num_tokens, int num_kv_heads, int chunks, int block_size,
    int64_t num_slots, unsigned* err) {
  griddep_launch_dependents();
  griddep_wait();
  const int64_t total = int64_t(num_tokens) * num_kv_heads * chunks;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < total; i += int64_t(gridDim.x) * blockDim.x) {
    const int c = int(i % chunks);
    const int64_t r = i / chunks;
    const int h = int(r % num_kv_heads);
    const int64_t t = r / num_kv_heads;
    const int64_t slot = slots[t];
    if (slot < 0) continue;
    if (slot >= num_slots) {
      if (c == 0 && h == 0) set_error(err, PKV_DEVERR_SLOT);
      continue;
    }
    const int64_t blk = slot / block_size, off = slot % block_size;
    const int64_t dst = ((blk * num_kv_heads + h) * block_size + off) * chunks + c;
    const float ks = k_scale[h], vs = v_scale[h];
    uint32_t kw[4], vw[4];
    const uint8_t* kp = k_new + i * 32;           // 16 input elements of 2 bytes
    const uint8_t* vp = v_new + i * 32;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      float2 a = load2<kBF16>(kp + 8 * w), b = load2<kBF16>(kp + 8 * w + 4);
      kw[w] = f32x2_to_e4m3x2(__fdiv_rn(a.x, ks), __fdiv_rn(a.y, ks)) |
              (f32x2_to_e4m3x2(__fdiv_rn(b.x, ks), __fdiv_rn(b.y, ks)) << 16);
      a = load2<kBF16>(vp + 8 * w);
      b = load2<kBF16>(vp + 8 * w + 4);
      vw[w] = f32x2_to_e4m3x2(__fdiv_rn(a.x, vs), __fdiv_rn(a.y, vs)) |
              (f32x2_to_e4m3x2(__fdiv_rn(b.x, vs), __fdiv_rn(b.y, vs)) << 16);
    }
    k_cache[dst] = make_uint4(kw[0], kw[1], kw[2], kw[3]);
    v_cache[dst] = make_uint4(vw[0], vw[1], vw[2], vw[3]);
  }
}

// One CTA per (pair, K or V): copies the whole block of `chunks` 16-byte vectors.
__global__ void __launch_bounds__(kThreads) copy_blocks_kernel(uint4* __restrict__ k_cache,
                                                               uint4* __restrict__ v_cache,
                                                               const int32_t* __restrict__ pairs, int num_pairs,
                                                               int num_blocks, int64_t chunks, unsigned* err) {
  griddep_launch_dependents();
  griddep_wait();
  const int pair = blockIdx.x;
  const int32_t src = pairs[2 * pair], dst = pairs[2 * pair + 1];
  // A pair is applied only when both ids are in the pool, its dst is nobody's src and no
  // other pair writes the same dst.
  bool bad = src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks;
  for (int j = threadIdx.x; j < num_pairs && !bad; j += blockDim.x) {
    if (pairs[2 * j] == dst || (j != pair && pairs[2 * j + 1] == dst)) bad = true;
  }
  bad = __syncthreads_or(bad);
  if (bad) {
    if (threadIdx.x == 0 && blockIdx.y == 0) set_error(err, PKV_DEVERR_COPY_PAIR);
    return;
  }
  uint4* cache = blockIdx.y == 0 ? k_cache : v_cache;
  const uint4* s = cache + int64_t(src) * chunks;
  uint4* d = cache + int64_t(dst) * chunks;
  for (int64_t i = threadIdx.x; i < chunks; i += blockDim.x) d[i] = s[i];
}

// One CTA per (pair, K or V) between two pools of the same block layout, either of which may
// be pinned host memory (Grace reaches it over NVLink-C2C).  Each thread keeps four 16-byte
// loads in flight, so a block is read with few round trips even from host memory.
__global__ void __launch_bounds__(kThreads) swap_blocks_kernel(uint4* __restrict__ dst_k, uint4* __restrict__ dst_v,
                                                               const uint4* __restrict__ src_k,
                                                               const uint4* __restrict__ src_v,
                                                               const int32_t* __restrict__ pairs, int num_pairs,
                                                               int src_blocks, int dst_blocks, int64_t chunks,
                                                               unsigned* err) {
  griddep_launch_dependents();
  griddep_wait();
  const int pair = blockIdx.x;
  const int32_t src = pairs[2 * pair], dst = pairs[2 * pair + 1];
  // Applied only when both ids are inside their pools and no other pair writes the same dst.
  bool bad = src < 0 || src >= src_blocks || dst < 0 || dst >= dst_blocks;
  for (int j = threadIdx.x; j < num_pairs && !bad; j += blockDim.x) {
    if (j != pair && pairs[2 * j + 1] == dst) bad = true;
  }
  bad = __syncthreads_or(bad);
  if (bad) {
    if (threadIdx.x == 0 && blockIdx.y == 0) set_error(err, PKV_DEVERR_COPY_PAIR);
    return;
  }
  const uint4* sp = (blockIdx.y == 0 ? src_k : src_v) + int64_t(src) * chunks;
  uint4* dp = (blockIdx.y == 0 ? dst_k : dst_v) + int64_t(dst) * chunks;
  constexpr int kUnroll = 4;
  int64_t i = threadIdx.x;
  for (; i + (kUnroll - 1) * int64_t(blockDim.x) < chunks; i += kUnroll * int64_t(blockDim.x)) {
    uint4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) v[u] = sp[i + u * int64_t(blockDim.x)];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) dp[i + u * int64_t(blockDim.x)] = v[u];
  }
  for (; i < chunks; i += blockDim.x) dp[i] = sp[i];
}

// One 16-byte chunk per thread: these kernels are latency-bound at serving sizes, so every
// thread should issue its loads once rather than loop.
int grid_for(int64_t work) {
  const int64_t per = kThreads;
  int64_t g = (work + per - 1) / per;
  const int cap = num_sms() > 0 ? num_sms() * 64 : 8192;
  if (g > cap) g = cap;
  return g < 1 ? 1 : int(g);
}

}  // namespace
}  // namespace pkv

extern "C" {

pkv_status pkv_kv_write(const void* k_new, const void* v_new, pkv_dtype in_dtype, int num_tokens,
                        const int64_t* slot_mapping, void* k_cache, void* v_cache, const pkv_cache_desc* cache,
                        pkv_stream_t stream) {
  using namespace pkv;
  pkv_status st = check_cache_desc(cache);
  if (st != PKV_OK) return st;
  if (num_tokens < 0) return PKV_ERR_INVALID_ARG;
  if (num_tokens == 0) return PKV_OK;
  if (!k_new || !v_new || !slot_mapping || !k_cache || !v_cache) return PKV_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache) ||
      (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
    return PKV_ERR_INVALID_ARG;
  if (in_dtype != PKV_F16 && in_dtype != PKV_BF16 && in_dtype != PKV_FP8_E4M3) return PKV_ERR_INVALID_ARG;
  unsigned* err = error_word_ptr();
  if (!err) return PKV_ERR_CUDA;
  const int64_t num_slots = int64_t(cache->num_blocks) * cache->block_size;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (in_dtype == cache->kv_dtype) {
    const int chunks = cache->head_dim * dtype_bytes(in_dtype) / 16;
    const int64_t work = int64_t(num_tokens) * cache->num_kv_heads * chunks;
    if (launch_pdl(kv_write_copy_kernel, dim3(grid_for(work)), dim3(kThreads), 0, s,
                   static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), slot_mapping,
                   static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), num_tokens, cache->num_kv_heads,
                   chunks, cache->block_size, num_slots, err) != cudaSuccess)
      return PKV_ERR_CUDA;
  } else if (cache->kv_dtype == PKV_FP8_E4M3 && (in_dtype == PKV_F16 || in_dtype == PKV_BF16)) {
    const int chunks = cache->head_dim / 16;
    const int64_t work = int64_t(num_tokens) * cache->num_kv_heads * chunks;
    auto kern = in_dtype == PKV_BF16 ? kv_write_quant_kernel<true> : kv_write_quant_kernel<false>;
    if (launch_pdl(kern, dim3(grid_for(work)), dim3(kThreads), 0, s, static_cast<const uint8_t*>(k_new),
                   static_cast<const uint8_t*>(v_new), slot_mapping, static_cast<uint4*>(k_cache),
                   static_cast<uint4*>(v_cache), cache->k_scale, cache->v_scale, num_tokens, cache->num_kv_heads,
                   chunks, cache->block_size, num_slots, err) != cudaSuccess)
      return PKV_ERR_CUDA;
  } else {
    return PKV_ERR_UNSUPPORTED;
  }
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

pkv_status pkv_copy_blocks(void* k_cache, void* v_cache, const pkv_cache_desc* cache, const int32_t* block_pairs,
                           int num_pairs, pkv_stream_t stream) {
  using namespace pkv;
  pkv_status st = check_cache_desc(cache);
  if (st != PKV_OK) return st;
  if (num_pairs < 0) return PKV_ERR_INVALID_ARG;
  if (num_pairs == 0) return PKV_OK;
  if (!k_cache || !v_cache || !block_pairs) return PKV_ERR_INVALID_ARG;
  if (!aligned16(k_cache) || !aligned16(v_cache) || (reinterpret_cast<uintptr_t>(block_pairs) & 7u))
    return PKV_ERR_INVALID_ARG;
  if (num_pairs > 65535) return PKV_ERR_UNSUPPORTED;
  unsigned* err = error_word_ptr();
  if (!err) return PKV_ERR_CUDA;
  const int64_t block_bytes =
      int64_t(cache->num_kv_heads) * cache->block_size * cache->head_dim * dtype_bytes(cache->kv_dtype);
  const int64_t chunks = block_bytes / 16;
  dim3 grid(num_pairs, 2);
  if (launch_pdl(copy_blocks_kernel, grid, dim3(kThreads), 0, reinterpret_cast<cudaStream_t>(stream),
                 static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), block_pairs, num_pairs,
                 cache->num_blocks, chunks, err) != cudaSuccess)
    return PKV_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

pkv_status pkv_swap_blocks(void* dst_k, void* dst_v, int dst_num_blocks, const void* src_k, const void* src_v,
                           int src_num_blocks, const pkv_cache_desc* layout, const int32_t* block_pairs,
                           int num_pairs, pkv_stream_t stream) {
  using namespace pkv;
  pkv_status st = check_cache_desc(layout);
  if (st != PKV_OK) return st;
  if (num_pairs < 0 || dst_num_blocks <= 0 || src_num_blocks <= 0) return PKV_ERR_INVALID_ARG;
  if (num_pairs == 0) return PKV_OK;
  if (!dst_k || !dst_v || !src_k || !src_v || !block_pairs) return PKV_ERR_INVALID_ARG;
  if (!aligned16(dst_k) || !aligned16(dst_v) || !aligned16(src_k) || !aligned16(src_v) ||
      (reinterpret_cast<uintptr_t>(block_pairs) & 7u))
    return PKV_ERR_INVALID_ARG;
  if (num_pairs > 65535) return PKV_ERR_UNSUPPORTED;
  unsigned* err = error_word_ptr();
  if (!err) return PKV_ERR_CUDA;
  const int64_t block_bytes =
      int64_t(layout->num_kv_heads) * layout->block_size * layout->head_dim * dtype_bytes(layout->kv_dtype);
  if (launch_pdl(swap_blocks_kernel, dim3(num_pairs, 2), dim3(kThreads), 0, reinterpret_cast<cudaStream_t>(stream),
                 static_cast<uint4*>(dst_k), static_cast<uint4*>(dst_v), static_cast<const uint4*>(src_k),
                 static_cast<const uint4*>(src_v), block_pairs, num_pairs, src_num_blocks, dst_num_blocks,
                 block_bytes / 16, err) != cudaSuccess)
    return PKV_ERR_CUDA;
  return PKV_OK;
}

}  // extern "C"
