// pkv_stream_tiles: the memory ceiling of a paged decode call, measured.
//
// It reads a given list of K/V tiles (16 pool rows of one (block, kv head), K and V) the way
// paged_decode reads them, and computes nothing: a persistent grid of one CTA per SM with
// 12 worker warps, each warp owning an equal contiguous range of the list and a ring of two
// stages of one K tile and one V tile, filled by bulk asynchronous copies completing on an
// mbarrier.  Each warp folds one word of every tile into a checksum so the reads cannot be
// dropped.  The benchmark times it on the same tile list as a decode call; the decode
// cannot move its bytes faster than this.
#include <algorithm>

#include "pkv_device.cuh"
#include "pkv_host.h"

namespace pkv {
namespace {

constexpr int kWarps = 12;
constexpr int kStages = 2;
constexpr int kRows = 16;

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}

struct StreamParams {
  const uint8_t* k;
  const uint8_t* v;
  const int32_t* tile_rows;   // first pool row of each tile
  int num_tiles;
  int tile_bytes;             // kRows * row bytes
  int64_t pool_rows;
  unsigned* checksum;
  unsigned* err;
};

__global__ void __launch_bounds__(kWarps * 32, 1) stream_tiles_kernel(const StreamParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bars[kWarps][kStages];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t W = int64_t(gridDim.x) * kWarps, w = int64_t(blockIdx.x) * kWarps + warp;
  const int t0 = int(w * p.num_tiles / W), t1 = int((w + 1) * p.num_tiles / W);
  if (lane == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&bars[warp][s], 1);
    fence_mbar_init();
  }
  __syncwarp();
  griddep_wait();
  griddep_launch_dependents();
  uint8_t* st = smem + int64_t(warp) * kStages * 2 * p.tile_bytes;
  const uint64_t pol = l2_policy_evict_first();
  uint32_t valid = 0;
  // Lane 0 starts tile t into stage s; a row outside the pool completes the phase empty.
  auto issue = [&](int t, int s) {
    uint64_t* bar = &bars[warp][s];
    const int64_t row = p.tile_rows[t];
    if (row < 0 || row + kRows > p.pool_rows) {
      set_error(p.err, PKV_DEVERR_BLOCK_ID);
      valid &= ~(1u << s);
      mbar_arrive(bar);
      return;
    }
    valid |= 1u << s;
    const int64_t off = row * (p.tile_bytes / kRows);
    mbar_arrive_expect_tx(bar, 2 * p.tile_bytes);
    bulk_load(st + s * 2 * p.tile_bytes, p.k + off, p.tile_bytes, bar, pol);
    bulk_load(st + s * 2 * p.tile_bytes + p.tile_bytes, p.v + off, p.tile_bytes, bar, pol);
  };
  if (lane == 0)
    for (int i = 0; i < kStages && t0 + i < t1; ++i) issue(t0 + i, i);
  unsigned acc = 0;
  for (int i = 0; t0 + i < t1; ++i) {
    const int s = i % kStages;
    if (!mbar_wait(&bars[warp][s], uint32_t(i / kStages) & 1u)) {
      // Give up: report, then wait (bounded) for this warp's copies still in flight.
      if (lane == 0) set_error(p.err, PKV_DEVERR_TIMEOUT);
      for (int k = i; k < min(t1 - t0, i + kStages); ++k)
        (void)mbar_wait(&bars[warp][k % kStages], uint32_t(k / kStages) & 1u);
      return;
    }
    if ((__shfl_sync(0xffffffffu, valid, 0) >> s) & 1u)
      acc ^= reinterpret_cast<const unsigned*>(st + s * 2 * p.tile_bytes)[lane];
    __syncwarp();                            // every lane's read of the stage is done
    if (lane == 0 && t0 + i + kStages < t1) issue(t0 + i + kStages, s);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc ^= __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0 && acc) atomicXor(p.checksum, acc);
}

}  // namespace
}  // namespace pkv

extern "C" pkv_status pkv_stream_tiles(const void* k_cache, const void* v_cache, const pkv_cache_desc* cache,
                                       const int32_t* tile_rows, int num_tiles, unsigned* checksum,
                                       pkv_stream_t stream) {
  using namespace pkv;
  pkv_status st = check_cache_desc(cache);
  if (st != PKV_OK) return st;
  if (num_tiles < 0) return PKV_ERR_INVALID_ARG;
  if (num_tiles == 0) return PKV_OK;
  if (!k_cache || !v_cache || !tile_rows || !checksum || !aligned16(k_cache) || !aligned16(v_cache) ||
      (reinterpret_cast<uintptr_t>(tile_rows) & 3u) || (reinterpret_cast<uintptr_t>(checksum) & 3u))
    return PKV_ERR_INVALID_ARG;
  const int tile_bytes = kRows * cache->head_dim * dtype_bytes(cache->kv_dtype);
  const size_t smem = size_t(kWarps) * kStages * 2 * tile_bytes;
  if (smem > 200 * 1024) return PKV_ERR_UNSUPPORTED;
  unsigned* err = error_word_ptr();
  if (!err) return PKV_ERR_CUDA;
  StreamParams prm;
  prm.k = static_cast<const uint8_t*>(k_cache);
  prm.v = static_cast<const uint8_t*>(v_cache);
  prm.tile_rows = tile_rows;
  prm.num_tiles = num_tiles;
  prm.tile_bytes = tile_bytes;
  prm.pool_rows = int64_t(cache->num_blocks) * cache->num_kv_heads * cache->block_size;
  prm.checksum = checksum;
  prm.err = err;
  if (cudaFuncSetAttribute(stream_tiles_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) !=
      cudaSuccess)
    return PKV_ERR_CUDA;
  const int grid = std::max(1, num_sms());
  return launch_pdl(stream_tiles_kernel, dim3(grid), dim3(kWarps * 32), smem, reinterpret_cast<cudaStream_t>(stream),
                    prm) == cudaSuccess
             ? PKV_OK
             : PKV_ERR_CUDA;
}
