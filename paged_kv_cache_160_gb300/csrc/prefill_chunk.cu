// paged_prefill_chunk: causal attention of a prefill chunk over its paged history.
//
// Method ("Lecture 33 — KV Cache management" §4.2): a long prompt is cut into chunks; a
// chunk's tokens attend, with a causal mask, the KV of the chunks already cached plus the
// chunk itself.  Query row r of a chunk that starts at position q_start sits at position
// p = q_start + r and attends keys 0..p of its sequence, read through the block table
// (§2.2–§2.3) — the same paged cache the decode kernel reads.
//
// GB300 design (one CTA per 128 query rows of one query head, 1 CTA per SM):
//   warp 0, one thread : TMA producer — Q once (128 rows x 128 dims), then per 128-key tile
//                        the 8 physical blocks of K and of V (16-row boxes gathered by block
//                        id), double buffered.
//   warp 1             : owns 512 TMEM columns; one thread issues tcgen05.mma —
//                        S_j = Q K_j^T (M = N = 128, K = 128, both operands K-major in smem)
//                        into one of two TMEM S buffers, and O += P_{j-1} V_{j-1} (P K-major,
//                        V MN-major) into the TMEM O accumulator, so S_j overlaps softmax_{j-1}.
//   warps 4..7         : softmax, one query row per thread (TMEM lane = row): causal mask,
//                        online softmax in base 2, P (bf16/f16) written to shared memory in
//                        the 128-byte-swizzled K-major layout the MMA reads.  The running max
//                        used for the exponents is only moved (and O rescaled in TMEM) when
//                        the row max grows by more than 2^8, so most tiles skip the rescale;
//                        the final division by the same-base sum keeps the result exact.
// Every wait is bounded; a timeout sets PKV_DEVERR_TIMEOUT and the CTA drains and exits.
#include "pkv_device.cuh"
#include "pkv_host.h"

namespace pkv {
namespace {

constexpr int kBS = 16;
constexpr int kD = 128;
constexpr int kTile = 128;                    // query rows per CTA and keys per iteration
constexpr int kThreads = 256;
constexpr uint32_t kTmemCols = 512;           // S0 | S1 | O (128 columns each) rounded up
constexpr int kHalfBytes = kTile * 128;       // [128 rows][64 elements] of 2 bytes = 16 KB
constexpr int kTileBytes = 2 * kHalfBytes;    // one 128 x 128 operand = 32 KB
constexpr int kSmemBytes = 1024 + 6 * kTileBytes;   // Q, K[2], V[2], P
constexpr float kRescaleThreshold = 8.f;      // log2 units

struct PrefillParams {
  void* out;
  const int32_t* cu_q_lens;
  const int32_t* q_start_pos;
  const int32_t* block_tables;
  int max_blocks;
  int num_blocks;
  int num_heads;
  int num_kv_heads;
  float scale_log2;
  unsigned* err;
};

template <bool kBF16>
__device__ __forceinline__ uint32_t pack_out(float a, float b) {
  return pack2<kBF16>(a, b);
}

template <bool kBF16>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_chunk_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                         const __grid_constant__ CUtensorMap tmv, const PrefillParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar_q, bar_kv_full[2], bar_kv_empty[2], bar_s_full[2], bar_p_full, bar_pv_done;
  __shared__ uint32_t tmem_base_sh;

  const int qt = blockIdx.x, hq = blockIdx.y, c = blockIdx.z;
  const int q0 = p.cu_q_lens[c];
  const int qlen = p.cu_q_lens[c + 1] - q0;
  const int r0 = qt * kTile;
  if (qlen <= 0 || r0 >= qlen) return;                       // no rows for this CTA
  const int start = p.q_start_pos[c];
  const int ctx = start + qlen;                              // keys 0 .. ctx-1 exist
  if (start < 0 || ctx > p.max_blocks * kBS) {
    if (threadIdx.x == 0) set_error(p.err, PKV_DEVERR_CHUNK);
    return;
  }
  const int row_hi = min(qlen, r0 + kTile);
  const int kmax = start + row_hi;                           // keys needed: 0 .. kmax-1
  const int nt = (kmax + kTile - 1) / kTile;
  const int G = p.num_heads / p.num_kv_heads;
  const int h = hq / G;
  const int nb = (ctx + kBS - 1) / kBS;
  const int32_t* table = p.block_tables + int64_t(c) * p.max_blocks;

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sK = smem + kTileBytes;                           // two stages
  uint8_t* sV = smem + 3 * kTileBytes;                       // two stages
  uint8_t* sP = smem + 5 * kTileBytes;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    prefetch_tensormap(&tmq);
    prefetch_tensormap(&tmk);
    prefetch_tensormap(&tmv);
    mbar_init(&bar_q, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar_kv_full[i], 1);
      mbar_init(&bar_kv_empty[i], 1);
      mbar_init(&bar_s_full[i], 1);
    }
    mbar_init(&bar_p_full, 128);
    mbar_init(&bar_pv_done, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  const uint32_t tS0 = tmem, tS1 = tmem + 128, tO = tmem + 256;

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer ----------------
    const uint64_t pol_q = l2_policy_evict_first();
    const uint64_t pol_kv = l2_policy_evict_last();          // re-read by the other query heads
    mbar_arrive_expect_tx(&bar_q, kTileBytes);
    tma_load_3d(sQ, &tmq, &bar_q, 0, hq, q0 + r0, pol_q);
    tma_load_3d(sQ + kHalfBytes, &tmq, &bar_q, 64, hq, q0 + r0, pol_q);
    int issued = 0;
    for (int j = 0; j < nt; ++j) {
      const int st = j & 1;
      if (j >= 2 && !mbar_wait(&bar_kv_empty[st], uint32_t((j - 2) >> 1) & 1u)) {
        set_error(p.err, PKV_DEVERR_TIMEOUT);
        break;
      }
      mbar_arrive_expect_tx(&bar_kv_full[st], 2 * kTileBytes);
      for (int b = 0; b < kTile / kBS; ++b) {
        const int lb = j * (kTile / kBS) + b;
        int pb = 0;                                          // blocks past the sequence: any valid
        if (lb < nb) {                                       // block; their rows are masked / zeroed
          pb = table[lb];
          if (pb < 0 || pb >= p.num_blocks) {
            set_error(p.err, PKV_DEVERR_BLOCK_ID);
            pb = 0;
          }
        }
        const int y = (pb * p.num_kv_heads + h) * kBS;
        for (int hf = 0; hf < 2; ++hf) {
          tma_load_2d(sK + st * kTileBytes + hf * kHalfBytes + b * 2048, &tmk, &bar_kv_full[st], hf * 64, y, pol_kv);
          tma_load_2d(sV + st * kTileBytes + hf * kHalfBytes + b * 2048, &tmv, &bar_kv_full[st], hf * 64, y, pol_kv);
        }
      }
      issued = j + 1;
    }
    // Drain: the last load of each stage must have landed before the CTA may exit.
    for (int j = issued - 2 < 0 ? 0 : issued - 2; j < issued; ++j) (void)mbar_wait(&bar_kv_full[j & 1], uint32_t(j >> 1) & 1u);
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer ----------------
    const uint32_t idesc_s = umma_idesc_f16(kBF16, 128, 128, false, false);
    const uint32_t idesc_o = umma_idesc_f16(kBF16, 128, 128, false, true);
    const uint32_t aQ = smem_u32(sQ), aK = smem_u32(sK), aV = smem_u32(sV), aP = smem_u32(sP);
    bool ok = mbar_wait(&bar_q, 0);
    for (int j = 0; ok && j <= nt; ++j) {
      if (j < nt) {
        const int st = j & 1;
        if (!(ok = mbar_wait(&bar_kv_full[st], uint32_t(j >> 1) & 1u))) break;
        tc_fence_after();
        const uint32_t tS = (j & 1) ? tS1 : tS0;
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint32_t koff = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
          umma_f16(tS, umma_sdesc_sw128(aQ + koff, 16, 1024), umma_sdesc_sw128(aK + st * kTileBytes + koff, 16, 1024),
                   idesc_s, kk > 0);
        }
        umma_commit(&bar_s_full[j & 1]);
      }
      if (j >= 1) {
        const int jj = j - 1, st = jj & 1;
        if (!(ok = mbar_wait(&bar_p_full, uint32_t(jj) & 1u))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) {
          const uint32_t poff = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
          umma_f16(tO, umma_sdesc_sw128(aP + poff, 16, 1024),
                   umma_sdesc_sw128(aV + st * kTileBytes + kk * 2048, kHalfBytes, 1024), idesc_o, jj > 0 || kk > 0);
        }
        umma_commit(&bar_pv_done);
        umma_commit(&bar_kv_empty[st]);
      }
    }
    if (!ok) set_error(p.err, PKV_DEVERR_TIMEOUT);
  } else if (warp >= 4) {
    // ---------------- softmax warpgroup: one query row per thread ----------------
    const int r = threadIdx.x - 128;                         // TMEM lane == row of the tile
    const uint32_t lane_off = uint32_t(32 * (warp & 3)) << 16;
    const int qrow = r0 + r;
    const int pos = start + qrow;                            // absolute position of this query
    const uint32_t aP = smem_u32(sP);
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nt; ++j) {
      if (!(ok = mbar_wait(&bar_s_full[j & 1], uint32_t(j >> 1) & 1u))) break;
      __syncwarp();
      tc_fence_after();
      float s[kTile];
#pragma unroll
      for (int cc = 0; cc < kTile / 32; ++cc) {
        float v[32];
        tmem_ld32(((j & 1) ? tS1 : tS0) + lane_off + 32 * cc, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) s[32 * cc + i] = v[i];
      }
      tmem_wait_ld();
      const int kb = j * kTile;
      const int lim = min(pos + 1, ctx) - kb;                // keys kb + i valid for i < lim
      float mt = -INFINITY;
#pragma unroll
      for (int i = 0; i < kTile; ++i) {
        s[i] = i < lim ? s[i] * p.scale_log2 : -INFINITY;
        mt = fmaxf(mt, s[i]);
      }
      // P buffer free and O up to date once the previous PV product is done.
      if (j >= 1) {
        if (!(ok = mbar_wait(&bar_pv_done, uint32_t(j - 1) & 1u))) break;
        tc_fence_after();
      }
      const bool grow = mt > m + kRescaleThreshold;          // also true for the first tile
      __syncwarp();
      if (__any_sync(0xffffffffu, grow && j >= 1)) {
        const float alpha = (grow && m != -INFINITY) ? fast_exp2(m - mt) : 1.f;
#pragma unroll
        for (int cc = 0; cc < kD / 32; ++cc) {
          float v[32];
          tmem_ld32(tO + lane_off + 32 * cc, v);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] *= alpha;
          tmem_st32(tO + lane_off + 32 * cc, v);
        }
        tmem_wait_st();
        if (grow) l *= alpha;
      }
      if (grow) m = mt;
      // The last key tile may reach past the sequence: zero those V rows so that 0 * garbage
      // cannot turn into NaN inside the PV product.
      if (kb + kTile > ctx) {
        if (!(ok = mbar_wait(&bar_kv_full[j & 1], uint32_t(j >> 1) & 1u))) break;
        if (kb + r >= ctx) {
          const uint32_t vrow = smem_u32(sV + (j & 1) * kTileBytes) + r * 128;
#pragma unroll
          for (int hf = 0; hf < 2; ++hf)
#pragma unroll
            for (int cc = 0; cc < 8; ++cc) sts128(vrow + hf * kHalfBytes + cc * 16, 0u, 0u, 0u, 0u);
        }
      }
      // P = 2^(s - m), written as the A operand (K-major, 128-byte swizzle).
      float lsum = 0.f;
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float a = fast_exp2(s[64 * hf + 8 * cc + 2 * e] - m);
            const float b = fast_exp2(s[64 * hf + 8 * cc + 2 * e + 1] - m);
            lsum += a + b;
            w[e] = pack_out<kBF16>(a, b);
          }
          sts128(aP + hf * kHalfBytes + r * 128 + ((cc ^ (r & 7)) << 4), w[0], w[1], w[2], w[3]);
        }
      }
      l += lsum;
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bar_p_full);
    }
    if (ok) ok = mbar_wait(&bar_pv_done, uint32_t(nt - 1) & 1u);
    __syncwarp();
    if (ok) {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const bool live = qrow < qlen;
      uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.out) +
                                            ((int64_t(q0) + qrow) * p.num_heads + hq) * (kD * 2));
#pragma unroll
      for (int cc = 0; cc < kD / 32; ++cc) {
        float v[32];
        tmem_ld32(tO + lane_off + 32 * cc, v);
        tmem_wait_ld();
        if (live) {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4)
            dst[cc * 4 + q4] = make_uint4(pack_out<kBF16>(v[8 * q4] * inv, v[8 * q4 + 1] * inv),
                                          pack_out<kBF16>(v[8 * q4 + 2] * inv, v[8 * q4 + 3] * inv),
                                          pack_out<kBF16>(v[8 * q4 + 4] * inv, v[8 * q4 + 5] * inv),
                                          pack_out<kBF16>(v[8 * q4 + 6] * inv, v[8 * q4 + 7] * inv));
        }
      }
    } else if (threadIdx.x == 128) {
      set_error(p.err, PKV_DEVERR_TIMEOUT);
    }
    tc_fence_before();
  }
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace
}  // namespace pkv

extern "C" pkv_status pkv_paged_prefill_chunk(void* out, const void* q, pkv_dtype q_dtype, const int32_t* cu_q_lens,
                                              const int32_t* q_start_pos, int num_chunks, int total_q,
                                              int max_q_len, int num_heads, const void* k_cache,
                                              const void* v_cache, const pkv_cache_desc* cache,
                                              const int32_t* block_tables, int max_blocks_per_seq, float scale,
                                              pkv_stream_t stream) {
  using namespace pkv;
  pkv_status st = check_cache_desc(cache);
  if (st != PKV_OK) return st;
  if (num_chunks < 0 || total_q < 0 || max_q_len < 0 || num_heads <= 0 || max_blocks_per_seq < 0)
    return PKV_ERR_INVALID_ARG;
  if (num_chunks == 0 || total_q == 0 || max_q_len == 0) return PKV_OK;
  if (!out || !q || !cu_q_lens || !q_start_pos || !k_cache || !v_cache || !block_tables) return PKV_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) ||
      (reinterpret_cast<uintptr_t>(cu_q_lens) & 3u) || (reinterpret_cast<uintptr_t>(q_start_pos) & 3u) ||
      (reinterpret_cast<uintptr_t>(block_tables) & 3u))
    return PKV_ERR_INVALID_ARG;
  if (num_heads % cache->num_kv_heads || max_blocks_per_seq == 0) return PKV_ERR_INVALID_ARG;
  if (q_dtype != PKV_F16 && q_dtype != PKV_BF16) return PKV_ERR_INVALID_ARG;
  if (cache->kv_dtype != q_dtype || cache->head_dim != kD || cache->block_size != kBS) return PKV_ERR_UNSUPPORTED;
  if (num_chunks > 65535 || num_heads > 65535) return PKV_ERR_UNSUPPORTED;
  if (int64_t(cache->num_blocks) * cache->num_kv_heads * kBS >= (int64_t(1) << 31)) return PKV_ERR_UNSUPPORTED;
  unsigned* err = error_word_ptr();
  if (!err) return PKV_ERR_CUDA;

  CUtensorMap tq, tk, tv;
  const uint64_t rows = uint64_t(cache->num_blocks) * cache->num_kv_heads * kBS;
  if (!encode_tmap_3d(&tq, CU_TENSOR_MAP_DATA_TYPE_UINT16, q, kD, uint64_t(num_heads), uint64_t(total_q), kD * 2,
                      uint64_t(num_heads) * kD * 2, 64, 1, kTile, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tmap_2d(&tk, CU_TENSOR_MAP_DATA_TYPE_UINT16, k_cache, kD, rows, kD * 2, 64, kBS,
                      CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tmap_2d(&tv, CU_TENSOR_MAP_DATA_TYPE_UINT16, v_cache, kD, rows, kD * 2, 64, kBS,
                      CU_TENSOR_MAP_SWIZZLE_128B))
    return PKV_ERR_CUDA;

  PrefillParams prm;
  prm.out = out;
  prm.cu_q_lens = cu_q_lens;
  prm.q_start_pos = q_start_pos;
  prm.block_tables = block_tables;
  prm.max_blocks = max_blocks_per_seq;
  prm.num_blocks = cache->num_blocks;
  prm.num_heads = num_heads;
  prm.num_kv_heads = cache->num_kv_heads;
  prm.scale_log2 = scale * 1.4426950408889634f;
  prm.err = err;

  auto kern = q_dtype == PKV_BF16 ? prefill_chunk_kernel<true> : prefill_chunk_kernel<false>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) != cudaSuccess)
    return PKV_ERR_CUDA;
  dim3 grid((max_q_len + kTile - 1) / kTile, num_heads, num_chunks);
  kern<<<grid, kThreads, kSmemBytes, reinterpret_cast<cudaStream_t>(stream)>>>(tq, tk, tv, prm);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}
