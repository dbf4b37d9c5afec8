// paged_prefill_chunk: causal attention of a prefill chunk over its paged history.
//
// Method ("Lecture 33 — KV Cache management" §4.2): a long prompt is cut into chunks; a
// chunk's tokens attend, with a causal mask, the KV of the chunks already cached plus the
// chunk itself.  Query row r of a chunk that starts at position q_start sits at position
// p = q_start + r and attends keys 0..p of its sequence, read through the block table
// (§2.2–§2.3) — the same paged cache the decode kernel reads.
//
// GB300 design (one CTA per 128 query rows of one query head, 1 CTA per SM):
//   warp 0             : TMA producer — Q once (128 rows x 128 dims), then per 128-key tile
//                        the 8 physical 16-row blocks of K and of V, gathered by block id
//                        (the block table is read 32 entries at a time, lane-parallel, one
//                        window ahead).  K lands as [64-dim half][block][16 rows] (two 2-D
//                        boxes per block), so its 8-row groups are evenly spaced and one
//                        N = 128 MMA covers the tile; V lands as [block][half][16 rows] (one
//                        3-D box per block).  K and V (3 stages each) run ahead, each stage
//                        refilled once every CTA of the cluster has released it.
//   warp 1             : owns 512 TMEM columns; one thread issues tcgen05.mma —
//                        S_j = Q K_j^T (M = N = 128, K = 128, both operands K-major in smem,
//                        column n of S = key n of the tile) into one of three TMEM S buffers, and
//                        O += P_j V_j into the TMEM O accumulator, with P read from TMEM (it
//                        overwrites S_j in place) and V from shared memory as an MN-major
//                        operand.  S of later tiles overlaps the softmax of earlier ones, and
//                        the softmax never waits for a PV product unless it must rescale O.
//   warps 2..9         : softmax, two warpgroups; each thread owns one query row (TMEM lane)
//                        and one half of its 128 columns, the halves swap only the tile's row
//                        max.  Causal mask on diagonal tiles, online softmax in base 2
//                        (2^(s*scale*log2e - m): one FFMA and one ex2 per score), P (bf16/f16)
//                        stored to TMEM over the tile's S.  The running max used for the
//                        exponents is only moved (and O rescaled in TMEM) when the row max
//                        grows by more than 2^8, so most tiles skip the rescale; the final
//                        division by the same-base sum keeps the result exact.
// Every wait is bounded; a timeout sets PKV_DEVERR_TIMEOUT and the CTA drains and exits.
#include "pkv_device.cuh"
#include "pkv_host.h"

namespace pkv {
namespace {

constexpr int kBS = 16;        // rows per TMA box: a 16-token block, or half of a 32-token one
constexpr int kD = 128;
constexpr int kTile = 128;                    // query rows per CTA and keys per iteration
constexpr int kThreads = 320;                 // warp 0 TMA, warp 1 MMA, warps 2..9 softmax
constexpr uint32_t kTmemCols = 512;           // S0 | S1 | S2 | O, 128 columns each
constexpr int kHalfBytes = kTile * 128;       // [128 rows][64 elements] of 2 bytes = 16 KB
constexpr int kTileBytes = 2 * kHalfBytes;    // one 128 x 128 operand = 32 KB
// A V tile holds 8 blocks of 4 KB: block b at 4 KB * b = [dims 0..63: 16 rows x 128 B]
// [dims 64..127: 16 rows x 128 B], each half 128-byte swizzled (one 3-D TMA box per block).
// A K tile holds the same bytes as [dims 0..63: block 0..7 x 16 rows][dims 64..127: ...]
// (two 2-D boxes of 2 KB per block).
constexpr int kBlockBytes = kBS * kD * 2;
constexpr int kKStages = 3;                   // K tiles in flight (released when their S product is done)
constexpr int kVStages = 3;                   // V tiles in flight (released when their PV product is done)
constexpr int kSBufs = 3;                     // TMEM S/P buffers (128 columns each; O takes the 4th)
// Q, K stages, V stages: 224 KB, which with the static barriers fills the 227 KB a CTA may
// use, so the dynamic region carries no alignment slack; the kernel checks that it starts on
// a 1 KB boundary (required by the 128-byte swizzle) and reports an error otherwise.
constexpr int kSmemBytes = (1 + kKStages + kVStages) * kTileBytes;
constexpr float kRescaleThreshold = 8.f;      // log2 units
// A cluster is kCluster consecutive query tiles of one head and chunk.  They read the same K/V
// tiles, so each CTA fetches a quarter of every tile's boxes and multicasts them to all: the
// per-SM TMA work per tile drops by kCluster (one SM's TMA unit, not HBM or L2, bounds a
// CTA that fetches all sixteen 4 KB boxes of a K+V tile itself).
constexpr int kCluster = 4;
constexpr uint16_t kClusterMask = (1u << kCluster) - 1;

struct PrefillParams {
  void* out;
  const int32_t* cu_q_lens;
  const int32_t* q_start_pos;
  const int32_t* block_tables;
  int max_blocks;
  int num_blocks;
  int block_size;         // tokens per pool block: 16 or 32
  int tile_shift;         // log2(block_size / 16)
  int num_heads;
  int num_kv_heads;
  float scale_log2;
  unsigned* err;
};

template <bool kBF16>
__device__ __forceinline__ uint32_t pack_out(float a, float b) {
  return pack2<kBF16>(a, b);
}

// 16 consecutive 32-bit columns of this thread's TMEM lane, from raw words.
__device__ __forceinline__ void tmem_st16u(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// Three-input maximum (one instruction on this architecture).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Two fp32 values in one 64-bit register pair, for the packed fp32 instructions.
__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float lo_f32(uint64_t v) { return __uint_as_float(uint32_t(v)); }
__device__ __forceinline__ float hi_f32(uint64_t v) { return __uint_as_float(uint32_t(v >> 32)); }
// a * b + c and a + b on both halves, rounded to nearest (the same results as fmaf / +).
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

template <bool kBF16>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_chunk_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                         const __grid_constant__ CUtensorMap tmv, const PrefillParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar_q, bar_k_full[kKStages], bar_k_empty[kKStages], bar_v_full[kVStages],
      bar_v_empty[kVStages], bar_s_full[kSBufs], bar_p_full[kSBufs], bar_pv_done[kSBufs];
  __shared__ uint32_t tmem_base_sh;
  __shared__ float row_xchg[2][2][kTile];                    // [use parity][half][row]: values the softmax halves swap
  __shared__ __align__(8) uint64_t bar_xchg[2];              // 256 arrivals: both halves have written

  const int qt = blockIdx.x, hq = blockIdx.y, c = blockIdx.z;
  const int q0 = p.cu_q_lens[c];
  const int qlen = p.cu_q_lens[c + 1] - q0;
  const int r0 = qt * kTile;
  // Decisions before the first cluster barrier must be the same for the whole cluster.
  const int r0_cl = (qt & ~(kCluster - 1)) * kTile;           // first row of the cluster
  if (qlen <= 0 || r0_cl >= qlen) return;                    // no rows for the whole cluster
  const int start = p.q_start_pos[c];
  const int ctx = start + qlen;                              // keys 0 .. ctx-1 exist
  if (start < 0 || ctx > p.max_blocks * p.block_size) {
    if (threadIdx.x == 0) set_error(p.err, PKV_DEVERR_CHUNK);
    return;
  }
  // Every CTA of the cluster walks the keys the cluster needs; a CTA whose rows end earlier
  // finds the extra keys in its rows' future, where the causal mask zeroes them.  A CTA with
  // no rows at all still takes part (its outputs are not stored).
  const int kmax = start + min(qlen, r0_cl + kCluster * kTile);
  const int nt = (kmax + kTile - 1) / kTile;
  const uint32_t crank = cluster_ctarank();
  const int G = p.num_heads / p.num_kv_heads;
  const int h = hq / G;
  const int nb = (ctx + kBS - 1) / kBS;
  const int32_t* table = p.block_tables + int64_t(c) * p.max_blocks;

  uint8_t* smem = smem_raw;
  if (smem_u32(smem) & 1023u) {                              // see kSmemBytes
    if (threadIdx.x == 0) set_error(p.err, PKV_DEVERR_CHUNK);
    return;
  }
  uint8_t* sQ = smem;
  uint8_t* sK = smem + kTileBytes;                           // kKStages stages
  uint8_t* sV = smem + (1 + kKStages) * kTileBytes;          // kVStages stages
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    prefetch_tensormap(&tmq);
    prefetch_tensormap(&tmk);
    prefetch_tensormap(&tmv);
    mbar_init(&bar_q, 1);
    // A stage is free again once every CTA of the cluster has released it.
    for (int i = 0; i < kKStages; ++i) {
      mbar_init(&bar_k_full[i], 1);
      mbar_init(&bar_k_empty[i], kCluster);
    }
    for (int i = 0; i < kVStages; ++i) {
      mbar_init(&bar_v_full[i], 1);
      mbar_init(&bar_v_empty[i], kCluster);
    }
    // The softmax warps signal P and the row-value swaps once per warp (lane 0, after the
    // warp's own accesses): 8 arrivals a phase.
    for (int i = 0; i < kSBufs; ++i) {
      mbar_init(&bar_s_full[i], 1);
      mbar_init(&bar_p_full[i], 8);
    }
    mbar_init(&bar_xchg[0], 8);
    mbar_init(&bar_xchg[1], 8);
    // PV_t's completion arrives on bar_pv_done[t % kSBufs].  A waiter for PV_t is always at most
    // one phase behind that barrier (PV_{t+kSBufs} needs P_{t+kSBufs}, which the softmax has not
    // produced yet), so waiting by phase parity is exact.  One barrier for every PV would not
    // be: the softmax checks it only now and then, and the barrier can run two phases ahead.
    for (int i = 0; i < kSBufs; ++i) mbar_init(&bar_pv_done[i], 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();                                            // every peer's barriers are initialised
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  const uint32_t tO = tmem + 128 * kSBufs;
  auto tS = [&](int j) -> uint32_t { return tmem + 128 * uint32_t(j % kSBufs); };   // S_j, then P_j

  if (warp == 0) {
    // ---------------- TMA producer (the whole warp; lane 0 issues) ----------------
    const uint64_t pol_q = l2_policy_evict_first();
    const uint64_t pol_kv = l2_policy_evict_last();          // re-read by the other query heads
    if (lane == 0) {
      mbar_arrive_expect_tx(&bar_q, kTileBytes);
      tma_load_3d(sQ, &tmq, &bar_q, 0, hq, q0 + r0, pol_q);
      tma_load_3d(sQ + kHalfBytes, &tmq, &bar_q, 64, hq, q0 + r0, pol_q);
    }
    // Pool rows of the sequence's 16-row units, 32 per window (4 tiles): lane i holds unit
    // 32 * w + i, which is block unit >> tile_shift at row offset 16 * (unit & mask).  Units
    // past the sequence map to block 0 (their rows are masked / zeroed).
    auto load_window = [&](int w) -> int {
      const int lb = 32 * w + lane;
      int pb = 0;
      if (lb < nb) {
        pb = table[lb >> p.tile_shift];
        if (pb < 0 || pb >= p.num_blocks) {
          set_error(p.err, PKV_DEVERR_BLOCK_ID);
          pb = 0;
        }
      }
      return (pb * p.num_kv_heads + h) * p.block_size + (lb & ((1 << p.tile_shift) - 1)) * kBS;
    };
    struct Window {
      int cur, nxt, w;
    };
    // The window holding tile j (one ahead is always loaded, so the loads overlap the TMAs).
    auto seek = [&](Window& win, int j) {
      while (j / 4 > win.w) {
        win.cur = win.nxt;
        ++win.w;
        win.nxt = load_window(win.w + 1);
      }
    };
    Window wk{load_window(0), load_window(1), 0};
    Window wv = wk;
    // The 8 lanes that hold the tile's block rows issue its boxes that fall to this CTA
    // (box % kCluster == rank), multicast to the whole cluster, in the same instruction.
    // Each CTA's own full barrier expects the whole tile, most of it sent by its peers.
    auto issue_k = [&](uint8_t* dst, uint64_t* bar, int j) {
      seek(wk, j);
      const int first = (8 * j) % 32;
      if (lane == first) mbar_arrive_expect_tx(bar, kTileBytes);
      __syncwarp();
      const int blk = lane - first;
      if (blk >= 0 && blk < kTile / kBS) {
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          if (uint32_t((2 * blk + hf) % kCluster) == crank)
            tma_load_3d_mc(dst + hf * kHalfBytes + blk * (kBlockBytes / 2), &tmk, bar, 0, wk.cur, hf, kClusterMask,
                           pol_kv);
        }
      }
    };
    auto issue_v = [&](uint8_t* dst, uint64_t* bar, int j) {
      seek(wv, j);
      const int first = (8 * j) % 32;
      if (lane == first) mbar_arrive_expect_tx(bar, kTileBytes);
      __syncwarp();
      const int blk = lane - first;
      if (blk >= 0 && blk < kTile / kBS && uint32_t(blk % kCluster) == crank)
        tma_load_3d_mc(dst + blk * kBlockBytes, &tmv, bar, 0, wv.cur, 0, kClusterMask, pol_kv);
    };
    // K runs ahead of V; each is issued as soon as its stage has been released.  Lane 0
    // polls the barriers and broadcasts, so the warp stays converged.
    auto ready = [&](uint64_t* bar, uint32_t parity) -> bool {
      uint32_t r = 0;
      if (lane == 0) r = mbar_test(bar, parity) ? 1u : 0u;
      return __shfl_sync(0xffffffffu, r, 0) != 0;
    };
    int kj = 0, vj = 0;
    uint64_t t0 = 0;
    bool ok = true;
    while (ok && (kj < nt || vj < nt)) {
      bool progress = false;
      if (kj < nt && (kj < kKStages || ready(&bar_k_empty[kj % kKStages], uint32_t((kj - kKStages) / kKStages) & 1u))) {
        issue_k(sK + (kj % kKStages) * kTileBytes, &bar_k_full[kj % kKStages], kj);
        ++kj;
        progress = true;
      }
      if (vj < kj && (vj < kVStages || ready(&bar_v_empty[vj % kVStages], uint32_t((vj - kVStages) / kVStages) & 1u))) {
        issue_v(sV + (vj % kVStages) * kTileBytes, &bar_v_full[vj % kVStages], vj);
        ++vj;
        progress = true;
      }
      // Lane 0 keeps the clock, so every lane takes the same decision.  Idle polls back off
      // so they do not take issue slots from the softmax warps on the same SM sub-partition.
      if (!progress) __nanosleep(100);
      uint32_t give_up = 0;
      if (lane == 0) {
        if (progress) {
          t0 = 0;
        } else if (t0 == 0) {
          t0 = global_timer_ns();
        } else if (global_timer_ns() - t0 > kWaitLimitNs) {
          set_error(p.err, PKV_DEVERR_TIMEOUT);
          give_up = 1;
        }
      }
      ok = __shfl_sync(0xffffffffu, give_up, 0) == 0;
    }
    // Drain: the last load of each stage must have landed, and every peer's release of the
    // last tiles must have reached this CTA's barriers, before the CTA may leave the cluster.
    if (lane == 0) {
      for (int j = kj - kKStages < 0 ? 0 : kj - kKStages; j < kj; ++j)
        (void)mbar_wait(&bar_k_full[j % kKStages], uint32_t(j / kKStages) & 1u);
      for (int j = vj - kVStages < 0 ? 0 : vj - kVStages; j < vj; ++j)
        (void)mbar_wait(&bar_v_full[j % kVStages], uint32_t(j / kVStages) & 1u);
      for (int j = kj - kKStages < 0 ? 0 : kj - kKStages; j < kj; ++j)
        (void)mbar_wait(&bar_k_empty[j % kKStages], uint32_t(j / kKStages) & 1u);
      for (int j = vj - kVStages < 0 ? 0 : vj - kVStages; j < vj; ++j)
        (void)mbar_wait(&bar_v_empty[j % kVStages], uint32_t(j / kVStages) & 1u);
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer ----------------
    // S_j needs K_j and a free S buffer (PV_{j-2}, which reads P_{j-2} from that buffer,
    // issued: tcgen05 ops of one thread execute in order); PV_j needs P_j and V_j.  Whichever
    // is ready is issued first.
    const uint32_t idesc_s = umma_idesc_f16(kBF16, 128, 128, false, false);
    const uint32_t idesc_o = umma_idesc_f16(kBF16, 128, 128, false, true);
    const uint32_t aQ = smem_u32(sQ), aK = smem_u32(sK), aV = smem_u32(sV);
    bool ok = mbar_wait(&bar_q, 0);
    int js = 0, jp = 0;
    uint64_t t0 = 0;
    while (ok && jp < nt) {
      bool progress = false;
      if (js < nt && js - jp < kSBufs && mbar_test(&bar_k_full[js % kKStages], uint32_t(js / kKStages) & 1u)) {
        tc_fence_after();
        const int st = js % kKStages;
        const uint32_t tSj = tS(js);
        // k-step kk: dims 16kk .. 16kk + 15 of Q and K, both stored as [64-dim half][rows]
        // with 8-row groups 1 KB apart, so S column n is key n of the tile.
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
          umma_f16(tSj, umma_sdesc_sw128(aQ + off, 16, 1024), umma_sdesc_sw128(aK + st * kTileBytes + off, 16, 1024),
                   idesc_s, kk > 0);
        }
        umma_commit(&bar_s_full[js % kSBufs]);
        umma_commit_mc(&bar_k_empty[st], kClusterMask);     // released in every CTA of the cluster
        ++js;
        progress = true;
      }
      if (jp < js && mbar_test(&bar_p_full[jp % kSBufs], uint32_t(jp / kSBufs) & 1u) &&
          mbar_test(&bar_v_full[jp % kVStages], uint32_t(jp / kVStages) & 1u)) {
        tc_fence_after();
        const int st = jp % kVStages;
        // P_jp sits in the first 64 columns of its S buffer, two 16-bit values per column.
        const uint32_t tP = tS(jp);
        // k-step kk covers P columns 16kk .. 16kk + 15 = keys of block kk: its two 8-row
        // groups sit 1 KB apart, its two 64-dim halves 2 KB apart.
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) {
          umma_f16_ts(tO, tP + 8 * kk, umma_sdesc_sw128(aV + st * kTileBytes + kk * kBlockBytes, kBlockBytes / 2, 1024),
                      idesc_o, jp > 0 || kk > 0);
        }
        umma_commit(&bar_pv_done[jp % kSBufs]);
        umma_commit_mc(&bar_v_empty[st], kClusterMask);
        ++jp;
        progress = true;
      }
      if (progress) {
        t0 = 0;
      } else {
        __nanosleep(50);
        if (t0 == 0) {
          t0 = global_timer_ns();
        } else if (global_timer_ns() - t0 > kWaitLimitNs) {
          ok = false;
        }
      }
    }
    if (!ok) set_error(p.err, PKV_DEVERR_TIMEOUT);
  } else if (warp >= 2) {
    // ---------------- softmax: two warpgroups, one query row per thread in each ----------
    // Warp w reaches TMEM lanes 32 * (w % 4) .. + 31, so warps 2..5 and 6..9 each cover all
    // 128 rows; warpgroup `half` owns columns 64 * half .. + 63 of S, O and P.
    const int half = (warp - 2) >> 2;
    const int r = 32 * (warp & 3) + lane;                    // TMEM lane == row of the tile
    const uint32_t lane_off = uint32_t(32 * (warp & 3)) << 16;
    const uint32_t col0 = 64 * half;
    const int qrow = r0 + r;
    const int pos = start + qrow;                            // absolute position of this query
    const float sl = p.scale_log2;                           // > 0, so max(s) * sl = max(s * sl)
    // Swap one float per row with the other half through shared memory; the k-th swap uses
    // buffer and barrier k % 2 (bounded wait; the barrier's arrive/wait order the accesses).
    int n_swaps = 0;
    auto swap_halves = [&](float mine, float& theirs) -> bool {
      const int b = n_swaps & 1;
      row_xchg[b][half][r] = mine;
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_xchg[b]);
      const bool done = mbar_wait(&bar_xchg[b], uint32_t(n_swaps >> 1) & 1u);
      theirs = row_xchg[b][half ^ 1][r];
      ++n_swaps;
      return done;
    };
    float m = -INFINITY, l = 0.f;                            // m in scaled log2 units
    bool ok = true;
    for (int j = 0; j < nt; ++j) {
      if (!(ok = mbar_wait(&bar_s_full[j % kSBufs], uint32_t(j / kSBufs) & 1u))) break;
      __syncwarp();
      tc_fence_after();
      float s[64];
      {
        float v[32];
        const uint32_t tSj = tS(j) + lane_off + col0;
        tmem_ld32(tSj, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) s[i] = v[i];
        tmem_ld32(tSj + 32, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) s[32 + i] = v[i];
      }
      tmem_wait_ld();
      // Column i of this half holds key kb + 64 * half + i.
      const int lim = min(pos + 1, ctx) - (j * kTile + 64 * half);  // valid iff i < lim
      float mraw = -INFINITY;
      if (lim >= 64) {                                       // all 64 columns of this half valid
#pragma unroll
        for (int i = 0; i < 64; ++i) mraw = fmaxf(mraw, s[i]);
      } else {
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          s[i] = i < lim ? s[i] : -INFINITY;
          mraw = fmaxf(mraw, s[i]);
        }
      }
      float other;
      if (!(ok = swap_halves(mraw, other))) break;
      const float mt = fmaxf(mraw, other) * sl;              // row max of the tile
      const bool grow = mt > m + kRescaleThreshold;          // also true for the first tile
      if (__any_sync(0xffffffffu, grow && j >= 1)) {
        // O must be up to date (the previous PV product done) before it is rescaled.
        if (!(ok = mbar_wait(&bar_pv_done[(j - 1) % kSBufs], uint32_t((j - 1) / kSBufs) & 1u))) break;
        __syncwarp();
        tc_fence_after();
        const float alpha = (grow && m != -INFINITY) ? fast_exp2(m - mt) : 1.f;
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          float v[32];
          tmem_ld32(tO + lane_off + col0 + 32 * cc, v);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] *= alpha;
          tmem_st32(tO + lane_off + col0 + 32 * cc, v);
        }
        tmem_wait_st();
        if (grow) l *= alpha;
      }
      if (grow) m = mt;
      // The last key tile may reach past the sequence: zero those V rows so that 0 * garbage
      // cannot turn into NaN inside the PV product.
      const int kb = j * kTile;
      if (kb + kTile > ctx) {
        if (!(ok = mbar_wait(&bar_v_full[j % kVStages], uint32_t(j / kVStages) & 1u))) break;
        if (kb + r >= ctx) {
          const uint32_t vrow = smem_u32(sV + (j % kVStages) * kTileBytes) + (r / kBS) * kBlockBytes +
                                half * (kBlockBytes / 2) + (r % kBS) * 128;
#pragma unroll
          for (int cc = 0; cc < 8; ++cc) sts128(vrow + cc * 16, 0u, 0u, 0u, 0u);
        }
      }
      // P = 2^(s * sl - m) as 16-bit pairs, written over this tile's S in TMEM: keys
      // 64 * half .. + 63 go to columns 32 * half .. + 31 (the S values are in registers).
      float lsum = 0.f;
      uint32_t w[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const float a = fast_exp2(fmaf(s[2 * e], sl, -m));
        const float b = fast_exp2(fmaf(s[2 * e + 1], sl, -m));
        lsum += a + b;
        w[e] = pack_out<kBF16>(a, b);
      }
      tmem_st32u(tS(j) + lane_off + 32 * half, w);
      tmem_wait_st();
      l += lsum;
      if (kb + kTile > ctx) fence_proxy_async_smem();        // the zeroed V rows, to the tensor cores
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_p_full[j % kSBufs]);
    }
    if (ok) ok = mbar_wait(&bar_pv_done[(nt - 1) % kSBufs], uint32_t((nt - 1) / kSBufs) & 1u);
    // Row sum = the two halves' partial sums (both used the same m).
    if (ok) {
      float other;
      ok = swap_halves(l, other);
      l += other;
    }
    __syncwarp();
    if (ok) {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const bool live = qrow < qlen;
      uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.out) +
                                            ((int64_t(q0) + qrow) * p.num_heads + hq) * (kD * 2) + col0 * 2);
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        float v[32];
        tmem_ld32(tO + lane_off + col0 + 32 * cc, v);
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
    } else if (r == 0 && half == 0) {
      set_error(p.err, PKV_DEVERR_TIMEOUT);
    }
    tc_fence_before();
  }
  __syncthreads();
  cluster_sync();                                            // no peer sends to this CTA any more
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}


// ---------------------------------------------------------------------------------------
// Two query heads per CTA, the key range split in two, in clusters of four CTAs.
//
// The query heads of a GQA group read the same K/V.  A CTA here takes two heads of one kv head
// (128 rows each), so every K/V tile it receives feeds 256 query rows.  A cluster is two
// adjacent q-tiles x two halves of their key range: the two CTAs of a half read the same keys,
// each issues half of every tile's TMA boxes and multicasts them to both; the two halves of a
// q-tile merge their partial results at the end.
//   warp 0     : TMA producer: Q of both heads once, then its half of the boxes of K and V
//                of the half's key tiles (2 stages each), multicast to the q-tile partner.  A
//                stage is refilled once both CTAs' tensor-core commits have released it.
//   warp 1     : TMEM owner (512 columns: S_A | S_B | O_A | O_B) and MMA issuer, in the
//                fixed order S_A(0) S_B(0) | PV_A(t) S_A(t+1) PV_B(t) S_B(t+1) | ... so that
//                one head's softmax overlaps the other head's products.
//   warps 2-5  : softmax of head A, warps 6-9: head B; one query row per thread.  The row's
//                128 scores are read from TMEM once; the max uses 3-input max, P = 2^(s*c - m)
//                uses packed fp32x2 multiply-add and add; P goes over S in TMEM; O is rescaled
//                only when the row max grows by more than 2^8.
// At the end the first-half CTA of a q-tile finishes head A and the second-half CTA head B.
// Each CTA stages the other head's unnormalised O rows and (max, sum) in its idle stages and
// sends them to its peer with bulk shared-memory copies; the receiver combines the two parts
// by log-sum-exp, stages the 16-bit rows in the idle Q area and writes them out coalesced.
// ---------------------------------------------------------------------------------------
constexpr int kPairThreads = 320;
constexpr int kPairKStages = 2;
constexpr int kPairVStages = 2;
// The merge's exchange block: [128 rows][kXStride] fp32 O, then 128 row maxima and 128 row sums.
constexpr int kXStride = kD + 4;
constexpr int kXBytes = (kTile * kXStride + 2 * kTile) * 4;
constexpr int kXAreaBytes = (kXBytes + 1023) / 1024 * 1024;
static_assert((32 * kXStride * 4) % 16 == 0 && (kTile * kXStride * 4) % 16 == 0,
              "each warp's rows, and the max and sum arrays after them, start and end on 16 bytes");
// Output rows staged as 16-bit values in the Q area, padded by 16 bytes per row.
constexpr int kOStride = kD * 2 + 16;
static_assert(kTile * kOStride <= 2 * kTileBytes, "the staged output rows fit in the Q area");
// Q_A, Q_B, 2 K and 2 V stages (192 KB); after the main loop the K/V stages and 8 KB past
// them hold the receive and staging areas of the merge (200 KB in all).
constexpr int kPairKVBytes = (kPairKStages + kPairVStages) * kTileBytes;
constexpr int kPairSmemBytes = 2 * kTileBytes + (2 * kXAreaBytes > kPairKVBytes ? 2 * kXAreaBytes : kPairKVBytes);

__device__ __forceinline__ uint32_t peer_smem_addr(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}

// Copies `bytes` (a multiple of 16) from this CTA's shared memory to a peer CTA's, completing
// on the peer's mbarrier; dst and bar are shared::cluster addresses (from mapa).
__device__ __forceinline__ void bulk_copy_to_peer(uint32_t dst, uint32_t src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "r"(src), "r"(bytes), "r"(bar)
               : "memory");
}

// Non-blocking check of a phase whose arrivals include other CTAs' (acquire at cluster scope).
__device__ __forceinline__ bool mbar_test_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// One arrival on an mbarrier of a peer CTA (a shared::cluster address from mapa), as a bare
// signal: relaxed, it orders none of this thread's memory accesses.  Every use below signals
// an event whose memory effects are ordered otherwise (a tensor-core commit that has been
// observed, a CTA barrier after the last store to the area, a completed bulk copy).
__device__ __forceinline__ void remote_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

template <bool kBF16>
__global__ void __launch_bounds__(kPairThreads, 1)
    prefill_pair_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                        const __grid_constant__ CUtensorMap tmv, const PrefillParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar_q, bar_k_full[kPairKStages], bar_k_empty[kPairKStages],
      bar_v_full[kPairVStages], bar_v_empty[kPairVStages], bar_s_full[2], bar_p_full[2], bar_pv_done[2], bar_x,
      bar_ready, bar_done;
  __shared__ uint32_t tmem_base_sh;

  const int qt = blockIdx.x, slot = blockIdx.y, c = blockIdx.z >> 1;
  const uint32_t crank = cluster_ctarank();                 // (q-tile of the pair) + 2 * (key half)
  const uint32_t khalf = crank >> 1;
  const uint16_t mc_mask = uint16_t(3u << (2 * khalf));     // the two CTAs reading this half's keys
  // Launched as a programmatic dependent: the CTA may start while the previous kernel runs,
  // and reads nothing that kernel may write before this point.
  griddep_wait();
  const int q0 = p.cu_q_lens[c];
  const int qlen = p.cu_q_lens[c + 1] - q0;
  const int r0 = qt * kTile;
  const int r0_pair = (qt & ~1) * kTile;
  // Every decision before the first cluster barrier is the same for all CTAs of the cluster.
  if (qlen <= 0 || r0_pair >= qlen) return;
  const int start = p.q_start_pos[c];
  const int ctx = start + qlen;                              // keys 0 .. ctx-1 exist
  if (start < 0 || ctx > p.max_blocks * p.block_size) {
    if (threadIdx.x == 0) set_error(p.err, PKV_DEVERR_CHUNK);
    return;
  }
  // Both q-tiles of the pair walk the keys the later one needs (the earlier one finds the
  // extra keys in its rows' future, masked); a q-tile past the chunk still takes part.
  const int kmax = start + min(qlen, r0_pair + 2 * kTile);
  const int nt = (kmax + kTile - 1) / kTile;
  const int mid = (nt + 1) / 2;
  const int j0 = khalf ? mid : 0;                            // this CTA's key tiles j0 .. j0 + n - 1
  const int n = khalf ? nt - mid : mid;
  const int G = p.num_heads / p.num_kv_heads;
  const int spg = (G + 1) / 2;                               // head pairs (slots) per kv head
  const int h = slot / spg;
  const int hq0 = h * G + 2 * (slot % spg);
  const int hq1 = 2 * (slot % spg) + 1 < G ? hq0 + 1 : hq0;  // an odd group's last slot repeats a head
  const int nb = (ctx + kBS - 1) / kBS;
  const int32_t* table = p.block_tables + int64_t(c) * p.max_blocks;

  uint8_t* smem = smem_raw;
  if (smem_u32(smem) & 1023u) {                              // the 128-byte swizzle needs 1 KB alignment
    if (threadIdx.x == 0) set_error(p.err, PKV_DEVERR_CHUNK);
    return;
  }
  uint8_t* sQ = smem;                                        // [head][64-dim half][128 rows]
  uint8_t* sK = smem + 2 * kTileBytes;
  uint8_t* sV = smem + (2 + kPairKStages) * kTileBytes;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    prefetch_tensormap(&tmq);
    prefetch_tensormap(&tmk);
    prefetch_tensormap(&tmv);
    mbar_init(&bar_q, 1);
    // A stage is free again once both CTAs reading this half's keys have released it: each
    // CTA's tensor-core commit arrives on the stage's empty barrier in both.
    for (int i = 0; i < kPairKStages; ++i) {
      mbar_init(&bar_k_full[i], 1);
      mbar_init(&bar_k_empty[i], 2);
    }
    for (int i = 0; i < kPairVStages; ++i) {
      mbar_init(&bar_v_full[i], 1);
      mbar_init(&bar_v_empty[i], 2);
    }
    // One phase per key tile each.  A head's softmax waits on its pv_done only for the
    // product of the previous tile, and the next product needs this tile's P first, so the
    // barrier is never two phases ahead of its waiter.
    for (int x = 0; x < 2; ++x) {
      mbar_init(&bar_s_full[x], 1);
      mbar_init(&bar_p_full[x], 4);                          // one arrival per softmax warp
      mbar_init(&bar_pv_done[x], 1);
    }
    // The merge's bulk copies from the peer complete this barrier's first phase.
    mbar_init(&bar_x, 1);
    mbar_arrive_expect_tx(&bar_x, kXBytes);
    mbar_init(&bar_ready, 1);                                // the peer's receive area is free
    mbar_init(&bar_done, 1);                                 // the peer has this CTA's whole block
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();                                            // every CTA's barriers are initialised
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    const uint64_t pol_q = l2_policy_evict_first();
    const uint64_t pol_kv = l2_policy_evict_last();          // re-read by the other query heads
    if (lane == 0) {
      mbar_arrive_expect_tx(&bar_q, 2 * kTileBytes);
      tma_load_3d(sQ, &tmq, &bar_q, 0, hq0, q0 + r0, pol_q);
      tma_load_3d(sQ + kHalfBytes, &tmq, &bar_q, 64, hq0, q0 + r0, pol_q);
      tma_load_3d(sQ + kTileBytes, &tmq, &bar_q, 0, hq1, q0 + r0, pol_q);
      tma_load_3d(sQ + kTileBytes + kHalfBytes, &tmq, &bar_q, 64, hq1, q0 + r0, pol_q);
    }
    // Pool rows of the sequence's 16-row units, 32 per window (4 tiles); units past the
    // sequence map to block 0 (their rows are masked / zeroed).
    auto load_window = [&](int w) -> int {
      const int lb = 32 * w + lane;
      int pb = 0;
      if (lb < nb) {
        pb = table[lb >> p.tile_shift];
        if (pb < 0 || pb >= p.num_blocks) {
          set_error(p.err, PKV_DEVERR_BLOCK_ID);
          pb = 0;
        }
      }
      return (pb * p.num_kv_heads + h) * p.block_size + (lb & ((1 << p.tile_shift) - 1)) * kBS;
    };
    struct Window {
      int cur, nxt, w;
    };
    auto seek = [&](Window& win, int j) {
      while (j / 4 > win.w) {
        win.cur = win.nxt;
        ++win.w;
        win.nxt = load_window(win.w + 1);
      }
    };
    Window wk{load_window(j0 / 4), load_window(j0 / 4 + 1), j0 / 4};
    Window wv = wk;
    auto issue_k = [&](uint8_t* dst, uint64_t* bar, int j) {
      seek(wk, j);
      const int first = (8 * j) % 32;
      if (lane == first) mbar_arrive_expect_tx(bar, kTileBytes);
      __syncwarp();
      const int blk = lane - first;
      if (blk >= 0 && blk < kTile / kBS) {                   // this CTA's half: the 64-dim half hf
        const int hf = int(crank & 1u);
        tma_load_3d_mc(dst + hf * kHalfBytes + blk * (kBlockBytes / 2), &tmk, bar, 0, wk.cur, hf, mc_mask, pol_kv);
      }
    };
    auto issue_v = [&](uint8_t* dst, uint64_t* bar, int j) {
      seek(wv, j);
      const int first = (8 * j) % 32;
      if (lane == first) mbar_arrive_expect_tx(bar, kTileBytes);
      __syncwarp();
      const int blk = lane - first;
      if (blk >= 0 && blk < kTile / kBS && uint32_t(blk & 1) == (crank & 1u))   // every other block
        tma_load_3d_mc(dst + blk * kBlockBytes, &tmv, bar, 0, wv.cur, 0, mc_mask, pol_kv);
    };
    // The empty barriers also collect the partner CTA's releases: acquire at cluster scope.
    auto ready = [&](uint64_t* bar, uint32_t parity) -> bool {
      uint32_t r = 0;
      if (lane == 0) r = mbar_test_cluster(bar, parity) ? 1u : 0u;
      return __shfl_sync(0xffffffffu, r, 0) != 0;
    };
    int kt = 0, vt = 0;                                      // tiles issued, counted from j0
    uint64_t t0 = 0;
    bool ok = true;
    while (ok && (kt < n || vt < n)) {
      bool progress = false;
      if (kt < n && (kt < kPairKStages ||
                     ready(&bar_k_empty[kt % kPairKStages], uint32_t((kt - kPairKStages) / kPairKStages) & 1u))) {
        issue_k(sK + (kt % kPairKStages) * kTileBytes, &bar_k_full[kt % kPairKStages], j0 + kt);
        ++kt;
        progress = true;
      }
      if (vt < kt && (vt < kPairVStages ||
                      ready(&bar_v_empty[vt % kPairVStages], uint32_t((vt - kPairVStages) / kPairVStages) & 1u))) {
        issue_v(sV + (vt % kPairVStages) * kTileBytes, &bar_v_full[vt % kPairVStages], j0 + vt);
        ++vt;
        progress = true;
      }
      if (!progress) __nanosleep(100);
      uint32_t give_up = 0;
      if (lane == 0) {
        if (progress) {
          t0 = 0;
        } else if (t0 == 0) {
          t0 = global_timer_ns();
        } else if (global_timer_ns() - t0 > kWaitLimitNs) {
          set_error(p.err, PKV_DEVERR_TIMEOUT);
          give_up = 1;
        }
      }
      ok = __shfl_sync(0xffffffffu, give_up, 0) == 0;
    }
    // Drain: the last loads of each stage have landed, and the partner's releases of the last
    // tiles have reached this CTA's barriers, before the CTA may leave.
    if (lane == 0) {
      for (int t = kt - kPairKStages < 0 ? 0 : kt - kPairKStages; t < kt; ++t)
        (void)mbar_wait(&bar_k_full[t % kPairKStages], uint32_t(t / kPairKStages) & 1u);
      for (int t = vt - kPairVStages < 0 ? 0 : vt - kPairVStages; t < vt; ++t)
        (void)mbar_wait(&bar_v_full[t % kPairVStages], uint32_t(t / kPairVStages) & 1u);
      for (int t = kt - kPairKStages < 0 ? 0 : kt - kPairKStages; t < kt; ++t)
        (void)mbar_wait(&bar_k_empty[t % kPairKStages], uint32_t(t / kPairKStages) & 1u);
      for (int t = vt - kPairVStages < 0 ? 0 : vt - kPairVStages; t < vt; ++t)
        (void)mbar_wait(&bar_v_empty[t % kPairVStages], uint32_t(t / kPairVStages) & 1u);
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer ----------------
    const uint32_t idesc_s = umma_idesc_f16(kBF16, 128, 128, false, false);
    const uint32_t idesc_o = umma_idesc_f16(kBF16, 128, 128, false, true);
    const uint32_t aQ = smem_u32(sQ), aK = smem_u32(sK), aV = smem_u32(sV);
    bool ok = mbar_wait(&bar_q, 0);
    // S_x(t) = Q_x K_t^T into TMEM columns 128x .. 128x + 127.
    auto issue_s = [&](int x, int t) -> bool {
      const int st = t % kPairKStages;
      if (!mbar_wait(&bar_k_full[st], uint32_t(t / kPairKStages) & 1u)) return false;
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < kD / 16; ++kk) {
        const uint32_t off = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
        umma_f16(tmem + 128 * x, umma_sdesc_sw128(aQ + x * kTileBytes + off, 16, 1024),
                 umma_sdesc_sw128(aK + st * kTileBytes + off, 16, 1024), idesc_s, kk > 0);
      }
      umma_commit(&bar_s_full[x]);
      if (x == 1) umma_commit_mc(&bar_k_empty[st], mc_mask); // both heads have read K_t: release it in both CTAs
      return true;
    };
    // O_x += P_x(t) V_t, P_x in the first 64 columns of S_x.
    auto issue_pv = [&](int x, int t) -> bool {
      const int st = t % kPairVStages;
      if (!mbar_wait(&bar_p_full[x], uint32_t(t) & 1u)) return false;
      if (!mbar_wait(&bar_v_full[st], uint32_t(t / kPairVStages) & 1u)) return false;
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < kTile / 16; ++kk) {
        umma_f16_ts(tmem + 256 + 128 * x, tmem + 128 * x + 8 * kk,
                    umma_sdesc_sw128(aV + st * kTileBytes + kk * kBlockBytes, kBlockBytes / 2, 1024), idesc_o,
                    t > 0 || kk > 0);
      }
      umma_commit(&bar_pv_done[x]);
      if (x == 1) umma_commit_mc(&bar_v_empty[st], mc_mask); // both heads have read V_t: release it in both CTAs
      return true;
    };
    if (ok && n > 0) ok = issue_s(0, 0) && issue_s(1, 0);
    for (int t = 0; ok && t < n; ++t) {
      ok = issue_pv(0, t) && (t + 1 >= n || issue_s(0, t + 1)) && issue_pv(1, t) && (t + 1 >= n || issue_s(1, t + 1));
    }
    if (!ok) set_error(p.err, PKV_DEVERR_TIMEOUT);
  }

  // ---------------- softmax: warps 2-5 head A, 6-9 head B; one row per thread ----------------
  const int x = (warp - 2) >> 2;                             // head of this warpgroup (softmax warps)
  const int r = 32 * (warp & 3) + lane;                      // TMEM lane == row of the tile
  const uint32_t lane_off = uint32_t(32 * (warp & 3)) << 16;
  const int qrow = r0 + r;
  float m = -INFINITY, l = 0.f;                              // m in scaled log2 units
  if (warp >= 2) {
    const int pos = start + qrow;                            // absolute position of this query
    const float sl = p.scale_log2;                           // > 0, so max(s) * sl = max(s * sl)
    const uint32_t tS = tmem + 128 * x + lane_off, tO = tmem + 256 + 128 * x + lane_off;
    bool ok = true;
    for (int t = 0; t < n; ++t) {
      const int j = j0 + t;
      if (!(ok = mbar_wait(&bar_s_full[x], uint32_t(t) & 1u))) break;
      __syncwarp();
      tc_fence_after();
      const int lim = min(pos + 1, ctx) - j * kTile;         // keys 0 .. lim-1 of the tile are valid
      // The whole row of S in registers: one read of TMEM per tile.
      float s[kTile];
#pragma unroll
      for (int cc = 0; cc < kTile / 32; ++cc) tmem_ld32(tS + 32 * cc, *reinterpret_cast<float(*)[32]>(s + 32 * cc));
      tmem_wait_ld();
      if (lim < kTile) {                                     // the tile crosses this row's diagonal or the end
#pragma unroll
        for (int i = 0; i < kTile; ++i) s[i] = i < lim ? s[i] : -INFINITY;
      }
      float mraw;
      {
        float c4[4] = {s[0], s[1], s[2], s[3]};              // four independent chains of 3-input max
#pragma unroll
        for (int i = 4; i < kTile; i += 8) {
#pragma unroll
          for (int u = 0; u < 4; ++u) c4[u] = fmax3(c4[u], s[i + 2 * u], s[i + 2 * u + 1]);
        }
        mraw = fmaxf(fmaxf(c4[0], c4[1]), fmaxf(c4[2], c4[3]));
      }
      const float mt = mraw * sl;
      const bool grow = mt > m + kRescaleThreshold;          // also true for the first tile
      const float m_prev = m;
      if (grow) m = mt;
      // The sequence's last key tile may reach past its end: zero those V rows so that
      // 0 * garbage cannot turn into NaN inside the PV product (both heads write the same zeros).
      const int kb = j * kTile;
      if (kb + kTile > ctx) {
        if (!(ok = mbar_wait(&bar_v_full[t % kPairVStages], uint32_t(t / kPairVStages) & 1u))) break;
        if (kb + r >= ctx) {
          const uint32_t vrow = smem_u32(sV + (t % kPairVStages) * kTileBytes) + (r / kBS) * kBlockBytes + (r % kBS) * 128;
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
            for (int cc = 0; cc < 8; ++cc) sts128(vrow + hf * (kBlockBytes / 2) + cc * 16, 0u, 0u, 0u, 0u);
          }
        }
      }
      // P = 2^(s * sl - m) as 16-bit pairs written over this tile's S (keys 2e, 2e+1 go to
      // column e), two elements per packed fp32 operation.  A row with no valid key so far has
      // m = -inf and every s = -inf: m = 0 then gives P = 0.
      const float mu = m == -INFINITY ? 0.f : m;
      const uint64_t sl2 = pack_f32x2(sl, sl), nm2 = pack_f32x2(-mu, -mu);
      uint64_t acc0 = pack_f32x2(0.f, 0.f), acc1 = acc0;
#pragma unroll
      for (int hb = 0; hb < 4; ++hb) {
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int c0 = 32 * hb + 2 * e;
          const uint64_t x2 = fma_f32x2(pack_f32x2(s[c0], s[c0 + 1]), sl2, nm2);
          const float pa = fast_exp2(lo_f32(x2)), pb = fast_exp2(hi_f32(x2));
          const uint64_t p2 = pack_f32x2(pa, pb);
          if (e & 1) acc1 = add_f32x2(acc1, p2);
          else acc0 = add_f32x2(acc0, p2);
          w[e] = pack_out<kBF16>(pa, pb);
        }
        tmem_st16u(tS + 16 * hb, w);
      }
      const uint64_t acc = add_f32x2(acc0, acc1);
      const float lsum = lo_f32(acc) + hi_f32(acc);
      if (__any_sync(0xffffffffu, grow && t >= 1)) {
        // A row whose max grew rescales O, once the previous PV product has landed in it (the
        // S values are dead by now, so the rescale does not add to the loop's live registers).
        if (!(ok = mbar_wait(&bar_pv_done[x], uint32_t(t - 1) & 1u))) break;
        __syncwarp();
        tc_fence_after();
        const float alpha = (grow && m_prev != -INFINITY) ? fast_exp2(m_prev - m) : 1.f;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          float v[32];
          tmem_ld32(tO + 32 * cc, v);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] *= alpha;
          tmem_st32(tO + 32 * cc, v);
        }
        if (grow) l *= alpha;
      }
      tmem_wait_st();
      l += lsum;
      if (kb + kTile > ctx) fence_proxy_async_smem();        // the zeroed V rows, to the tensor cores
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_p_full[x]);
    }
    if (ok && n > 0) ok = mbar_wait(&bar_pv_done[x], uint32_t(n - 1) & 1u);
    if (!ok && r == 0) set_error(p.err, PKV_DEVERR_TIMEOUT);
    __syncwarp();
    tc_fence_after();
  }

  // ---------------- merge the two parts of the key range ----------------
  // The sending warpgroup stages its head's unnormalised O rows and (max, sum) in its own idle
  // K/V stages; once the peer says its receive area is free, bulk copies (one set per warp)
  // move the block there, completing on the peer's bar_x.  Layout of both areas: [row][kXStride] fp32 O (rows
  // padded by 16 bytes so that the threads' 16-byte row accesses spread over all banks), then
  // the rows' max and sum.  Only the two CTAs of a q-tile take part: the peer signals with
  // remote mbarrier arrivals, and each CTA waits for every arrival aimed at it before it leaves.
  float* xO = reinterpret_cast<float*>(sK);                  // receive area
  float* xM = xO + kTile * kXStride;
  float* xL = xM + kTile;
  float* yO = reinterpret_cast<float*>(sK + kXAreaBytes);    // staging area
  float* yM = yO + kTile * kXStride;
  float* yL = yM + kTile;
  const uint32_t xpeer = cluster_ctarank() ^ 2u;             // the same q-tile's other key half
  const int fin = int(cluster_ctarank() >> 1);               // the head this CTA finishes: its key half
  tc_fence_before();
  __syncthreads();                                           // this CTA's loads and products are all done
  tc_fence_after();
  griddep_launch_dependents();                               // the next kernel may start its prologue
  if (warp >= 2 && x != fin) {
    const uint32_t tO = tmem + 256 + 128 * x + lane_off;
    const bool have = n > 0 && m != -INFINITY;
    const uint32_t row = smem_u32(yO + r * kXStride);
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
      float v[32];
      tmem_ld32(tO + 32 * cc, v);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 32; i += 4) {
        if (have)
          sts128(row + (32 * cc + i) * 4, __float_as_uint(v[i]), __float_as_uint(v[i + 1]), __float_as_uint(v[i + 2]),
                 __float_as_uint(v[i + 3]));
        else
          sts128(row + (32 * cc + i) * 4, 0u, 0u, 0u, 0u);
      }
    }
    yM[r] = have ? m : -INFINITY;
    yL[r] = have ? l : 0.f;
    fence_proxy_async_smem();                                // the staged rows, to the bulk copy
    __syncwarp();                                            // this warp's 32 rows are staged
    if (lane == 0) {
      // Each warp sends its own rows as soon as they are staged: four copies in flight.
      const int w32 = 32 * (warp & 3);
      if (mbar_wait(&bar_ready, 0)) {
        const uint32_t bar = peer_smem_addr(smem_u32(&bar_x), xpeer);
        bulk_copy_to_peer(peer_smem_addr(smem_u32(xO + w32 * kXStride), xpeer), smem_u32(yO + w32 * kXStride),
                          32 * kXStride * 4, bar);
        bulk_copy_to_peer(peer_smem_addr(smem_u32(xM + w32), xpeer), smem_u32(yM + w32), 32 * 4, bar);
        bulk_copy_to_peer(peer_smem_addr(smem_u32(xL + w32), xpeer), smem_u32(yL + w32), 32 * 4, bar);
      } else {
        set_error(p.err, PKV_DEVERR_TIMEOUT);
      }
    }
    // The staging area is read until the peer has the whole block.
    if (r == 0 && !mbar_wait(&bar_done, 0)) set_error(p.err, PKV_DEVERR_TIMEOUT);
  } else if (warp >= 2) {
    // Finish this head: take the peer's part, combine the two by log-sum-exp, stage the output
    // rows in the idle Q area and write them out a row pair per warp instruction.
    if (r == 0) remote_arrive(peer_smem_addr(smem_u32(&bar_ready), xpeer));   // the receive area is free
    const bool got = mbar_wait(&bar_x, 0);
    if (r == 0 && got) remote_arrive(peer_smem_addr(smem_u32(&bar_done), xpeer));
    __syncwarp();
    if (!got) {
      if (r == 0) set_error(p.err, PKV_DEVERR_TIMEOUT);
    } else if (x == 0 || hq1 != hq0) {                       // the whole warp: tcgen05.ld is collective
      const float mp = xM[r], lp = xL[r];
      const bool have = n > 0 && m != -INFINITY;
      const float mo = have ? m : -INFINITY;
      const float M = fmaxf(mo, mp);
      const float wo = mo == -INFINITY ? 0.f : fast_exp2(mo - M);
      const float wp = mp == -INFINITY ? 0.f : fast_exp2(mp - M);
      const float den = wo * (have ? l : 0.f) + wp * lp;
      const float inv = den > 0.f ? 1.f / den : 0.f;
      const uint32_t tO = tmem + 256 + 128 * x + lane_off;
      const float4* po = reinterpret_cast<const float4*>(xO + r * kXStride);
      const uint32_t orow = smem_u32(sQ) + r * kOStride;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        float v[32];
        tmem_ld32(tO + 32 * cc, v);
        tmem_wait_ld();
#pragma unroll
        for (int i4 = 0; i4 < 8; ++i4) {
          const float4 q = po[8 * cc + i4];
          const int i = 4 * i4;
          v[i] = ((have ? wo * v[i] : 0.f) + wp * q.x) * inv;
          v[i + 1] = ((have ? wo * v[i + 1] : 0.f) + wp * q.y) * inv;
          v[i + 2] = ((have ? wo * v[i + 2] : 0.f) + wp * q.z) * inv;
          v[i + 3] = ((have ? wo * v[i + 3] : 0.f) + wp * q.w) * inv;
        }
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4)
          sts128(orow + (cc * 4 + q4) * 16, pack_out<kBF16>(v[8 * q4], v[8 * q4 + 1]),
                 pack_out<kBF16>(v[8 * q4 + 2], v[8 * q4 + 3]), pack_out<kBF16>(v[8 * q4 + 4], v[8 * q4 + 5]),
                 pack_out<kBF16>(v[8 * q4 + 6], v[8 * q4 + 7]));
      }
      __syncwarp();                                          // this warp's 32 rows are staged
      const int hq = x == 0 ? hq0 : hq1;
      const int rw = 32 * (warp & 3);
#pragma unroll 4
      for (int k = 0; k < 16; ++k) {
        const int rr = rw + 2 * k + (lane >> 4);
        const uint4 val = lds128(smem_u32(sQ) + rr * kOStride + (lane & 15) * 16);
        if (r0 + rr < qlen)
          reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.out) +
                                   ((int64_t(q0) + r0 + rr) * p.num_heads + hq) * (kD * 2))[lane & 15] = val;
      }
    }
  }
  tc_fence_before();
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
  if (cache->kv_dtype != q_dtype || cache->head_dim != kD || (cache->block_size != 16 && cache->block_size != 32))
    return PKV_ERR_UNSUPPORTED;
  if (num_chunks > 65535 || num_heads > 65535) return PKV_ERR_UNSUPPORTED;
  if (!(scale > 0.f)) return PKV_ERR_INVALID_ARG;          // the softmax takes max(s) * scale
  if (int64_t(cache->num_blocks) * cache->num_kv_heads * cache->block_size >= (int64_t(1) << 31))
    return PKV_ERR_UNSUPPORTED;
  // The K/V tiles are multicast across the CTAs of a cluster, so q and both caches must be
  // device memory of the current GPU: host, managed or another GPU's memory is refused
  // before any tensor map is built.
  if (!on_current_device(q) || !on_current_device(k_cache) || !on_current_device(v_cache))
    return PKV_ERR_INVALID_ARG;
  unsigned* err = error_word_ptr();
  if (!err) return PKV_ERR_CUDA;

  CUtensorMap tq, tk, tv;
  const uint64_t rows = uint64_t(cache->num_blocks) * cache->num_kv_heads * cache->block_size;
  if (!encode_tmap_3d(&tq, CU_TENSOR_MAP_DATA_TYPE_UINT16, q, kD, uint64_t(num_heads), uint64_t(total_q), kD * 2,
                      uint64_t(num_heads) * kD * 2, 64, 1, kTile, CU_TENSOR_MAP_SWIZZLE_128B) ||
      // K / V as (64 dims, rows, 2 halves): a K box is 16 rows of one half, a V box both halves
      !encode_tmap_3d(&tk, CU_TENSOR_MAP_DATA_TYPE_UINT16, k_cache, 64, rows, 2, kD * 2, 128, 64, kBS, 1,
                      CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tmap_3d(&tv, CU_TENSOR_MAP_DATA_TYPE_UINT16, v_cache, 64, rows, 2, kD * 2, 128, 64, kBS, 2,
                      CU_TENSOR_MAP_SWIZZLE_128B))
    return PKV_ERR_CUDA;

  PrefillParams prm;
  prm.out = out;
  prm.cu_q_lens = cu_q_lens;
  prm.q_start_pos = q_start_pos;
  prm.block_tables = block_tables;
  prm.max_blocks = max_blocks_per_seq;
  prm.num_blocks = cache->num_blocks;
  prm.block_size = cache->block_size;
  prm.tile_shift = cache->block_size == 32 ? 1 : 0;
  prm.num_heads = num_heads;
  prm.num_kv_heads = cache->num_kv_heads;
  prm.scale_log2 = scale * 1.4426950408889634f;
  prm.err = err;

  const int G = num_heads / cache->num_kv_heads;
  if (G >= 2) {
    // Two query heads of a kv head per CTA; clusters of 2 q-tiles x 2 halves of the key range.
    const int spg = (G + 1) / 2;
    if (int64_t(num_chunks) * 2 > 65535 || int64_t(cache->num_kv_heads) * spg > 65535) return PKV_ERR_UNSUPPORTED;
    auto pk = q_dtype == PKV_BF16 ? prefill_pair_kernel<true> : prefill_pair_kernel<false>;
    if (cudaFuncSetAttribute(pk, cudaFuncAttributeMaxDynamicSharedMemorySize, kPairSmemBytes) != cudaSuccess)
      return PKV_ERR_CUDA;
    cudaLaunchConfig_t pc = {};
    pc.gridDim = dim3(((max_q_len + kTile - 1) / kTile + 1) & ~1, cache->num_kv_heads * spg, num_chunks * 2);
    pc.blockDim = dim3(kPairThreads);
    pc.dynamicSmemBytes = kPairSmemBytes;
    pc.stream = reinterpret_cast<cudaStream_t>(stream);
    cudaLaunchAttribute pa[2];
    pa[0].id = cudaLaunchAttributeClusterDimension;
    pa[0].val.clusterDim.x = 2;
    pa[0].val.clusterDim.y = 1;
    pa[0].val.clusterDim.z = 2;
    pa[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pa[1].val.programmaticStreamSerializationAllowed = 1;
    pc.attrs = pa;
    pc.numAttrs = 2;
    return cudaLaunchKernelEx(&pc, pk, tq, tk, tv, prm) == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
  }
  auto kern = q_dtype == PKV_BF16 ? prefill_chunk_kernel<true> : prefill_chunk_kernel<false>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) != cudaSuccess)
    return PKV_ERR_CUDA;
  // Query tiles rounded up to whole clusters; tiles past a chunk's rows only help fetch K/V.
  const int qtiles = (max_q_len + kTile - 1) / kTile;
  dim3 grid((qtiles + kCluster - 1) / kCluster * kCluster, num_heads, num_chunks);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = reinterpret_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, prm) == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}
