// paged_prefill_chunk: causal attention of a prefill chunk over its paged history.
//
// Method ("Lecture 33 — KV Cache management" §4.2): a long prompt is cut into chunks; a
// chunk's tokens attend, with a causal mask, the KV of the chunks already cached plus the
// chunk itself.  Query row r of a chunk that starts at position q_start sits at position
// p = q_start + r and attends keys 0..p of its sequence, read through the block table
// (§2.2–§2.3) — the same paged cache the decode kernel reads.
//
// GB300 design: one CTA per SM holds two row blocks of 128 query rows that read the same K/V
// (two query heads of a kv head, or two adjacent query tiles of a head when each query head has
// its own kv head), and walks half of their key range; the CTA with the other half finishes the
// rows with it.  Roles, TMEM layout and the merge are described above the kernel below.
// K and V are gathered from the paged cache by TMA, one box per 16-row half block (K, in two
// 64-dim halves so that one N = 128 product covers a tile) or per block (V), by physical block
// id from the block table, read 32 entries at a time, lane-parallel, one window ahead.
// Every wait is bounded; a timeout sets PKV_DEVERR_TIMEOUT and the CTA drains and exits.
#include "pkv_device.cuh"
#include "pkv_host.h"

namespace pkv {
namespace {

constexpr int kBS = 16;        // rows per TMA box: a 16-token block, or half of a 32-token one
constexpr int kD = 128;
constexpr int kTile = 128;                    // query rows per CTA and keys per iteration
constexpr uint32_t kTmemCols = 512;           // S_A | S_B | O_A | O_B, 128 columns each
constexpr int kHalfBytes = kTile * 128;       // [128 rows][64 elements] of 2 bytes = 16 KB
constexpr int kTileBytes = 2 * kHalfBytes;    // one 128 x 128 operand = 32 KB
// A V tile holds 8 blocks of 4 KB: block b at 4 KB * b = [dims 0..63: 16 rows x 128 B]
// [dims 64..127: 16 rows x 128 B], each half 128-byte swizzled (one 3-D TMA box per block).
// A K tile holds the same bytes as [dims 0..63: block 0..7 x 16 rows][dims 64..127: ...]
// (two 2-D boxes of 2 KB per block).
constexpr int kBlockBytes = kBS * kD * 2;
constexpr float kRescaleThreshold = 8.f;      // log2 units

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

// ---------------------------------------------------------------------------------------
// Two row blocks A and B of 128 query rows per CTA, the key range split between two CTAs.
//
// Rows that read the same K/V share a CTA, so every K/V tile it receives feeds 256 query rows:
// - grouped heads (kQPair false): A and B are the same q-tile of two query heads of one kv head.
//   A cluster is two adjacent q-tiles x two halves of their key range.  The two CTAs of a half
//   read the same keys; each issues half of every tile's TMA boxes and multicasts them to both;
// - one query head per kv head (kQPair true): A and B are two adjacent q-tiles of one head, and
//   the cluster is the two halves of their key range; each CTA loads its tiles itself.
// Both row blocks walk the keys the later rows need; the causal mask drops the rest.
//   warp 0     : TMA producer: Q of both row blocks once, then the boxes of K and V of the
//                half's key tiles (2 stages each).  A stage is refilled once every CTA that
//                reads it has released it with a tensor-core commit.
//   warp 1     : TMEM owner (512 columns: S_A | S_B | O_A | O_B) and MMA issuer, in the
//                fixed order S_A(0) S_B(0) | PV_A(t) S_A(t+1) PV_B(t) S_B(t+1) | ... so that
//                one block's softmax overlaps the other block's products.
//   warps 2-5  : softmax of block A, warps 6-9: block B; one query row per thread.  The row's
//                128 scores are read from TMEM once; the max uses 3-input max, P = 2^(s*c - m)
//                uses packed fp32x2 multiply-add and add; P goes over S in TMEM; O is rescaled
//                only when the row max grows by more than 2^8.
// At the end the first-half CTA finishes block A and the second-half CTA block B.  Each CTA
// stages the other block's unnormalised O rows and (max, sum) in its idle stages and sends
// them to its peer with bulk shared-memory copies; the receiver combines the two parts by
// log-sum-exp, stages the 16-bit rows in the idle Q area and writes them out coalesced.
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

template <bool kBF16, bool kQPair>
__global__ void __launch_bounds__(kPairThreads, 1)
    prefill_pair_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                        const __grid_constant__ CUtensorMap tmv, const PrefillParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar_q, bar_k_full[kPairKStages], bar_k_empty[kPairKStages],
      bar_v_full[kPairVStages], bar_v_empty[kPairVStages], bar_s_full[2], bar_p_full[2], bar_pv_done[2], bar_x,
      bar_ready, bar_done;
  __shared__ uint32_t tmem_base_sh;

  const int qt = blockIdx.x, slot = blockIdx.y, c = blockIdx.z >> 1;
  // Grouped heads: crank = (q-tile of the pair) + 2 * (key half).  Query-tile pairs: the
  // cluster is the two key halves, crank = key half.
  const uint32_t crank = cluster_ctarank();
  const uint32_t khalf = kQPair ? crank : crank >> 1;
  const uint16_t mc_mask = uint16_t(3u << (2 * khalf));     // the two CTAs reading this half's keys (grouped heads)
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
    // A stage is free again once every CTA reading it has released it: with grouped heads the
    // two CTAs of this key half (each one's tensor-core commit arrives on the stage's empty
    // barrier in both), with query-tile pairs this CTA alone.
    for (int i = 0; i < kPairKStages; ++i) {
      mbar_init(&bar_k_full[i], 1);
      mbar_init(&bar_k_empty[i], kQPair ? 1 : 2);
    }
    for (int i = 0; i < kPairVStages; ++i) {
      mbar_init(&bar_v_full[i], 1);
      mbar_init(&bar_v_empty[i], kQPair ? 1 : 2);
    }
    // One phase per key tile each.  A row block's softmax waits on its pv_done on every tile,
    // for the previous tile's product, and the next product needs this tile's P first, so the
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

  // Launched as a programmatic dependent: the CTA may start while the previous kernel runs.
  // Everything above reads no input; nothing below runs before that kernel has finished.
  griddep_wait();
  const int q0 = p.cu_q_lens[c];
  const int qlen = p.cu_q_lens[c + 1] - q0;
  // First query row of each of the CTA's two row blocks ("heads" A and B): the same q-tile of
  // two query heads, or two adjacent q-tiles of one head.
  const int r0_pair = kQPair ? 2 * qt * kTile : (qt & ~1) * kTile;
  const int r0a = kQPair ? r0_pair : qt * kTile;
  const int r0b = kQPair ? r0_pair + kTile : qt * kTile;
  const int start = p.q_start_pos[c];
  const int ctx = start + qlen;                              // keys 0 .. ctx-1 exist
  // Nothing to do, or a bad chunk: the same for every CTA of the cluster, and nothing has been
  // started that another CTA waits for; give back the TMEM and leave.
  const bool idle = qlen <= 0 || r0_pair >= qlen;
  const bool bad = !idle && (start < 0 || ctx > p.max_blocks * p.block_size);
  // A chunk longer than the grid covers (max_q_len below its length) leaves rows unwritten.
  if (qt == int(gridDim.x) - 1 && threadIdx.x == 0 && qlen > int(gridDim.x) * (kQPair ? 2 : 1) * kTile)
    set_error(p.err, PKV_DEVERR_CHUNK);
  if (idle || bad) {
    if (bad && threadIdx.x == 0) set_error(p.err, PKV_DEVERR_CHUNK);
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
      __syncwarp();
      tc_fence_after();
      tmem_dealloc(tmem, kTmemCols);
    }
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
  const int spg = kQPair ? 1 : (G + 1) / 2;                  // head pairs (slots) per kv head
  const int h = slot / spg;                                  // kv head
  const int hq0 = kQPair ? slot : h * G + 2 * (slot % spg);
  // An odd group's last slot repeats a head (its second part is computed and dropped).
  const int hq1 = kQPair ? slot : (2 * (slot % spg) + 1 < G ? hq0 + 1 : hq0);
  const bool b_live = kQPair || hq1 != hq0;                  // row block B is output
  const int nb = (ctx + kBS - 1) / kBS;
  const int32_t* table = p.block_tables + int64_t(c) * p.max_blocks;


  if (warp == 0) {
    // ---------------- TMA producer ----------------
    const uint64_t pol_q = l2_policy_evict_first();
    const uint64_t pol_kv = l2_policy_evict_last();          // re-read by the other query heads
    if (lane == 0) {
      mbar_arrive_expect_tx(&bar_q, 2 * kTileBytes);
      tma_load_3d(sQ, &tmq, &bar_q, 0, hq0, q0 + r0a, pol_q);
      tma_load_3d(sQ + kHalfBytes, &tmq, &bar_q, 64, hq0, q0 + r0a, pol_q);
      tma_load_3d(sQ + kTileBytes, &tmq, &bar_q, 0, hq1, q0 + r0b, pol_q);
      tma_load_3d(sQ + kTileBytes + kHalfBytes, &tmq, &bar_q, 64, hq1, q0 + r0b, pol_q);
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
      if (blk >= 0 && blk < kTile / kBS) {
        if constexpr (kQPair) {                              // both 64-dim halves, this CTA alone
#pragma unroll
          for (int hf = 0; hf < 2; ++hf)
            tma_load_3d(dst + hf * kHalfBytes + blk * (kBlockBytes / 2), &tmk, bar, 0, wk.cur, hf, pol_kv);
        } else {                                             // this CTA's half hf, to both CTAs
          const int hf = int(crank & 1u);
          tma_load_3d_mc(dst + hf * kHalfBytes + blk * (kBlockBytes / 2), &tmk, bar, 0, wk.cur, hf, mc_mask, pol_kv);
        }
      }
    };
    auto issue_v = [&](uint8_t* dst, uint64_t* bar, int j) {
      seek(wv, j);
      const int first = (8 * j) % 32;
      if (lane == first) mbar_arrive_expect_tx(bar, kTileBytes);
      __syncwarp();
      const int blk = lane - first;
      if constexpr (kQPair) {
        if (blk >= 0 && blk < kTile / kBS) tma_load_3d(dst + blk * kBlockBytes, &tmv, bar, 0, wv.cur, 0, pol_kv);
      } else {
        if (blk >= 0 && blk < kTile / kBS && uint32_t(blk & 1) == (crank & 1u))   // every other block, to both
          tma_load_3d_mc(dst + blk * kBlockBytes, &tmv, bar, 0, wv.cur, 0, mc_mask, pol_kv);
      }
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
      if (x == 1) {                                          // both row blocks have read K_t: release it
        if constexpr (kQPair) umma_commit(&bar_k_empty[st]);
        else umma_commit_mc(&bar_k_empty[st], mc_mask);      // in both CTAs that read it
      }
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
      if (x == 1) {                                          // both row blocks have read V_t: release it
        if constexpr (kQPair) umma_commit(&bar_v_empty[st]);
        else umma_commit_mc(&bar_v_empty[st], mc_mask);      // in both CTAs that read it
      }
      return true;
    };
    if (ok && n > 0) ok = issue_s(0, 0) && issue_s(1, 0);
    for (int t = 0; ok && t < n; ++t) {
      ok = issue_pv(0, t) && (t + 1 >= n || issue_s(0, t + 1)) && issue_pv(1, t) && (t + 1 >= n || issue_s(1, t + 1));
    }
    if (!ok) set_error(p.err, PKV_DEVERR_TIMEOUT);
  }

  // ---------------- softmax: warps 2-5 row block A, 6-9 row block B; one row per thread ----------------
  const int x = (warp - 2) >> 2;                             // row block of this warpgroup (softmax warps)
  const int r = 32 * (warp & 3) + lane;                      // TMEM lane == row of the tile
  const uint32_t lane_off = uint32_t(32 * (warp & 3)) << 16;
  const int qrow = (x == 0 ? r0a : r0b) + r;
  float m = -INFINITY, l = 0.f;                              // m in scaled log2 units
  if (warp >= 2) {
    const int pos = start + qrow;                            // absolute position of this query
    const float sl = p.scale_log2;                           // > 0, so max(s) * sl = max(s * sl)
    const uint32_t tS = tmem + 128 * x + lane_off, tO = tmem + 256 + 128 * x + lane_off;
    bool ok = true;
    for (int t = 0; t < n; ++t) {
      const int j = j0 + t;
      if (!(ok = mbar_wait(&bar_s_full[x], uint32_t(t) & 1u))) break;
      // Observe every phase of pv_done: PV(t-1) is done by now (S(t) was issued after it), and
      // waiting for it on every tile keeps the barrier at most one phase ahead of this wait, so
      // the parity waits here and after the loop cannot mistake a phase two behind for a
      // completed one (completion arrivals on different barriers may land out of order).
      if (t >= 1 && !(ok = mbar_wait(&bar_pv_done[x], uint32_t(t - 1) & 1u))) break;
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
        // A row whose max grew rescales O, into which the previous PV product has landed
        // (waited for at the top of the tile).
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
  const uint32_t xpeer = cluster_ctarank() ^ (kQPair ? 1u : 2u);   // the same rows' other key half
  const int fin = int(kQPair ? cluster_ctarank() : cluster_ctarank() >> 1);   // the row block this CTA finishes
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
    } else if (x == 0 || b_live) {                           // the whole warp: tcgen05.ld is collective
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
        const int orow = (x == 0 ? r0a : r0b) + rr;
        const uint4 val = lds128(smem_u32(sQ) + rr * kOStride + (lane & 15) * 16);
        if (orow < qlen)
          reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.out) +
                                   ((int64_t(q0) + orow) * p.num_heads + hq) * (kD * 2))[lane & 15] = val;
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
  // The kernel bounds a chunk's context by max_blocks_per_seq * block_size in 32-bit arithmetic.
  if (int64_t(max_blocks_per_seq) * cache->block_size >= (int64_t(1) << 31)) return PKV_ERR_UNSUPPORTED;
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

  // Two row blocks of 128 query rows per CTA, the key range split between two CTAs.  Grouped
  // heads: two query heads of a kv head, clusters of 2 q-tiles x 2 key halves.  One query
  // head per kv head: two adjacent q-tiles of a head, clusters of the 2 key halves.
  const int G = num_heads / cache->num_kv_heads;
  {
    const bool qpair = G == 1;
    const int spg = (G + 1) / 2;
    const int qtiles = (max_q_len + kTile - 1) / kTile;
    const dim3 grid = qpair ? dim3((qtiles + 1) / 2, num_heads, num_chunks * 2)
                            : dim3((qtiles + 1) & ~1, cache->num_kv_heads * spg, num_chunks * 2);
    if (int64_t(num_chunks) * 2 > 65535 || grid.y > 65535) return PKV_ERR_UNSUPPORTED;
    auto pk = qpair ? (q_dtype == PKV_BF16 ? prefill_pair_kernel<true, true> : prefill_pair_kernel<false, true>)
                    : (q_dtype == PKV_BF16 ? prefill_pair_kernel<true, false> : prefill_pair_kernel<false, false>);
    if (cudaFuncSetAttribute(pk, cudaFuncAttributeMaxDynamicSharedMemorySize, kPairSmemBytes) != cudaSuccess)
      return PKV_ERR_CUDA;
    cudaLaunchConfig_t pc = {};
    pc.gridDim = grid;
    pc.blockDim = dim3(kPairThreads);
    pc.dynamicSmemBytes = kPairSmemBytes;
    pc.stream = reinterpret_cast<cudaStream_t>(stream);
    cudaLaunchAttribute pa[2];
    pa[0].id = cudaLaunchAttributeClusterDimension;
    pa[0].val.clusterDim.x = qpair ? 1 : 2;
    pa[0].val.clusterDim.y = 1;
    pa[0].val.clusterDim.z = 2;
    pa[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pa[1].val.programmaticStreamSerializationAllowed = 1;
    pc.attrs = pa;
    pc.numAttrs = 2;
    return cudaLaunchKernelEx(&pc, pk, tq, tk, tv, prm) == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
  }
}
