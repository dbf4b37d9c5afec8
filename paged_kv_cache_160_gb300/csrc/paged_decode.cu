// paged_decode: one query token per running sequence over its paged K/V.
//
// Method ("Lecture 33 — KV Cache management" §2.3): for each sequence and head, walk the
// sequence's logical blocks, look up each physical block in the block table, load its
// 16 K rows, form the scores with the query, keep a running (online) softmax, then load
// the 16 V rows and accumulate; no gather copy is ever made.  The result equals plain
// softmax attention (§8.1 row 1).  GQA: query head h reads kv head h / group
// ("PagedAttention: manage the KV cache like virtual memory" §9 names GQA; the
// contiguous grouping is this library's reading).
//
// GB300 design
//   * Work unit = one (sequence, kv head, logical block) tile: 16 tokens x head_dim of K and
//     of V, each a contiguous run in the [block][kv_head][row][dim] pool.
//   * Persistent grid, one CTA per SM, 12 independent worker warps per CTA.  The flattened
//     tile list (sequence-major, kv head, block) is cut into equal contiguous ranges, one
//     per worker ("balanced" split), or into equal runs of whole partition_size-token
//     partitions.  A worker's online softmax runs across consecutive partitions.
//   * Each worker warp owns a ring of TMA stages: lane 0 issues one tensor load for the K
//     tile and one for the V tile (128-byte swizzled; a 256-byte row arrives as two swizzled
//     halves) straight from the physical block named by the block table, completing on an
//     mbarrier; the warp waits, computes, and refills the stage.  (TMA instruction issue, not
//     bytes, limits small boxes, so each tile is a single box.)
//   * All query heads of a kv head (group <= 8) are processed together on tensor cores:
//     S^T[16 tok x 8 heads] = K[16 x D] * Q^T (m16n8k16, K as the A operand from ldmatrix),
//     online softmax in registers (warp shuffles over the 16 tokens), P^T transposed with
//     movmatrix, O^T[D x 8] += V^T[D x 16] * P^T (V^T via ldmatrix.trans).  For e4m3 caches
//     the fragments are loaded with plain shared loads in a head_dim/token order chosen so
//     every lane reads 16 contiguous bytes, and converted exactly to fp16.
//   * A range that covers only part of a (sequence, kv head) writes a partial (m, l, o) to
//     the workspace (at most two per worker) and the worker holding the segment's first
//     tile describes its pieces; a second kernel, launched as a programmatic dependent,
//     merges them by log-sum-exp.  A segment that lies inside one range is written directly.
//   * Everything that depends only on lengths and block tables (prefix sums, ranges,
//     cursors, first block ids, the pool rows of the first tiles) runs before the wait on
//     the previous kernel, in 32-bit arithmetic; after it only the TMA issues remain.
//   * Fused append (pkv_paged_decode_append): the warp holding a segment's last tile also
//     places the step's new K/V row there, in the staged tile and in the cache.
#include <algorithm>
#include <atomic>
#include <utility>

#include "pkv_device.cuh"
#include "pkv_host.h"

namespace pkv {
namespace {

enum { KV_F16 = 0, KV_BF16 = 1, KV_E4M3 = 2 };

constexpr int kBS = 16;        // tokens per tile: a 16-token block, or half of a 32-token one
constexpr int kMaxWarps = 12;  // worker warps per CTA (3 per SM sub-partition)
constexpr int kMaxGroup = 8;   // query heads per kv head handled by one n=8 MMA tile

template <int KV, int D>
struct Cfg {
  static constexpr int kElt = KV == KV_E4M3 ? 1 : 2;
  static constexpr int kRowBytes = D * kElt;
  static constexpr int kNBox = kRowBytes / 128;       // 128-byte-wide TMA boxes per row
  static constexpr int kRowChunks = kRowBytes / 16;   // 16-byte chunks per cache row
  static constexpr int kTileBytes = kBS * kRowBytes;  // one 16-row K (or V) tile
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kKSteps = D / 16;
  static constexpr int kMTiles = D / 16;
  static constexpr bool kBF16 = KV == KV_BF16;        // MMA input type (e4m3 computes in fp16)
  static_assert(kRowBytes % 128 == 0, "rows must span whole 128-byte swizzle atoms");
  static_assert(KV != KV_E4M3 || D == 128, "e4m3 path is written for head_dim 128");
};

struct DecodeParams {
  void* out;
  const void* q;
  const int32_t* block_tables;
  const int32_t* context_lens;
  const float* k_scale;
  const float* v_scale;
  int num_seqs;
  int num_kv_heads;
  int group;
  int max_blocks;
  int max_len;            // min(max_blocks * block_size, max_context_len): lengths are clamped to it
  int num_blocks;
  int block_size;         // tokens per pool block: 16 or 32 (1 or 2 tiles)
  int tile_shift;         // log2(block_size / 16)
  int part_blocks;        // tiles per partition; 0 = balanced split
  int num_workers;        // gridDim.x * worker warps per CTA
  int defer_dependents;   // 1: the merge kernel launches when this grid completes, not at its start
  float scale_log2;       // softmax scale * log2(e)
  float2* ml;             // [slots][group] (running max in log2 units, sum of exponentials)
  float* po;              // [slots][group][D] unnormalised partial outputs
  unsigned* err;
  // Fused append (null k_new: plain decode): each sequence's new K/V row, [num_seqs][num_kv_heads][D]
  // in the q dtype, belongs at position context_len - 1; it is written to the caches and attended.
  const void* k_new;
  const void* v_new;
  void* k_cache;
  void* v_cache;
};

struct Tile {
  int s, h, b, nb, len;
};

// Largest s in [lo, hi] with mult * cum[s] <= t, given mult * cum[lo] <= t.  cum is a
// non-decreasing prefix array whose scaled entries stay below 2^31 (checked on the host).
__device__ __forceinline__ int find_seq(const int* cum, int lo, int hi, int t, int mult) {
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (mult * cum[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// The same search over [0, S) done by a whole warp for one t: each round the 32 lanes probe
// 32 evenly spaced candidates and a ballot keeps the chunk holding the answer, so S entries
// take ceil(log32 S) rounds instead of log2 S dependent probes.
__device__ __forceinline__ int find_seq_warp(const int* cum, int S, int t, int mult, int lane) {
  int lo = 0, n = S;                         // the answer lies in [lo, lo + n); mult * cum[lo] <= t
  while (n > 1) {
    const int step = (n + 31) >> 5;
    const int pos = lo + lane * step;
    const bool ok = lane * step < n && mult * cum[pos] <= t;
    const unsigned b = __ballot_sync(0xffffffffu, ok);   // lane 0 always holds: b != 0
    const int k = 31 - __clz(b);
    lo += k * step;
    n = min(step, n - k * step);
  }
  return lo;
}

__device__ __forceinline__ int clamp_len(int L, int max_len) { return min(max(L, 0), max_len); }

template <int QT>
__device__ __forceinline__ float2 q_pair(const void* q, int64_t elem) {
  if constexpr (QT == KV_BF16) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(static_cast<const __nv_bfloat16*>(q) + elem));
  } else {
    return __half22float2(*reinterpret_cast<const __half2*>(static_cast<const __half*>(q) + elem));
  }
}

template <int QT>
__device__ __forceinline__ void store_out(void* out, int64_t elem, float v) {
  if constexpr (QT == KV_BF16) {
    static_cast<__nv_bfloat16*>(out)[elem] = __float2bfloat16_rn(v);
  } else {
    static_cast<__half*>(out)[elem] = __float2half_rn(v);
  }
}

// head_dim index held by accumulator row `r` (0: row g, 1: row g + 8) of m-tile i.
template <int KV>
__device__ __forceinline__ int out_dim(int i, int r, int g) {
  if constexpr (KV == KV_E4M3) return 16 * g + 2 * i + r;
  else return 16 * i + g + 8 * r;
}

template <int KV, int QT, int D, int kWarps, int kStages>
__global__ void __launch_bounds__(kWarps * 32, 1)
    paged_decode_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                        const DecodeParams p) {
  using C = Cfg<KV, D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[kWarps][kStages];
  __shared__ int warp_tot[kWarps * 2];

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int S = p.num_seqs;
  const int Hkv = p.num_kv_heads;
  const int G = p.group;
  const int PB = p.part_blocks;
  int* cum_nb = reinterpret_cast<int*>(smem + kWarps * kStages * C::kStageBytes);   // [S + 1]
  int* cum_np = cum_nb + (S + 1);                                                    // [S + 1]
  int* lenc = cum_np + (S + 1);                                                      // [S] clamped lengths

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, tq = lane & 3;

  if (threadIdx.x == 0) {
    prefetch_tensormap(&tmk);
    prefetch_tensormap(&tmv);
  }
  if (lane == 0) {
    for (int st = 0; st < kStages; ++st) mbar_init(&bars[warp][st], 1);
    fence_mbar_init();
  }

  // ---- per-CTA prefix sums of blocks (and partitions) per sequence ---------------------
  // The lengths are read from global memory once; the clamped values stay in shared memory
  // for the second pass and for every cursor step below.
  {
    const int per = (S + blockDim.x - 1) / blockDim.x;
    const int s0 = min(S, int(threadIdx.x) * per), s1 = min(S, s0 + per);
    int a = 0, u = 0;
    for (int s = s0; s < s1; ++s) {
      const int L = p.context_lens[s];
      const int Lc = clamp_len(L, p.max_len);
      if (Lc != L) set_error(p.err, PKV_DEVERR_CONTEXT_LEN);
      lenc[s] = Lc;
      const int nb = (Lc + kBS - 1) / kBS;
      a += nb;
      u += PB ? (nb + PB - 1) / PB : 0;
    }
    int ia = a, iu = u;   // inclusive warp scan
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int va = __shfl_up_sync(0xffffffffu, ia, o), vu = __shfl_up_sync(0xffffffffu, iu, o);
      if (lane >= o) { ia += va; iu += vu; }
    }
    if (lane == 31) { warp_tot[warp] = ia; warp_tot[kWarps + warp] = iu; }
    __syncthreads();
    int ba = 0, bu = 0;
    for (int w = 0; w < warp; ++w) { ba += warp_tot[w]; bu += warp_tot[kWarps + w]; }
    int ra = ba + ia - a, ru = bu + iu - u;   // exclusive prefix at s0
    for (int s = s0; s < s1; ++s) {
      const int nb = (lenc[s] + kBS - 1) / kBS;
      cum_nb[s] = ra;
      cum_np[s] = ru;
      ra += nb;
      ru += PB ? (nb + PB - 1) / PB : 0;
    }
    if (threadIdx.x == blockDim.x - 1) {
      int ta = 0, tu = 0;
      for (int w = 0; w < kWarps; ++w) { ta += warp_tot[w]; tu += warp_tot[kWarps + w]; }
      cum_nb[S] = ta;
      cum_np[S] = tu;
    }
  }
  __syncthreads();

  // Sequences with nothing to attend produce zeros (their tiles never exist).
  auto zero_empty = [&]() {
    for (int s = blockIdx.x; s < S; s += gridDim.x) {
      if (cum_nb[s + 1] != cum_nb[s]) continue;
      const int n = Hkv * G * D;
      for (int e = threadIdx.x; e < n; e += blockDim.x) store_out<QT>(p.out, int64_t(s) * n + e, 0.f);
    }
  };

  // Tile and unit counts stay below 2^31 (checked on the host), so the index arithmetic
  // from here on is 32-bit.
  const int T = Hkv * cum_nb[S];
  const int U = Hkv * cum_np[S];
  const int nunits = PB ? U : T;
  const int W = min(p.num_workers, nunits);
  const int w = blockIdx.x * kWarps + warp;
  if (w >= W) {                              // no tiles for this warp
    griddep_wait();
    if (!p.defer_dependents) griddep_launch_dependents();
    zero_empty();
    return;
  }

  // Cursor of tile t, searching sequences lo..hi (which must hold it).
  auto locate_in = [&](int t, int lo, int hi) -> Tile {
    Tile r;
    r.s = find_seq(cum_nb, lo, hi, t, Hkv);
    r.nb = cum_nb[r.s + 1] - cum_nb[r.s];
    const int off = t - Hkv * cum_nb[r.s];
    r.h = off / r.nb;
    r.b = off - r.h * r.nb;
    r.len = lenc[r.s];
    return r;
  };
  auto locate = [&](int t) -> Tile {         // whole warp, same t
    const int s = find_seq_warp(cum_nb, S, t, Hkv, lane);
    return locate_in(t, s, s);
  };
  // First tile of unit u (partition mode) in the flattened tile order; whole warp.
  auto unit_tile = [&](int u) -> int {
    if (u >= U) return T;
    const int s = find_seq_warp(cum_np, S, u, Hkv, lane);
    const int np = cum_np[s + 1] - cum_np[s];
    const int nb = cum_nb[s + 1] - cum_nb[s];
    const int off = u - Hkv * cum_np[s];
    const int h = off / np, part = off - h * np;
    return Hkv * cum_nb[s] + h * nb + part * PB;
  };
  // Worker wi starts at unit floor(wi * nunits / W).  With nunits = uq * W + ur that is
  // wi * uq + floor(wi * ur / W), and wi * ur < W^2 fits 32 unsigned bits.
  const unsigned uq = unsigned(nunits) / unsigned(W), ur = unsigned(nunits) % unsigned(W);
  auto start_of = [&](int wi) -> int { return int(unsigned(wi) * uq + unsigned(wi) * ur / unsigned(W)); };

  int t_begin, t_end;
  if (PB) {
    t_begin = unit_tile(start_of(w));
    t_end = unit_tile(start_of(w + 1));
  } else {
    t_begin = start_of(w);
    t_end = start_of(w + 1);
  }
  const int n = t_end - t_begin;
  const Tile first = locate(t_begin);
  const Tile last = locate(t_end - 1);

  uint8_t* my_stages = smem + warp * kStages * C::kStageBytes;
  const uint64_t pol = l2_policy_evict_first();

  // Walk to the next tile in flattened order (sequence, kv head, block), skipping
  // sequences without tiles.
  auto advance = [&](Tile& c) {
    if (++c.b < c.nb) return;
    c.b = 0;
    if (++c.h < Hkv) return;
    c.h = 0;
    do { ++c.s; } while (c.s < S && cum_nb[c.s + 1] == cum_nb[c.s]);
    if (c.s < S) {
      c.nb = cum_nb[c.s + 1] - cum_nb[c.s];
      c.len = lenc[c.s];
    }
  };

  // Block ids of the worker's tiles, 32 per window: lane l holds the id of tile
  // 32 * window + l of the range.  The next window is loaded one window ahead so the
  // table lookups never sit on the path from one TMA issue to the next.  The range's tiles
  // lie in sequences first.s .. last.s, so each lane searches only those.
  auto load_window = [&](int win) -> int {
    const int t = t_begin + win * 32 + lane;
    if (t >= t_end) return -1;
    const Tile c = locate_in(t, first.s, last.s);
    return p.block_tables[int64_t(c.s) * p.max_blocks + (c.b >> p.tile_shift)];
  };
  int bid_cur = load_window(0);
  int bid_nxt = n > 32 ? load_window(1) : -1;

  // First pool row of tile c in block pb: the (block, kv head) rows start at
  // (pb * Hkv + h) * block_size and a 32-token block holds the tile's 16 rows at offset 0
  // or 16.  -1 marks a block id outside the pool.
  auto tile_row = [&](const Tile& c, int pb) -> int {
    if (pb < 0 || pb >= p.num_blocks) return -1;
    return int((int64_t(pb) * Hkv + c.h) * p.block_size + (c.b & ((1 << p.tile_shift) - 1)) * kBS);
  };
  // Lane 0 starts the TMA loads of one tile (pool row y) into stage st and records in
  // `valid` (bit st) whether the tile's block id was inside the pool.
  uint32_t valid = 0;
  auto launch_tile = [&](int y, int st) {
    uint64_t* bar = &bars[warp][st];
    if (y < 0) {
      set_error(p.err, PKV_DEVERR_BLOCK_ID);
      valid &= ~(1u << st);
      mbar_arrive(bar);                      // completes the phase without data
      return;
    }
    valid |= 1u << st;
    mbar_arrive_expect_tx(bar, C::kStageBytes);
    uint8_t* kdst = my_stages + st * C::kStageBytes;
    if constexpr (C::kNBox == 2) {
      // One 3-D box brings both 128-byte halves of the 16 rows: [half 0: 16 x 128 B][half 1].
      tma_load_3d(kdst, &tmk, bar, 0, y, 0, pol);
      tma_load_3d(kdst + C::kTileBytes, &tmv, bar, 0, y, 0, pol);
    } else {
      tma_load_2d(kdst, &tmk, bar, 0, y, pol);
      tma_load_2d(kdst + C::kTileBytes, &tmv, bar, 0, y, pol);
    }
  };
  // Issues the worker's tile j (cursor c) into stage st.  Whole warp calls it.
  auto issue = [&](const Tile& c, int j, int st) {
    if (j % 32 == 0 && j > 0) {
      bid_cur = bid_nxt;
      bid_nxt = load_window(j / 32 + 1);
    }
    const int pb = __shfl_sync(0xffffffffu, bid_cur, j % 32);
    if (lane == 0) launch_tile(tile_row(c, pb), st);
  };

  // Pool rows of the first kStages tiles, so that only the TMA issue itself follows the wait.
  Tile pc = first;                           // producer cursor, kStages tiles ahead
  int y0[kStages];
#pragma unroll
  for (int i = 0; i < kStages; ++i) {
    const int pb = __shfl_sync(0xffffffffu, bid_cur, i);
    y0[i] = tile_row(pc, pb);
    if (i + 1 < kStages && i + 1 < n) advance(pc);
  }

  // Up to here the kernel has read only lengths and block tables.  The cache, the queries,
  // the outputs and the workspace are touched only after the preceding kernel on the stream
  // (typically the KV write of this step) has finished.
  griddep_wait();
  // The merge kernel may be launched now, so that its CTAs take the SMs this grid frees and
  // work out their pieces while the last tiles stream.  Under an SM budget the SMs outside
  // this grid belong to another kernel: the merge then waits for this grid to finish.
  if (!p.defer_dependents) griddep_launch_dependents();
  if (lane == 0) {
#pragma unroll
    for (int i = 0; i < kStages; ++i)
      if (i < n) launch_tile(y0[i], i);
  }
  if (n > kStages - 1) advance(pc);          // pc now points at tile kStages of the range
  zero_empty();

  // The query rows of the segment this range ends in are read only when that piece starts,
  // late in the range: bring them into L1 now so the switch does not wait on memory.
  if (first.s != last.s || first.h != last.h) {
    const int qbytes = G * D * 2;                      // f16 / bf16 queries
    const uint8_t* qrow0 = static_cast<const uint8_t*>(p.q) + (int64_t(last.s) * Hkv + last.h) * G * D * 2;
    for (int off = lane * 128; off < qbytes; off += 32 * 128) prefetch_l1(qrow0 + off);
  }

  Tile tl = first;                           // consumer cursor

  // Per-piece state.
  uint32_t qf[C::kKSteps][2];
  float o[C::kMTiles][4];
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float sl = p.scale_log2;
  int piece_b0 = 0;

  for (int i = 0; i < n; ++i, advance(tl)) {
    const int st = i % kStages;
    const bool piece_start = i == 0 || tl.b == 0;
    if (piece_start) {
      piece_b0 = tl.b;
      m0 = m1 = -INFINITY;
      l0 = l1 = 0.f;
#pragma unroll
      for (int mt = 0; mt < C::kMTiles; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
      sl = p.scale_log2 * (KV == KV_E4M3 ? p.k_scale[tl.h] : 1.f);
      const bool live = gq < G;
      const int64_t qrow = (int64_t(tl.s) * Hkv * G + int64_t(tl.h) * G + gq) * D;
#pragma unroll
      for (int j = 0; j < C::kKSteps; ++j) {
        if constexpr (KV == KV_E4M3) {
          float2 a = live ? q_pair<QT>(p.q, qrow + 32 * tq + 4 * j) : make_float2(0.f, 0.f);
          float2 b = live ? q_pair<QT>(p.q, qrow + 32 * tq + 4 * j + 2) : make_float2(0.f, 0.f);
          qf[j][0] = pack2<false>(a.x, a.y);
          qf[j][1] = pack2<false>(b.x, b.y);
        } else {
          const uint32_t* qw = reinterpret_cast<const uint32_t*>(p.q);
          qf[j][0] = live ? qw[(qrow + 16 * j + 2 * tq) >> 1] : 0u;
          qf[j][1] = live ? qw[(qrow + 16 * j + 8 + 2 * tq) >> 1] : 0u;
        }
      }
    }

    // Fused append: the segment's last tile holds the new token's row.  Lane l < 2 * kRowChunks
    // fetches 16 cache bytes' worth of it (K for the first half of the lanes, V for the rest)
    // while the tile is still in flight.
    const bool app = p.k_new != nullptr && tl.b + 1 == tl.nb;
    uint4 na = make_uint4(0u, 0u, 0u, 0u), nb2 = make_uint4(0u, 0u, 0u, 0u);
    int apb = -1, araw = -1;
    if (app) {
      araw = p.context_lens[tl.s];           // a clamped length has no new row to place
      apb = p.block_tables[int64_t(tl.s) * p.max_blocks + ((tl.len - 1) >> (4 + p.tile_shift))];
      if (lane < 2 * C::kRowChunks) {
        const int c = lane % C::kRowChunks;
        const uint4* src = static_cast<const uint4*>(lane < C::kRowChunks ? p.k_new : p.v_new) +
                           ((int64_t(tl.s) * Hkv + tl.h) * D * 2) / 16 + c * (KV == KV_E4M3 ? 2 : 1);
        na = src[0];
        if constexpr (KV == KV_E4M3) nb2 = src[1];
      }
    }

    if (!mbar_wait(&bars[warp][st], uint32_t(i / kStages) & 1u)) {
      // Give up: report, then wait (bounded) for this warp's loads still in flight.
      if (lane == 0) set_error(p.err, PKV_DEVERR_TIMEOUT);
      for (int k = i; k < min(n, i + kStages); ++k) (void)mbar_wait(&bars[warp][k % kStages], uint32_t(k / kStages) & 1u);
      return;
    }

    const bool ok = (__shfl_sync(0xffffffffu, valid, 0) >> st) & 1u;
    if (app && ok && araw == tl.len) {
      // Row r of the tile is position len - 1.  Put the new row into the staged tile (same
      // swizzled layout as the TMA box) and into the cache at that position.
      if (lane < 2 * C::kRowChunks) {
        const bool isv = lane >= C::kRowChunks;
        const int c = lane % C::kRowChunks;
        const int r = (tl.len - 1) & (kBS - 1);
        uint4 v = na;
        if constexpr (KV == KV_E4M3) v = quant16_e4m3<QT == KV_BF16>(na, nb2, (isv ? p.v_scale : p.k_scale)[tl.h]);
        const uint32_t tbase = smem_u32(my_stages + st * C::kStageBytes) + (isv ? C::kTileBytes : 0);
        const uint32_t a = C::kNBox == 2 ? tbase + (c >> 3) * 2048 + swz128(r, c & 7) : tbase + swz128(r, c);
        sts128(a, v.x, v.y, v.z, v.w);
        fence_proxy_async_smem();                // orders this write before the stage's next TMA fill
        const int64_t row = (int64_t(apb) * Hkv + tl.h) * p.block_size + ((tl.len - 1) & (p.block_size - 1));
        static_cast<uint4*>(isv ? p.v_cache : p.k_cache)[row * C::kRowChunks + c] = v;
      }
      __syncwarp();
    }
    const int nv = ok ? min(kBS, tl.len - tl.b * kBS) : 0;
    if (nv > 0) {
      const uint32_t kbase = smem_u32(my_stages + st * C::kStageBytes);
      const uint32_t vbase = kbase + C::kTileBytes;
      // ---- S^T = K Q^T -------------------------------------------------------------
      float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
      if constexpr (KV == KV_E4M3) {
        uint32_t kr[2][8];
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
          const int row = gq + 8 * rr;
          const uint4 c0 = lds128(kbase + swz128(row, 2 * tq));
          const uint4 c1 = lds128(kbase + swz128(row, 2 * tq + 1));
          kr[rr][0] = c0.x; kr[rr][1] = c0.y; kr[rr][2] = c0.z; kr[rr][3] = c0.w;
          kr[rr][4] = c1.x; kr[rr][5] = c1.y; kr[rr][6] = c1.z; kr[rr][7] = c1.w;
        }
#pragma unroll
        for (int j = 0; j < C::kKSteps; ++j) {
          uint32_t a[4];
          a[0] = e4m3x2_to_f16x2(kr[0][j]);
          a[1] = e4m3x2_to_f16x2(kr[1][j]);
          a[2] = e4m3x2_to_f16x2(kr[0][j] >> 16);
          a[3] = e4m3x2_to_f16x2(kr[1][j] >> 16);
          if (j & 1) mma16816<false>(sb, a, qf[j][0], qf[j][1]);
          else mma16816<false>(sa, a, qf[j][0], qf[j][1]);
        }
      } else {
        const int mi = lane >> 3;
        const int row = (lane & 7) + ((mi & 1) << 3);
#pragma unroll
        for (int j = 0; j < C::kKSteps; ++j) {
          const int chunk = 2 * j + (mi >> 1);
          uint32_t a[4];
          ldsm_x4(kbase + (chunk >> 3) * 2048 + swz128(row, chunk & 7), a[0], a[1], a[2], a[3]);
          if (j & 1) mma16816<C::kBF16>(sb, a, qf[j][0], qf[j][1]);
          else mma16816<C::kBF16>(sa, a, qf[j][0], qf[j][1]);
        }
      }
      // s[0]: (token g, head 2t)  s[1]: (token g, head 2t+1)  s[2]/s[3]: token g + 8.
      float x[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) x[e] = (sa[e] + sb[e]) * sl;
      const bool v0 = gq < nv, v8 = gq + 8 < nv;
      if (!v0) { x[0] = -INFINITY; x[1] = -INFINITY; }
      if (!v8) { x[2] = -INFINITY; x[3] = -INFINITY; }
      // ---- online softmax over the tile's 16 tokens ----------------------------------
      float mx0 = fmaxf(x[0], x[2]), mx1 = fmaxf(x[1], x[3]);
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
      }
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      const bool grew = mn0 > m0 || mn1 > m1;
      const float al0 = fast_exp2(m0 - mn0), al1 = fast_exp2(m1 - mn1);
      m0 = mn0;
      m1 = mn1;
      const float p0 = fast_exp2(x[0] - mn0), p1 = fast_exp2(x[1] - mn1);
      const float p2 = fast_exp2(x[2] - mn0), p3 = fast_exp2(x[3] - mn1);
      l0 = l0 * al0 + p0 + p2;
      l1 = l1 * al1 + p1 + p3;
      if (__any_sync(0xffffffffu, grew)) {     // the running max moved: rescale O
#pragma unroll
        for (int mt = 0; mt < C::kMTiles; ++mt) {
          o[mt][0] *= al0; o[mt][1] *= al1; o[mt][2] *= al0; o[mt][3] *= al1;
        }
      }
      // P^T as the B operand: lane (g, t) needs head g, tokens {2t, 2t+1} and {2t+8, 2t+9}.
      constexpr bool kPB = C::kBF16;
      const uint32_t pb0 = movmatrix_trans(pack2<kPB>(p0, p1));
      const uint32_t pb1 = movmatrix_trans(pack2<kPB>(p2, p3));
      // ---- O^T += V^T P^T -----------------------------------------------------------
      if constexpr (KV == KV_E4M3) {
        uint4 vr[4];   // tokens 2t, 2t+1, 2t+8, 2t+9; bytes 16g .. 16g+15
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int tok = 2 * tq + (k & 1) + 8 * (k >> 1);
          vr[k] = tok < nv ? lds128(vbase + swz128(tok, gq)) : make_uint4(0u, 0u, 0u, 0u);
        }
        const uint32_t x01[4] = {vr[0].x, vr[0].y, vr[0].z, vr[0].w};
        const uint32_t y01[4] = {vr[1].x, vr[1].y, vr[1].z, vr[1].w};
        const uint32_t x89[4] = {vr[2].x, vr[2].y, vr[2].z, vr[2].w};
        const uint32_t y89[4] = {vr[3].x, vr[3].y, vr[3].z, vr[3].w};
#pragma unroll
        for (int mt = 0; mt < C::kMTiles; ++mt) {
          const uint32_t sel = (mt & 1) ? 0x7362u : 0x5140u;
          const uint32_t w01 = prmt(x01[mt >> 1], y01[mt >> 1], sel);
          const uint32_t w89 = prmt(x89[mt >> 1], y89[mt >> 1], sel);
          uint32_t a[4];
          a[0] = e4m3x2_to_f16x2(w01);
          a[1] = e4m3x2_to_f16x2(w01 >> 16);
          a[2] = e4m3x2_to_f16x2(w89);
          a[3] = e4m3x2_to_f16x2(w89 >> 16);
          mma16816<false>(o[mt], a, pb0, pb1);
        }
      } else {
        const int mi = lane >> 3;
        const int row = (lane & 7) + ((mi >> 1) << 3);
        uint32_t m01 = 0xffffffffu, m89 = 0xffffffffu;
        if (nv < kBS) {
          m01 = (2 * tq < nv ? 0x0000ffffu : 0u) | (2 * tq + 1 < nv ? 0xffff0000u : 0u);
          m89 = (2 * tq + 8 < nv ? 0x0000ffffu : 0u) | (2 * tq + 9 < nv ? 0xffff0000u : 0u);
        }
#pragma unroll
        for (int mt = 0; mt < C::kMTiles; ++mt) {
          const int chunk = 2 * mt + (mi & 1);
          uint32_t a[4];
          ldsm_x4_trans(vbase + (chunk >> 3) * 2048 + swz128(row, chunk & 7), a[0], a[1], a[2], a[3]);
          if (nv < kBS) { a[0] &= m01; a[1] &= m01; a[2] &= m89; a[3] &= m89; }
          mma16816<C::kBF16>(o[mt], a, pb0, pb1);
        }
      }
    }

    // Release the stage and refill it with the tile kStages ahead.  Every lane's shared
    // loads of this stage have returned (their values fed the MMAs above), so the TMA
    // write cannot overtake them.
    __syncwarp();
    if (i + kStages < n) {
      issue(pc, i + kStages, st);
      advance(pc);
    }

    const bool piece_end = i == n - 1 || tl.b + 1 == tl.nb;
    if (!piece_end) continue;

    // ---- finish the piece [piece_b0, tl.b] of segment (s, h) -----------------------------
    float ls0 = l0, ls1 = l1;
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      ls0 += __shfl_xor_sync(0xffffffffu, ls0, off);
      ls1 += __shfl_xor_sync(0xffffffffu, ls1, off);
    }
    const float vs = KV == KV_E4M3 ? p.v_scale[tl.h] : 1.f;
    const int h0 = 2 * tq, h1 = 2 * tq + 1;
    const int Hq = Hkv * G;
    const int64_t seg_t0 = int64_t(Hkv) * cum_nb[tl.s] + int64_t(tl.h) * tl.nb;
    const int64_t piece_t0 = seg_t0 + piece_b0;
    // A segment's pieces belong to consecutive workers, one each; the merge kernel works out
    // which from the lengths.  A piece that starts its worker's range goes to the worker's
    // first slot (2w), any other to its second (2w + 1): a range holds at most one piece
    // that starts inside it and runs past its end.
    const bool complete = piece_b0 == 0 && tl.b + 1 == tl.nb;
    if (complete) {
      const float inv0 = ls0 > 0.f ? vs / ls0 : 0.f, inv1 = ls1 > 0.f ? vs / ls1 : 0.f;
      const int64_t base = (int64_t(tl.s) * Hq + int64_t(tl.h) * G) * D;
#pragma unroll
      for (int mt = 0; mt < C::kMTiles; ++mt) {
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const int d = out_dim<KV>(mt, r, gq);
          if (h0 < G) store_out<QT>(p.out, base + int64_t(h0) * D + d, o[mt][2 * r] * inv0);
          if (h1 < G) store_out<QT>(p.out, base + int64_t(h1) * D + d, o[mt][2 * r + 1] * inv1);
        }
      }
      continue;
    }
    // Partial piece: (running max, sum of exponentials, unnormalised output) per head.
    const int64_t slot = 2 * int64_t(w) + (piece_t0 == t_begin ? 0 : 1);
    float* po = p.po + slot * G * D;
#pragma unroll
    for (int mt = 0; mt < C::kMTiles; ++mt) {
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int d = out_dim<KV>(mt, r, gq);
        if (h0 < G) po[h0 * D + d] = o[mt][2 * r] * vs;
        if (h1 < G) po[h1 * D + d] = o[mt][2 * r + 1] * vs;
      }
    }
    if (gq == 0) {
      if (h0 < G) p.ml[slot * G + h0] = make_float2(m0, ls0);
      if (h1 < G) p.ml[slot * G + h1] = make_float2(m1, ls1);
    }
  }
}

struct MergeParams {
  void* out;
  const float2* ml;
  const float* po;
  const int32_t* context_lens;
  int num_seqs;
  int num_kv_heads;
  int num_segments;       // num_seqs * num_kv_heads
  int group;
  int max_len;            // the decode call's length clamp
  int part_blocks;        // the decode call's tiles per partition (0: balanced split)
  int num_workers;        // the decode call's worker warps
};

constexpr int kMergeWarps = 8;

// Split-KV merge: one warp per (segment, query head) whose segment was split.  With
// M = max_k m_k over the pieces k,  out = sum_k 2^(m_k - M) o_k / sum_k 2^(m_k - M) l_k.
// Lane k fetches piece k's (m, l) while every lane fetches its 16-byte chunk of up to
// kChunk pieces' rows; the weights come from warp reductions over the lanes, so the
// loads of a block of 32 pieces overlap and no exponential sits between a load and the sum.
template <int QT, int D>
__global__ void __launch_bounds__(kMergeWarps * 32, 2) split_kv_merge_kernel(const MergeParams p) {
  constexpr int kLanesPerHead = D / 4;       // 16-byte chunks of one head's row
  constexpr int kHP = 32 / kLanesPerHead;    // rows per load instruction of the warp
  constexpr int kChunk = 16;                 // loads in flight per lane
  const int lane = threadIdx.x & 31;
  const int G = p.group;
  const int64_t item = int64_t(blockIdx.x) * kMergeWarps + (threadIdx.x >> 5);
  const bool active = item < int64_t(p.num_segments) * G;
  const int seg = active ? int(item / G) : 0, hh = active ? int(item % G) : 0;

  // The segment's pieces, from the lengths alone and before the wait (so while the decode
  // grid's last CTAs still run).  The decode kernel splits the flattened units (tiles, or
  // partitions of part_blocks tiles) of all (sequence, kv head) segments into num_workers
  // ranges, range w starting at unit floor(w * units / W); the worker of unit u is
  // floor(((u + 1) W - 1) / units).  The segment's pieces belong to workers w0 .. w0 + np - 1;
  // worker w0's piece is in its first slot (2 w0) if the segment starts its range, else in its
  // second (2 w0 + 1), and every later worker's piece is in its first.
  int w0 = 0, np = 0, z = 0;
  if (active) {
    const int S = p.num_seqs, Hkv = p.num_kv_heads, PB = p.part_blocks;
    const int s = seg / Hkv, h = seg - s * Hkv;
    int tot = 0, pre = 0, mine = 0;          // units of all sequences, of those before s, of s
    for (int i = lane; i < S; i += 32) {
      const int nb = (clamp_len(__ldg(p.context_lens + i), p.max_len) + kBS - 1) / kBS;
      const int nu = PB ? (nb + PB - 1) / PB : nb;
      tot += nu;
      if (i < s) pre += nu;
      if (i == s) mine = nu;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      tot += __shfl_xor_sync(0xffffffffu, tot, o);
      pre += __shfl_xor_sync(0xffffffffu, pre, o);
      mine += __shfl_xor_sync(0xffffffffu, mine, o);
    }
    const int64_t units = int64_t(Hkv) * tot;
    const int64_t W = min(int64_t(p.num_workers), units);
    if (mine > 0 && W > 0) {
      const int64_t u0 = int64_t(Hkv) * pre + int64_t(h) * mine, u1 = u0 + mine - 1;
      w0 = int(((u0 + 1) * W - 1) / units);
      np = int(((u1 + 1) * W - 1) / units) - w0 + 1;
      z = int64_t(w0) * units / W == u0 ? 0 : 1;
    }
  }
  griddep_wait();                            // the decode kernel's partials are complete
  griddep_launch_dependents();               // the next kernel may start its own prologue
  if (np <= 1) return;                       // empty, or finished by the decode kernel itself
  auto slot_of = [&](int k) -> int64_t { return k == 0 ? 2 * int64_t(w0) + z : 2 * int64_t(w0 + k); };
  const int rsub = lane / kLanesPerHead, dof = (lane % kLanesPerHead) * 4;
  float M = -INFINITY, den = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int kb = 0; kb < np; kb += 32) {
    const int nb = min(32, np - kb);
    float mk = -INFINITY, lk = 0.f;
    if (lane < nb) {
      const float2 t2 = __ldcg(p.ml + slot_of(kb + lane) * G + hh);   // L2: written by the decode grid
      mk = t2.x;
      lk = t2.y;
    }
    float wk = 0.f;
    for (int r0 = 0; r0 < nb; r0 += kChunk * kHP) {
      float4 v[kChunk];
#pragma unroll
      for (int c = 0; c < kChunk; ++c) {
        const int r = r0 + c * kHP + rsub;
        v[c] = r < nb ? __ldcg(reinterpret_cast<const float4*>(p.po + (slot_of(kb + r) * G + hh) * D + dof))
                      : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      if (r0 == 0) {                         // weights of this block, while its rows arrive
        float mb = mk;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, o));
        const float Mn = fmaxf(M, mb);
        const float Mz = Mn == -INFINITY ? 0.f : Mn;   // every piece so far empty: weights 0
        const float rescale = fast_exp2(M - Mz);       // 0 while M = -inf
        wk = fast_exp2(mk - Mz);
        float lw = lk * wk;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) lw += __shfl_xor_sync(0xffffffffu, lw, o);
        den = den * rescale + lw;
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[e] *= rescale;
        M = Mn;
      }
#pragma unroll
      for (int c = 0; c < kChunk; ++c) {
        const int r = r0 + c * kHP + rsub;
        const float wr = __shfl_sync(0xffffffffu, wk, r & 31);
        if (r < nb) {
          acc[0] += wr * v[c].x;
          acc[1] += wr * v[c].y;
          acc[2] += wr * v[c].z;
          acc[3] += wr * v[c].w;
        }
      }
    }
  }
  if constexpr (kHP > 1) {                   // fold the rows the half-warps took
#pragma unroll
    for (int e = 0; e < 4; ++e) {
#pragma unroll
      for (int o = kLanesPerHead; o < 32; o <<= 1) acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], o);
    }
  }
  if (rsub == 0) {
    const float inv = den > 0.f ? 1.f / den : 0.f;
    const int64_t obase = (int64_t(seg) * G + hh) * D + dof;   // out[s][h * G + hh][:]
#pragma unroll
    for (int e = 0; e < 4; ++e) store_out<QT>(p.out, obase + e, acc[e] * inv);
  }
}

// ---------------------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------------------
struct Layout {
  size_t ml = 0, po = 0, total = 0;
};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

int64_t num_slots(int workers) { return 2 * int64_t(workers); }

Layout layout(int group, int head_dim, int64_t slots) {
  Layout l;
  l.ml = 0;
  l.po = l.ml + align256(sizeof(float2) * size_t(slots) * group);
  l.total = l.po + align256(sizeof(float) * size_t(slots) * group * head_dim);
  return l;
}

// Dynamic shared memory a launch of `kern` may request: the device's per-CTA opt-in limit
// less the kernel's static arrays.
template <typename K>
size_t dynamic_smem_limit(K kern) {
  int dev = 0, optin = 0;
  cudaFuncAttributes fa = {};
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
      cudaFuncGetAttributes(&fa, kern) != cudaSuccess || size_t(optin) <= fa.sharedSizeBytes)
    return 0;
  return size_t(optin) - fa.sharedSizeBytes;
}

template <int KV, int D, int NW, int NS>
size_t smem_bytes(int num_seqs) {
  return 1024 + size_t(NW) * NS * Cfg<KV, D>::kStageBytes + 3 * sizeof(int) * size_t(num_seqs + 1);
}

template <int KV, int QT, int D, int NW, int NS>
pkv_status launch_cfg(DecodeParams prm, const CUtensorMap& tk, const CUtensorMap& tv, int grid,
                      cudaStream_t stream) {
  auto kern = paged_decode_kernel<KV, QT, D, NW, NS>;
  const size_t smem = smem_bytes<KV, D, NW, NS>(prm.num_seqs);
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) != cudaSuccess)
    return PKV_ERR_CUDA;
  prm.num_workers = grid * NW;
  if (launch_pdl(kern, dim3(grid), dim3(NW * 32), smem, stream, tk, tv, prm) != cudaSuccess) return PKV_ERR_CUDA;
  MergeParams mp;
  mp.out = prm.out;
  mp.ml = prm.ml;
  mp.po = prm.po;
  mp.context_lens = prm.context_lens;
  mp.num_seqs = prm.num_seqs;
  mp.num_kv_heads = prm.num_kv_heads;
  mp.num_segments = prm.num_seqs * prm.num_kv_heads;
  mp.group = prm.group;
  mp.max_len = prm.max_len;
  mp.part_blocks = prm.part_blocks;
  mp.num_workers = prm.num_workers;
  const int64_t items = int64_t(mp.num_segments) * mp.group;
  const int mgrid = int((items + kMergeWarps - 1) / kMergeWarps);
  if (launch_pdl(split_kv_merge_kernel<QT, D>, dim3(mgrid), dim3(kMergeWarps * 32), 0, stream, mp) != cudaSuccess)
    return PKV_ERR_CUDA;
  return PKV_OK;
}

// 12 worker warps with 2 stages each when the per-sequence prefix arrays fit next to the
// stages, else 4 warps with 2 stages (very large batches).
template <int KV, int QT, int D>
pkv_status launch(const DecodeParams& prm, const CUtensorMap& tk, const CUtensorMap& tv, int grid,
                  cudaStream_t stream) {
  static thread_local int cached_dev = -1;
  static thread_local size_t lim12 = 0, lim4 = 0;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
  if (dev != cached_dev) {                   // looked up once per device and thread
    lim12 = dynamic_smem_limit(paged_decode_kernel<KV, QT, D, kMaxWarps, 2>);
    lim4 = dynamic_smem_limit(paged_decode_kernel<KV, QT, D, 4, 2>);
    cached_dev = dev;
  }
  if (smem_bytes<KV, D, kMaxWarps, 2>(prm.num_seqs) <= lim12)
    return launch_cfg<KV, QT, D, kMaxWarps, 2>(prm, tk, tv, grid, stream);
  if (smem_bytes<KV, D, 4, 2>(prm.num_seqs) <= lim4) return launch_cfg<KV, QT, D, 4, 2>(prm, tk, tv, grid, stream);
  return PKV_ERR_UNSUPPORTED;
}

// One persistent CTA per SM, or per SM of the budget set with pkv_set_decode_sm_budget.
// The workspace is always sized for the whole device, so any budget fits it.
std::atomic<int> g_sm_budget{0};
int full_grid() { return std::max(1, num_sms()); }
int decode_grid() {
  const int n = full_grid(), b = g_sm_budget.load(std::memory_order_relaxed);
  return b > 0 && b < n ? b : n;
}

}  // namespace
}  // namespace pkv

extern "C" {

size_t pkv_decode_workspace_bytes(int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size,
                                  int max_context_len, int partition_size) {
  using namespace pkv;
  if (num_seqs <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads || (block_size != 16 && block_size != 32) ||
      partition_size < 0 || partition_size % kBS)
    return 0;
  const int group = num_heads / num_kv_heads;
  const int workers = full_grid() * kMaxWarps;
  const int64_t slots = num_slots(workers);
  return layout(group, head_dim, slots).total;
}

pkv_status pkv_set_decode_sm_budget(int num_sms) {
  if (num_sms < 0) return PKV_ERR_INVALID_ARG;
  pkv::g_sm_budget.store(num_sms, std::memory_order_relaxed);
  return PKV_OK;
}

int pkv_get_decode_sm_budget(void) { return pkv::g_sm_budget.load(std::memory_order_relaxed); }

}  // extern "C"

namespace pkv {

// The argument checks shared by every decode entry point.  On PKV_OK, *need holds the
// workspace bytes the call needs (0 when num_seqs == 0: nothing to do).
pkv_status decode_check(const void* out, const void* q, pkv_dtype q_dtype, int num_seqs, int num_heads,
                        const void* k_cache, const void* v_cache, const pkv_cache_desc* cache,
                        const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                        int max_context_len, int partition_size, size_t* need) {
  *need = 0;
  pkv_status st = check_cache_desc(cache);
  if (st != PKV_OK) return st;
  if (num_seqs < 0 || num_heads <= 0 || max_blocks_per_seq < 0 || max_context_len < 0 || partition_size < 0)
    return PKV_ERR_INVALID_ARG;
  if (num_seqs == 0) return PKV_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens) return PKV_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) ||
      (reinterpret_cast<uintptr_t>(block_tables) & 3u) || (reinterpret_cast<uintptr_t>(context_lens) & 3u))
    return PKV_ERR_INVALID_ARG;
  if (num_heads % cache->num_kv_heads) return PKV_ERR_INVALID_ARG;
  if (partition_size % kBS) return PKV_ERR_INVALID_ARG;
  if (max_blocks_per_seq == 0) return PKV_ERR_INVALID_ARG;
  const int group = num_heads / cache->num_kv_heads;
  if ((cache->block_size != 16 && cache->block_size != 32) || group > kMaxGroup) return PKV_ERR_UNSUPPORTED;
  if (q_dtype != PKV_F16 && q_dtype != PKV_BF16) return PKV_ERR_INVALID_ARG;
  const int D = cache->head_dim;
  if (D != 64 && D != 128) return PKV_ERR_UNSUPPORTED;
  if (cache->kv_dtype != PKV_FP8_E4M3 && cache->kv_dtype != q_dtype) return PKV_ERR_UNSUPPORTED;
  if (cache->kv_dtype == PKV_FP8_E4M3 && D != 128) return PKV_ERR_UNSUPPORTED;
  if (int64_t(cache->num_blocks) * cache->num_kv_heads * cache->block_size >= (int64_t(1) << 31))
    return PKV_ERR_UNSUPPORTED;

  // The kernel indexes tiles (16 rows of one kv head) and workers in 32 bits.
  const int64_t max_len = std::min<int64_t>(int64_t(max_blocks_per_seq) * cache->block_size, max_context_len);
  if (int64_t(cache->num_kv_heads) * num_seqs * ((max_len + kBS - 1) / kBS) >= (int64_t(1) << 31))
    return PKV_ERR_UNSUPPORTED;
  const int grid = full_grid();
  if (int64_t(grid) * kMaxWarps >= (int64_t(1) << 16)) return PKV_ERR_UNSUPPORTED;
  *need = layout(group, D, num_slots(grid * kMaxWarps)).total;
  return PKV_OK;
}

namespace {

// Both decode entry points: plain (k_new == v_new == nullptr) or with the fused append.
pkv_status decode_impl(void* out, const void* q, pkv_dtype q_dtype, int num_seqs, int num_heads,
                       const void* k_cache, const void* v_cache, const pkv_cache_desc* cache,
                       const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                       int max_context_len, float scale, int partition_size, void* workspace,
                       size_t workspace_bytes, pkv_stream_t stream, const void* k_new, const void* v_new) {
  size_t need = 0;
  pkv_status st = decode_check(out, q, q_dtype, num_seqs, num_heads, k_cache, v_cache, cache, block_tables,
                               max_blocks_per_seq, context_lens, max_context_len, partition_size, &need);
  if (st != PKV_OK || num_seqs == 0) return st;
  if ((k_new != nullptr) != (v_new != nullptr) || (k_new && (!aligned16(k_new) || !aligned16(v_new))))
    return PKV_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return PKV_ERR_WORKSPACE;
  const int group = num_heads / cache->num_kv_heads;
  const int D = cache->head_dim;
  const int64_t max_len = std::min<int64_t>(int64_t(max_blocks_per_seq) * cache->block_size, max_context_len);
  const int grid = decode_grid();
  const int part_blocks = partition_size / kBS;
  const Layout lay = layout(group, D, num_slots(grid * kMaxWarps));
  unsigned* err = error_word_ptr();
  if (!err) return PKV_ERR_CUDA;

  // Tensor maps: the pool as rows of head_dim elements; a box is one 16-row tile of a (block,
  // kv head).  Rows of 128 bytes are one 2-D box; rows of 256 bytes (2-byte, head_dim 128) are
  // viewed as (64 elements, rows, 2 halves) so one 3-D box lands as two swizzled halves.
  CUtensorMap tk, tv;
  const bool fp8 = cache->kv_dtype == PKV_FP8_E4M3;
  const CUtensorMapDataType dt = fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16;
  const uint64_t rows = uint64_t(cache->num_blocks) * cache->num_kv_heads * cache->block_size;
  const uint64_t row_bytes = uint64_t(D) * dtype_bytes(cache->kv_dtype);
  bool enc;
  if (row_bytes == 256) {
    enc = encode_tmap_3d(&tk, dt, k_cache, 64, rows, 2, 256, 128, 64, kBS, 2, CU_TENSOR_MAP_SWIZZLE_128B) &&
          encode_tmap_3d(&tv, dt, v_cache, 64, rows, 2, 256, 128, 64, kBS, 2, CU_TENSOR_MAP_SWIZZLE_128B);
  } else {
    enc = encode_tmap_2d(&tk, dt, k_cache, D, rows, row_bytes, uint32_t(D), kBS, CU_TENSOR_MAP_SWIZZLE_128B) &&
          encode_tmap_2d(&tv, dt, v_cache, D, rows, row_bytes, uint32_t(D), kBS, CU_TENSOR_MAP_SWIZZLE_128B);
  }
  if (!enc) return PKV_ERR_CUDA;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  DecodeParams prm;
  prm.out = out;
  prm.q = q;
  prm.block_tables = block_tables;
  prm.context_lens = context_lens;
  prm.k_scale = cache->k_scale;
  prm.v_scale = cache->v_scale;
  prm.num_seqs = num_seqs;
  prm.num_kv_heads = cache->num_kv_heads;
  prm.group = group;
  prm.max_blocks = max_blocks_per_seq;
  prm.max_len = int(max_len);
  prm.num_blocks = cache->num_blocks;
  prm.block_size = cache->block_size;
  prm.tile_shift = cache->block_size == 32 ? 1 : 0;
  prm.part_blocks = part_blocks;
  prm.scale_log2 = scale * 1.4426950408889634f;
  prm.ml = reinterpret_cast<float2*>(ws + lay.ml);
  prm.po = reinterpret_cast<float*>(ws + lay.po);
  prm.err = err;
  prm.k_new = k_new;
  prm.v_new = v_new;
  prm.k_cache = const_cast<void*>(k_cache);
  prm.v_cache = const_cast<void*>(v_cache);
  prm.defer_dependents = grid < full_grid() ? 1 : 0;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool qbf = q_dtype == PKV_BF16;
  switch (cache->kv_dtype) {
    case PKV_BF16:
      return D == 128 ? launch<KV_BF16, KV_BF16, 128>(prm, tk, tv, grid, s)
                      : launch<KV_BF16, KV_BF16, 64>(prm, tk, tv, grid, s);
    case PKV_F16:
      return D == 128 ? launch<KV_F16, KV_F16, 128>(prm, tk, tv, grid, s)
                      : launch<KV_F16, KV_F16, 64>(prm, tk, tv, grid, s);
    case PKV_FP8_E4M3:
      return qbf ? launch<KV_E4M3, KV_BF16, 128>(prm, tk, tv, grid, s)
                 : launch<KV_E4M3, KV_F16, 128>(prm, tk, tv, grid, s);
  }
  return PKV_ERR_UNSUPPORTED;
}

}  // namespace
}  // namespace pkv

extern "C" {

pkv_status pkv_paged_decode(void* out, const void* q, pkv_dtype q_dtype, int num_seqs, int num_heads,
                            const void* k_cache, const void* v_cache, const pkv_cache_desc* cache,
                            const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                            int max_context_len, float scale, int partition_size, void* workspace,
                            size_t workspace_bytes, pkv_stream_t stream) {
  return pkv::decode_impl(out, q, q_dtype, num_seqs, num_heads, k_cache, v_cache, cache, block_tables,
                          max_blocks_per_seq, context_lens, max_context_len, scale, partition_size, workspace,
                          workspace_bytes, stream, nullptr, nullptr);
}

pkv_status pkv_paged_decode_append(void* out, const void* q, pkv_dtype q_dtype, int num_seqs, int num_heads,
                                   const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                                   const pkv_cache_desc* cache, const int32_t* block_tables, int max_blocks_per_seq,
                                   const int32_t* context_lens, int max_context_len, float scale,
                                   int partition_size, void* workspace, size_t workspace_bytes,
                                   pkv_stream_t stream) {
  if (num_seqs > 0 && (!k_new || !v_new)) return PKV_ERR_INVALID_ARG;
  return pkv::decode_impl(out, q, q_dtype, num_seqs, num_heads, k_cache, v_cache, cache, block_tables,
                          max_blocks_per_seq, context_lens, max_context_len, scale, partition_size, workspace,
                          workspace_bytes, stream, k_new, v_new);
}

}  // extern "C"
