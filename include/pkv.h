/*
 * pkv.h — C ABI of libpkv: attention over a paged KV cache on GB300 (sm_103a).
 *
 * The method: a sequence's K/V rows live in fixed-size physical blocks of one pool
 * tensor, found through a per-sequence block table (logical block -> physical block),
 * as in "Lecture 33 — KV Cache management: PagedAttention, Continuous Batching,
 * Chunked Prefill", §2.2; attention kernels read the blocks in place (§2.3); shared
 * blocks are split by copy-on-write (§2.4); a prefill chunk attends its cached
 * history causally (§4.2).  The host block manager follows "PagedAttention: manage
 * the KV cache like virtual memory", §3.2–§3.3.
 *
 * Conventions for every device call below
 *   - Pointers marked (device) are device pointers owned by the caller; the library
 *     never allocates, frees or retains them.  All tensors are dense, row-major, with
 *     the layouts given per argument, and 16-byte aligned.
 *   - Work is enqueued asynchronously on `stream` (NULL = legacy default stream).
 *     Argument checks run on the host before anything is enqueued; a failed check
 *     returns PKV_ERR_INVALID_ARG / PKV_ERR_UNSUPPORTED and enqueues nothing.
 *     A launch failure returns PKV_ERR_CUDA.
 *   - Data-dependent faults the host cannot see (a block id outside the pool, a slot
 *     outside the pool, a context_len beyond the block table, a copy pair that chains)
 *     never fault the GPU: the kernel skips the access and sets a bit in the library's
 *     device error word, read with pkv_get_device_error().
 *   - No call aborts, traps, prints or spins without bound.
 *
 * KV cache layout (both K and V): [num_blocks][num_kv_heads][block_size][head_dim]
 * of kv_dtype.  Slot s addresses token row s % block_size of physical block
 * s / block_size (Lecture 33 §2.2: base + block * block_stride + offset * token_stride).
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PKV_API __attribute__((visibility("default")))
#else
#define PKV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* pkv_stream_t;

typedef enum {
  PKV_OK = 0,
  PKV_ERR_INVALID_ARG = 1,   /* a host-visible argument is out of range / misaligned */
  PKV_ERR_UNSUPPORTED = 2,   /* valid, but the library has no kernel for it (e.g. head_dim 96) */
  PKV_ERR_WORKSPACE = 3,     /* workspace missing or smaller than pkv_decode_workspace_bytes() */
  PKV_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed */
  PKV_ERR_NO_BLOCKS = 5,     /* block manager: the free-block queue cannot cover the request */
  PKV_ERR_DEVICE_CHECK = 6   /* pkv_get_device_error() found a device-side check bit set */
} pkv_status;

typedef enum {
  PKV_F16 = 0,
  PKV_BF16 = 1,
  PKV_FP8_E4M3 = 2           /* e4m3 "fn": bias 7, max 448, no inf; value = code * scale[kv_head] */
} pkv_dtype;

/* Device error word bits (pkv_get_device_error). */
enum {
  PKV_DEVERR_BLOCK_ID = 1u << 0,      /* a block table entry was outside [0, num_blocks) */
  PKV_DEVERR_CONTEXT_LEN = 1u << 1,   /* context_len < 0, > max_blocks_per_seq * block_size or > max_context_len */
  PKV_DEVERR_SLOT = 1u << 2,          /* a slot was >= num_blocks * block_size */
  PKV_DEVERR_COPY_PAIR = 1u << 3,     /* a copy pair was out of range or its dst is also a src */
  PKV_DEVERR_TIMEOUT = 1u << 4,       /* a bounded wait on an async copy / MMA gave up */
  PKV_DEVERR_CHUNK = 1u << 5          /* a prefill chunk's cu_q_lens / q_start_pos were inconsistent */
};

/* The paged pool (Lecture 33 §2.2, "physical KV block pool"): K and V are two such tensors. */
typedef struct {
  int num_blocks;            /* physical blocks in the pool */
  int num_kv_heads;
  int block_size;            /* tokens per block: 16, or 32 (the attention kernels read it as two 16-row tiles) */
  int head_dim;              /* 64 or 128 */
  pkv_dtype kv_dtype;
  const float* k_scale;      /* (device) [num_kv_heads] fp32, e4m3 caches only, else NULL */
  const float* v_scale;      /* (device) [num_kv_heads] fp32, e4m3 caches only, else NULL */
} pkv_cache_desc;

PKV_API const char* pkv_status_string(pkv_status s);
PKV_API int pkv_version(void);       /* (major << 16) | minor */

/*
 * kv_write ("reshape_and_cache").  "PagedAttention: manage the KV cache like virtual
 * memory" §3.3: each new token fills its sequence's current last block; Lecture 33
 * §4.2: a prefill chunk's K/V is written into the cache too.
 *   k_new, v_new   (device) [num_tokens][num_kv_heads][head_dim] of in_dtype
 *   slot_mapping   (device) int64 [num_tokens]; slot < 0 = padding token, skipped
 *   k_cache/v_cache (device) pool tensors described by `cache`
 * For every token t with slot s >= 0 and every kv head h:
 *   k_cache[s / B][h][s % B][:] = k_new[t][h][:]   (same for V)
 * in_dtype == kv_dtype copies bytes.  in_dtype f16/bf16 into an e4m3 cache quantises
 * x / scale[h] (fp32 divide) to e4m3, round-to-nearest-even, saturating at ±448.
 * Slots that repeat within one call: one of the writers wins (unspecified which).
 * Launch order (kv_write and copy_blocks alike): launched as a programmatic dependent of
 * the previous kernel on `stream`; the kernel touches no memory before that kernel has
 * completed, so stream order holds as for a plain launch.
 */
PKV_API pkv_status pkv_kv_write(const void* k_new, const void* v_new, pkv_dtype in_dtype, int num_tokens,
                        const int64_t* slot_mapping, void* k_cache, void* v_cache,
                        const pkv_cache_desc* cache, pkv_stream_t stream);

/*
 * copy_blocks: the copy step of copy-on-write (Lecture 33 §2.4: the writer gets a new
 * block holding a copy of the shared block).
 *   block_pairs (device) int32 [num_pairs][2] = (src, dst)
 * For each pair, the whole block dst of K and of V (all kv heads, all rows) becomes a
 * copy of block src.  No dst may also appear as a src or twice as a dst (the result
 * would depend on order): such pairs, and ids outside the pool, are skipped and flagged
 * PKV_DEVERR_COPY_PAIR.
 */
PKV_API pkv_status pkv_copy_blocks(void* k_cache, void* v_cache, const pkv_cache_desc* cache,
                           const int32_t* block_pairs, int num_pairs, pkv_stream_t stream);

/*
 * swap_blocks: preemption by swapping ("Lecture 33 — KV Cache management" §5.2: the
 * victim's blocks are copied to host RAM, its device blocks are released, and later the
 * blocks are copied back so the sequence can resume).  Block copies between two pools of
 * the same block layout: num_kv_heads, block_size, head_dim and kv_dtype come from `layout`
 * (its num_blocks is not used).  Either pool may be pinned host memory (cudaHostAlloc /
 * cudaHostRegister), passed by its device-visible address (with unified addressing, the
 * host pointer itself).
 *   dst_k/dst_v, src_k/src_v  [num_blocks][num_kv_heads][block_size][head_dim] each
 *   dst_num_blocks, src_num_blocks  pool sizes in blocks (ids are checked against them)
 *   block_pairs (device) int32 [num_pairs][2] = (src block, dst block)
 * For each pair, block dst of dst_k (and dst_v) becomes a copy of block src of src_k
 * (src_v).  Pairs with an id outside its pool, or whose dst another pair also names, are
 * skipped and flagged PKV_DEVERR_COPY_PAIR.  pkv_bm_swap_out / pkv_bm_swap_in produce the
 * pairs.  Launched like kv_write (programmatic dependent, waits before touching memory).
 */
PKV_API pkv_status pkv_swap_blocks(void* dst_k, void* dst_v, int dst_num_blocks, const void* src_k,
                                   const void* src_v, int src_num_blocks, const pkv_cache_desc* layout,
                                   const int32_t* block_pairs, int num_pairs, pkv_stream_t stream);

/*
 * Workspace bytes pkv_paged_decode needs on the current device: two partial-result
 * slots per worker warp (running max, sum of exponentials and unnormalised output per
 * query head).  It depends on the device's SM count and the group size, not on the number
 * of sequences or the context lengths.  The workspace needs no initialisation; each call
 * rewrites what it reads.  Calls that share a workspace must not overlap.
 */
PKV_API size_t pkv_decode_workspace_bytes(int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                  int block_size, int max_context_len, int partition_size);

/*
 * paged_decode: one query token per running sequence (Lecture 33 §2.3).  For sequence
 * i, query head h and kv head g = h / (num_heads / num_kv_heads), with L = context_lens[i]:
 *   s_j = scale * q[i][h] . K_i[j]  for j < L, where K_i[j] = k_cache[T_i[j / B]][g][j % B]
 *   out[i][h] = sum_j softmax(s)_j V_i[j]                         (zeros when L == 0)
 * with T_i = block_tables[i].  Split-KV: the (sequence, kv head, block) tiles are cut into
 * one contiguous range per worker warp — at any block (partition_size = 0, "balanced")
 * or only at multiples of partition_size tokens.  A worker runs an online softmax over
 * its range (consecutive partitions merge in registers); pieces of one sequence held by
 * different workers are merged by log-sum-exp in a second kernel on the same stream,
 * launched as a programmatic dependent of the first.  fp32 accumulation.
 *   out            (device) [num_seqs][num_heads][head_dim] of q_dtype
 *   q              (device) [num_seqs][num_heads][head_dim] of q_dtype (f16 or bf16)
 *   block_tables   (device) int32 [num_seqs][max_blocks_per_seq]
 *   context_lens   (device) int32 [num_seqs]; tokens to attend, including any token
 *                  written this step
 *   max_context_len host upper bound of context_lens; larger lengths are clamped to it
 *                  (and to max_blocks_per_seq * block_size) and flagged PKV_DEVERR_CONTEXT_LEN
 *   partition_size  0 = balanced split; else split granularity in tokens (multiple of 16)
 *   workspace       (device) >= pkv_decode_workspace_bytes(...) bytes
 * out, q, block_tables and context_lens may instead be pinned host memory (cudaHostAlloc /
 * cudaHostRegister, reachable through unified addressing): the kernels then read and write
 * them in place over the host link, so a serving loop needs no separate copies.  The caches
 * and the workspace must be device memory.
 * Supported: kv f16/bf16 with the same q dtype, or e4m3 kv with f16/bf16 q (the e4m3
 * path computes in fp16, so |q| must stay below 65504); head_dim 64/128; block_size 16 or 32;
 * num_heads / num_kv_heads in 1..8; num_kv_heads * num_seqs * ceil(L_max / 16) < 2^31, where
 * L_max = min(max_context_len, max_blocks_per_seq * block_size) (else PKV_ERR_UNSUPPORTED).
 * Launch order: the decode kernel is launched as a programmatic dependent of the previous
 * kernel on `stream`.  If that kernel allows early dependent launch (pkv_kv_write does), the
 * decode kernel may already read context_lens and block_tables while it still runs; q, the
 * caches, out and the workspace are touched only after it has completed.  So the kernel
 * right before a decode call must not write context_lens or block_tables unless it leaves
 * dependent launch at its default (wait for completion).
 */
PKV_API pkv_status pkv_paged_decode(void* out, const void* q, pkv_dtype q_dtype, int num_seqs, int num_heads,
                            const void* k_cache, const void* v_cache, const pkv_cache_desc* cache,
                            const int32_t* block_tables, int max_blocks_per_seq,
                            const int32_t* context_lens, int max_context_len, float scale,
                            int partition_size, void* workspace, size_t workspace_bytes,
                            pkv_stream_t stream);

/*
 * paged_decode_append: pkv_kv_write of one new token per sequence fused into
 * pkv_paged_decode (PagedAttention §3.3: each new token fills its sequence's last block).
 * For every sequence i with L = context_lens[i] >= 1, the new rows k_new[i] and v_new[i] are
 * stored at position L - 1, i.e. slot block_tables[i][(L - 1) / B] * B + (L - 1) % B, quantised
 * to e4m3 with k_scale / v_scale for an e4m3 cache exactly as pkv_kv_write does, and the decode
 * then attends positions 0 .. L - 1, the new one included.  Caches and out are bit-identical to
 * pkv_kv_write (with those slots) followed by pkv_paged_decode.
 *   k_new, v_new  (device, or pinned host memory as for q) [num_seqs][num_kv_heads][head_dim]
 *                 of q_dtype, 16-byte aligned
 *   k_cache, v_cache  (device) written at those positions only
 * Sequences with L == 0 write nothing.  A length above the clamp bound (see pkv_paged_decode)
 * writes nothing and is flagged PKV_DEVERR_CONTEXT_LEN; a block id outside the pool writes
 * nothing and is flagged PKV_DEVERR_BLOCK_ID.  The written block must not be shared with
 * another sequence of the call (copy-on-write has run), as for pkv_kv_write.  Other
 * arguments, limits, launch order and results as pkv_paged_decode.
 */
PKV_API pkv_status pkv_paged_decode_append(void* out, const void* q, pkv_dtype q_dtype, int num_seqs,
                                   int num_heads, const void* k_new, const void* v_new, void* k_cache,
                                   void* v_cache, const pkv_cache_desc* cache, const int32_t* block_tables,
                                   int max_blocks_per_seq, const int32_t* context_lens,
                                   int max_context_len, float scale, int partition_size, void* workspace,
                                   size_t workspace_bytes, pkv_stream_t stream);

/*
 * paged_decode for callers that cannot allocate device memory.  The pages have no
 * counterpart to this entry point; it exists for callers that must not allocate at decode
 * time: a plain C host without a device allocator of its own for scratch space, or a
 * serving loop that may not call cudaMalloc on its hot path because cudaMalloc can
 * synchronise the whole device.  Same arguments and results as pkv_paged_decode, minus the
 * workspace: the library keeps one fixed scratch array of pkv_noalloc_scratch_bytes()
 * (24 MiB) on every device that loads it, resident until the process exits.  Arguments are
 * checked exactly as pkv_paged_decode checks them, in the same order, so an invalid call
 * returns the same status from both entry points.  The scratch a call needs (per
 * pkv_decode_workspace_bytes) depends on the SM count, the group size and head_dim only;
 * 24 MiB holds every supported call on a device of up to 252 SMs.  A valid call that needs
 * more than the array holds returns PKV_ERR_WORKSPACE and enqueues nothing.  No call allocates, frees or clears device memory: each call
 * rewrites the parts of the array it later reads, so leftovers of earlier calls do no
 * harm.  The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call before any
 * stream capture.  Every call on a device shares the one array, so calls whose kernels
 * may overlap on the GPU (different streams with no ordering between them) race and
 * corrupt each other's results: keep them on one stream or order them with events.
 */
PKV_API size_t pkv_noalloc_scratch_bytes(void);
PKV_API pkv_status pkv_paged_decode_noalloc(void* out, const void* q, pkv_dtype q_dtype, int num_seqs,
                                            int num_heads, const void* k_cache, const void* v_cache,
                                            const pkv_cache_desc* cache, const int32_t* block_tables,
                                            int max_blocks_per_seq, const int32_t* context_lens,
                                            int max_context_len, float scale, int partition_size,
                                            pkv_stream_t stream);

/*
 * SM budget of the decode calls (pkv_paged_decode, _append, _noalloc).  The decode runs one
 * persistent CTA per SM.  A budget n in 1 .. (SM count - 1) launches n CTAs instead, splitting
 * the same work over fewer worker warps and leaving the other SMs to a kernel that runs
 * beside it on another stream.  The use case is a chunk's tensor-bound prefill beside the
 * step's HBM-bound decodes (Lecture 33 §4.2 batches the two in one step).  Under a budget the
 * merge kernel launches when the decode grid has finished, not while it runs, so that its
 * waiting CTAs do not hold those SMs.
 *   num_sms  0 (the default) or >= the SM count: every SM.  Negative: PKV_ERR_INVALID_ARG,
 *            the budget is unchanged.
 * Results stay within the decode tolerances for any budget.  The split over workers
 * changes, so fp32 sums are rounded in another order, and outputs are not bit-identical
 * across budgets.  The setting is process-wide and applies to decode calls made after it,
 * on every device and thread.  A captured graph keeps the grid of the call it captured.
 * pkv_decode_workspace_bytes does not depend on the budget: it always sizes for every SM.
 */
PKV_API pkv_status pkv_set_decode_sm_budget(int num_sms);
PKV_API int pkv_get_decode_sm_budget(void);

/*
 * paged_prefill_chunk: causal attention of prefill chunks over their paged history
 * (Lecture 33 §4.2: a chunk attends the earlier chunks' cached KV, masked causally).
 * Chunk c holds query rows cu_q_lens[c] .. cu_q_lens[c+1]-1; row r of the chunk is at
 * absolute position p = q_start_pos[c] + r of sequence c and attends that sequence's
 * keys 0..p (its cached history and itself).  The chunk's own K/V must already be in the
 * cache (pkv_kv_write first).
 *   out, q        (device) [total_q][num_heads][head_dim] of q_dtype (bf16 or f16; same as kv)
 *   cu_q_lens     (device) int32 [num_chunks + 1], cu_q_lens[0] = 0, cu_q_lens[num_chunks] = total_q
 *   q_start_pos   (device) int32 [num_chunks]
 *   block_tables  (device) int32 [num_chunks][max_blocks_per_seq]
 *   max_q_len     host upper bound of the chunks' lengths (sizes the grid); a longer chunk
 *                 sets PKV_DEVERR_CHUNK and its rows past max_q_len stay unwritten
 * Supported: f16/bf16 cache with the same q dtype, head_dim 128, block_size 16 or 32,
 * num_heads a multiple of num_kv_heads (any group size).  Tensor cores (tcgen05, TMEM
 * accumulators), K/V tiles fetched by TMA straight from the physical blocks; with two or
 * more query heads per kv head they are multicast to the two CTAs of a cluster that read
 * the same keys.  q, k_cache and v_cache must be device memory of
 * the current GPU (checked with cudaPointerGetAttributes before anything is enqueued):
 * host, managed or another GPU's memory returns PKV_ERR_INVALID_ARG.
 * Launch order: launched as a programmatic dependent of the previous kernel on `stream`.
 * Only the kernel's own shared-memory and tensor-memory set-up runs before that kernel has
 * completed; no argument is read and no memory touched earlier, so stream order holds as
 * for a plain launch.
 */
PKV_API pkv_status pkv_paged_prefill_chunk(void* out, const void* q, pkv_dtype q_dtype,
                                   const int32_t* cu_q_lens, const int32_t* q_start_pos,
                                   int num_chunks, int total_q, int max_q_len, int num_heads,
                                   const void* k_cache, const void* v_cache, const pkv_cache_desc* cache,
                                   const int32_t* block_tables, int max_blocks_per_seq, float scale,
                                   pkv_stream_t stream);

/*
 * Waits for `stream`, then reads and clears the library's device error word on the
 * current device.  *code receives the PKV_DEVERR_* bits (0 = clean).  Returns
 * PKV_ERR_DEVICE_CHECK when any bit was set, PKV_OK otherwise.
 */
PKV_API pkv_status pkv_get_device_error(int* code, pkv_stream_t stream);

/*
 * Measurement aid, not part of the method: reads the num_tiles K/V tiles whose first pool
 * rows are tile_rows[i] (16 rows of one (block, kv head), in K and in V) with the memory
 * pipeline pkv_paged_decode uses (persistent grid, 12 warps per SM, two stages of one K and
 * one V tile per warp, bulk asynchronous copies) and computes nothing but a checksum, XORed
 * into *checksum.  Timed on the tiles of a decode call, it is the memory ceiling of that
 * call.  Rows outside the pool are skipped and flagged PKV_DEVERR_BLOCK_ID.
 *   tile_rows (device) int32 [num_tiles]; checksum (device) one uint32
 */
PKV_API pkv_status pkv_stream_tiles(const void* k_cache, const void* v_cache, const pkv_cache_desc* cache,
                                    const int32_t* tile_rows, int num_tiles, unsigned* checksum,
                                    pkv_stream_t stream);

/*
 * Diagnostic of the failure path every kernel shares: one warp waits on an mbarrier that
 * nothing arrives on, with the same bounded wait the kernels use, for limit_ns (0 < limit_ns
 * <= 1 s), then sets PKV_DEVERR_TIMEOUT and returns.  Nothing faults or hangs; the context
 * stays usable.  Read the bit with pkv_get_device_error.
 */
PKV_API pkv_status pkv_check_bounded_wait(uint64_t limit_ns, pkv_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * Host block manager ("PagedAttention: manage the KV cache like virtual memory" §3.2–§3.3;
 * Lecture 33 §2.2, §2.4).  A FIFO free-block queue (allocate pops the head, free pushes
 * the tail), a ref_cnt per block, and one block table per sequence.  It produces the
 * block tables, context lengths, slot mappings and copy-on-write pairs the device calls
 * consume.  Host memory only; not thread-safe (one manager per scheduler thread).
 * Every call that fails leaves the manager unchanged.
 * ------------------------------------------------------------------------------------- */
typedef struct pkv_block_manager pkv_block_manager;

/* A pool of num_blocks blocks of block_size tokens; the free queue starts as 0..num_blocks-1. */
PKV_API pkv_status pkv_bm_create(int num_blocks, int block_size, pkv_block_manager** out);
PKV_API void pkv_bm_destroy(pkv_block_manager* bm);

/* Claim the listed blocks for a new sequence holding n_tokens tokens (n_blocks must equal
 * ceil(n_tokens / block_size)); each block's ref_cnt rises by one and a free block leaves
 * the free queue.  Used to set up states such as shared prefixes. */
PKV_API pkv_status pkv_bm_import_seq(pkv_block_manager* bm, int64_t seq, const int32_t* blocks,
                             int n_blocks, int n_tokens);

/* Admit a sequence with an n_tokens prompt: pop ceil(n_tokens / block_size) blocks. */
PKV_API pkv_status pkv_bm_allocate(pkv_block_manager* bm, int64_t seq, int n_tokens);

/* Reserve the slot of the sequence's next token.  If the token starts a new block, one
 * block is popped.  If it lands in a block whose ref_cnt > 1, copy-on-write: a new block
 * is popped, (*cow_src, *cow_dst) = (old, new), the table points at the new block and the
 * old block's ref_cnt drops by one; otherwise both are set to -1. */
PKV_API pkv_status pkv_bm_append_slot(pkv_block_manager* bm, int64_t seq, int64_t* slot,
                              int32_t* cow_src, int32_t* cow_dst);

/* One decode step for a batch: append_slot for seqs[0..n) in order, then export.
 *   slot_mapping  int64 [n]; cow_pairs int32 [n][2] (first *n_cow rows used)
 *   tables        int32 [n][max_blocks] padded with -1; lens int32 [n] (after the step)
 * Fails with PKV_ERR_NO_BLOCKS, changing nothing, if the free queue cannot cover it. */
PKV_API pkv_status pkv_bm_step_decode(pkv_block_manager* bm, const int64_t* seqs, int n, int max_blocks,
                              int64_t* slot_mapping, int32_t* cow_pairs, int* n_cow,
                              int32_t* tables, int32_t* lens);

/* Reserve n consecutive slots (a prefill chunk); slots int64 [n], cow_pairs int32 [n][2]. */
PKV_API pkv_status pkv_bm_append_slots(pkv_block_manager* bm, int64_t seq, int n, int64_t* slots,
                               int32_t* cow_pairs, int* n_cow);

/* child's table becomes a copy of parent's; every block's ref_cnt rises by one. */
PKV_API pkv_status pkv_bm_fork(pkv_block_manager* bm, int64_t parent, int64_t child);

/* Drop the sequence: each block's ref_cnt falls by one; blocks reaching 0 go to the
 * tail of the free queue, in table order. */
PKV_API pkv_status pkv_bm_free(pkv_block_manager* bm, int64_t seq);

/* tables int32 [n][max_blocks] (padded with -1), lens int32 [n]. */
PKV_API pkv_status pkv_bm_export(const pkv_block_manager* bm, const int64_t* seqs, int n, int max_blocks,
                         int32_t* tables, int32_t* lens);

/* Prefix caching ("PagedAttention: manage the KV cache like virtual memory" §3.4–§3.5;
 * Lecture 33 §6.2–§6.3).  A full block is named by h_i = FNV-1a-64(h_{i-1} as 8 bytes
 * little-endian, then its block_size token ids as 4 bytes little-endian each), with h_{-1} =
 * the FNV offset basis 0xcbf29ce484222325, so equal hashes mean equal prefixes.  Admission of
 * a prompt matches its full blocks in order against the cached hashes and stops at the first
 * miss; each hit is "touched" (ref_cnt + 1, and a block nobody held is unlinked from the
 * middle of the free queue in O(1)).  The remaining blocks are popped from the free queue's
 * head, and the new full blocks are registered under their hashes.  *n_cached_tokens = hits x
 * block_size: those tokens' K/V are already in the pool and need no prefill; the others'
 * K/V become valid once the caller's prefill for this sequence has run.  Freed blocks keep
 * their hash (cached and free) until popped for new contents, which drops the hash.  Blocks
 * that fill up during decode are not registered (the manager does not see token ids there).
 * PKV_ERR_NO_BLOCKS, changing nothing, if the misses need more blocks than are free once the
 * hit blocks leave the queue. */
PKV_API pkv_status pkv_bm_allocate_cached(pkv_block_manager* bm, int64_t seq, const int32_t* tokens, int n_tokens,
                                          int* n_cached_tokens);
/* 1 and *hash = the block's registered hash; 0 if it has none; -1 on bad arguments. */
PKV_API int pkv_bm_block_hash(const pkv_block_manager* bm, int block, uint64_t* hash);
PKV_API int pkv_bm_num_cached(const pkv_block_manager* bm);   /* registered hashes */

/* Preemption by swapping ("Lecture 33 — KV Cache management" §5.2).  The host pool is a
 * second set of num_host_blocks blocks (ids 0..num_host_blocks-1 of a caller-owned pinned
 * buffer with the device pool's block layout) with its own FIFO free queue.  Resizing is
 * allowed only while no sequence is swapped out; the queue restarts as 0..n-1. */
PKV_API pkv_status pkv_bm_set_host_pool(pkv_block_manager* bm, int num_host_blocks);

/* Swap a resident sequence out: for each table entry in order a host block is popped and
 * pairs[i] = (device block, host block); then the device blocks are released in table order
 * (ref_cnt - 1, free at 0), as by pkv_bm_free.  A block shared with another sequence stays on
 * the device for it; this sequence takes its own host copy.  Until swapped in, the sequence
 * can only be freed or swapped in (other calls on it return PKV_ERR_INVALID_ARG).
 *   pairs int32 [max_pairs][2]; *n_pairs = number of table entries.
 * PKV_ERR_NO_BLOCKS, changing nothing, if the host queue holds fewer blocks than the table. */
PKV_API pkv_status pkv_bm_swap_out(pkv_block_manager* bm, int64_t seq, int32_t* pairs, int max_pairs,
                                   int* n_pairs);

/* Swap a sequence back in: for each host block in table order a device block is popped and
 * pairs[i] = (host block, device block); the host blocks return to the host queue's tail in
 * table order.  PKV_ERR_NO_BLOCKS, changing nothing, if too few device blocks are free. */
PKV_API pkv_status pkv_bm_swap_in(pkv_block_manager* bm, int64_t seq, int32_t* pairs, int max_pairs,
                                  int* n_pairs);
PKV_API int pkv_bm_num_free_host(const pkv_block_manager* bm);
PKV_API int pkv_bm_is_swapped(const pkv_block_manager* bm, int64_t seq);   /* 1, 0, or -1 if unknown */

PKV_API int pkv_bm_ref_cnt(const pkv_block_manager* bm, int block);      /* -1 if out of range */
PKV_API int pkv_bm_num_free(const pkv_block_manager* bm);
/* The free queue from head to tail into out[0..max_n); returns the queue length. */
PKV_API int pkv_bm_free_queue(const pkv_block_manager* bm, int32_t* out, int max_n);

#ifdef __cplusplus
}
#endif
#endif /* PKV_H_ */
