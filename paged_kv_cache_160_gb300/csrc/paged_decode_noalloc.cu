// pkv_paged_decode_noalloc: paged decode for callers that cannot allocate device memory.
//
// pkv_paged_decode needs a scratch workspace for its split-KV partial results, which the
// caller normally allocates.  Some callers cannot do that at decode time: a plain C host
// with no device allocator of its own, or a serving loop that must not call cudaMalloc
// on its hot path because cudaMalloc can synchronise the whole device and stall every
// stream.  This entry point gives them the same computation with the scratch memory held
// by the library itself, in one fixed-size device array.
#include <mutex>

#include "pkv_host.h"

namespace {

// Upper bound of the scratch this entry point can offer.  Every GPU that loads the library
// keeps this array resident until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(24) << 20;   // 24 MiB

static __device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device, looked up once per device.
// In host code `g_decode_scratch` names a host-side stand-in, never the device memory.
void* scratch_on_current_device() {
  const int dev = pkv::current_device();
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess) return nullptr;
    g_scratch_ptr[dev] = p;
  }
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" {

size_t pkv_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

pkv_status pkv_paged_decode_noalloc(void* out, const void* q, pkv_dtype q_dtype, int num_seqs, int num_heads,
                                    const void* k_cache, const void* v_cache, const pkv_cache_desc* cache,
                                    const int32_t* block_tables, int max_blocks_per_seq,
                                    const int32_t* context_lens, int max_context_len, float scale,
                                    int partition_size, pkv_stream_t stream) {
  // The same argument checks, in the same order, as pkv_paged_decode, so both calls give the
  // same status for the same invalid arguments; only then is the scratch size compared.
  size_t need = 0;
  pkv_status st = pkv::decode_check(out, q, q_dtype, num_seqs, num_heads, k_cache, v_cache, cache, block_tables,
                                    max_blocks_per_seq, context_lens, max_context_len, partition_size, &need);
  if (st != PKV_OK || num_seqs == 0) return st;
  if (need > kNoAllocScratchBytes) return PKV_ERR_WORKSPACE;   // more than the fixed array holds
  void* scratch = scratch_on_current_device();
  if (!scratch) return PKV_ERR_CUDA;
  return pkv_paged_decode(out, q, q_dtype, num_seqs, num_heads, k_cache, v_cache, cache, block_tables,
                          max_blocks_per_seq, context_lens, max_context_len, scale, partition_size, scratch,
                          kNoAllocScratchBytes, stream);
}

}  // extern "C"
