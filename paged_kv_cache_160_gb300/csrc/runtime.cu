// Library runtime: status strings, the device error word, device properties and TMA
// tensor-map encoding through the driver entry point (no link-time libcuda dependency,
// so the library also loads on machines without a GPU driver).
#include <mutex>

#include "pkv_device.cuh"
#include "pkv_host.h"

namespace {

// Bits set by kernels for data-dependent faults the host cannot check (bad block ids,
// slots, context lengths, copy pairs, timed-out waits).  One word per device.
__device__ unsigned g_pkv_error_word = 0;

constexpr int kMaxDevices = 64;

struct DeviceCache {
  unsigned* err = nullptr;
  int sms = 0;
};
DeviceCache g_dev[kMaxDevices];
std::mutex g_mu;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<EncodeTiledFn>(nullptr);
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

}  // namespace

namespace pkv {

int current_device() {
  int d = -1;
  if (cudaGetDevice(&d) != cudaSuccess) return -1;
  return d;
}

unsigned* error_word_ptr() {
  int d = current_device();
  if (d < 0 || d >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_dev[d].err) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_pkv_error_word) != cudaSuccess) return nullptr;
    g_dev[d].err = static_cast<unsigned*>(p);
  }
  return g_dev[d].err;
}

bool on_current_device(const void* p) {
  const int d = current_device();
  if (d < 0 || !p) return false;
  cudaPointerAttributes a = {};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeDevice && a.device == d;
}

int num_sms() {
  int d = current_device();
  if (d < 0 || d >= kMaxDevices) return 0;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_dev[d].sms) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, d) != cudaSuccess) return 0;
    g_dev[d].sms = v;
  }
  return g_dev[d].sms;
}

bool encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t dim0, uint64_t dim1,
                    uint64_t stride1_bytes, uint32_t box0, uint32_t box1, CUtensorMapSwizzle swizzle) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {dim0, dim1};
  cuuint64_t strides[1] = {stride1_bytes};
  cuuint32_t box[2] = {box0, box1};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_tmap_3d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t dim0, uint64_t dim1,
                    uint64_t dim2, uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box0, uint32_t box1,
                    uint32_t box2, CUtensorMapSwizzle swizzle) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {dim0, dim1, dim2};
  cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
  cuuint32_t box[3] = {box0, box1, box2};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, dtype, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

pkv_status check_cache_desc(const pkv_cache_desc* c) {
  if (!c) return PKV_ERR_INVALID_ARG;
  if (c->num_blocks <= 0 || c->num_kv_heads <= 0 || c->block_size <= 0 || c->head_dim <= 0)
    return PKV_ERR_INVALID_ARG;
  if (c->kv_dtype != PKV_F16 && c->kv_dtype != PKV_BF16 && c->kv_dtype != PKV_FP8_E4M3) return PKV_ERR_INVALID_ARG;
  if (c->kv_dtype == PKV_FP8_E4M3 && (!c->k_scale || !c->v_scale)) return PKV_ERR_INVALID_ARG;
  if (int64_t(c->head_dim) * dtype_bytes(c->kv_dtype) % 16 != 0) return PKV_ERR_INVALID_ARG;
  return PKV_OK;
}

}  // namespace pkv

extern "C" {

const char* pkv_status_string(pkv_status s) {
  switch (s) {
    case PKV_OK: return "ok";
    case PKV_ERR_INVALID_ARG: return "invalid argument";
    case PKV_ERR_UNSUPPORTED: return "unsupported configuration";
    case PKV_ERR_WORKSPACE: return "workspace missing or too small";
    case PKV_ERR_CUDA: return "CUDA error";
    case PKV_ERR_NO_BLOCKS: return "no free blocks";
    case PKV_ERR_DEVICE_CHECK: return "device-side check failed";
  }
  return "unknown status";
}

int pkv_version(void) { return (0 << 16) | 2; }

pkv_status pkv_get_device_error(int* code, pkv_stream_t stream) {
  if (!code) return PKV_ERR_INVALID_ARG;
  unsigned* p = pkv::error_word_ptr();
  if (!p) return PKV_ERR_CUDA;
  unsigned v = 0;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return PKV_ERR_CUDA;
  if (cudaMemcpy(&v, p, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return PKV_ERR_CUDA;
  if (v) {
    unsigned zero = 0;
    if (cudaMemcpy(p, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return PKV_ERR_CUDA;
  }
  *code = int(v);
  return v ? PKV_ERR_DEVICE_CHECK : PKV_OK;
}

}  // extern "C"

namespace {

// One warp waits on an mbarrier that nothing arrives on, with the bounded wait every kernel
// of the library uses; when the limit passes it reports PKV_DEVERR_TIMEOUT and returns.
__global__ void bounded_wait_check_kernel(uint64_t limit_ns, unsigned* err) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    pkv::mbar_init(&bar, 1);
    pkv::fence_mbar_init();
  }
  __syncthreads();
  const bool done = pkv::mbar_wait(&bar, 0, limit_ns);
  if (!done && threadIdx.x == 0) pkv::set_error(err, PKV_DEVERR_TIMEOUT);
}

}  // namespace

extern "C" pkv_status pkv_check_bounded_wait(uint64_t limit_ns, pkv_stream_t stream) {
  if (limit_ns == 0 || limit_ns > pkv::kWaitLimitNs) return PKV_ERR_INVALID_ARG;
  unsigned* err = pkv::error_word_ptr();
  if (!err) return PKV_ERR_CUDA;
  bounded_wait_check_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(limit_ns, err);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}
