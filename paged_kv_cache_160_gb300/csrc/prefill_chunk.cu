// placeholder until the tcgen05 prefill kernel lands
#include "pkv_host.h"
extern "C" pkv_status pkv_paged_prefill_chunk(void*, const void*, pkv_dtype, const int32_t*, const int32_t*, int, int,
                                              int, int, const void*, const void*, const pkv_cache_desc*,
                                              const int32_t*, int, float, pkv_stream_t) {
  return PKV_ERR_UNSUPPORTED;
}
