// Entry points whose kernels are not built yet: they validate nothing and
// report TS_ERR_UNSUPPORTED so callers fail loudly instead of silently.
#include "ts_common.cuh"

extern "C" size_t ts_mla_workspace_size(int32_t, int32_t, int32_t) { return 0; }
extern "C" ts_status ts_mla_paged_decode(const void*, const void*, const int32_t*, int32_t,
                                         const int32_t*, int32_t, int32_t, int32_t, int32_t,
                                         int32_t, int32_t, float, void*, float*, void*, size_t,
                                         void*) {
  return ts::fail(TS_ERR_UNSUPPORTED, "ts_mla_paged_decode: not built yet");
}
