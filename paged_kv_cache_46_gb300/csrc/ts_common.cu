// Status strings, error details, device-property cache and the error-word reader.
#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <string>

#include "ts_common.cuh"

namespace ts {

namespace {
thread_local std::string g_detail;
std::mutex g_sm_mutex;
int g_sm_count[64] = {0};
}  // namespace

ts_status fail(ts_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_detail = buf;
  return s;
}

ts_status cuda_check(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return TS_OK;
  return fail(TS_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  return dev;
}

int device_sm_count() {
  const int dev = current_device();
  if (dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(g_sm_mutex);
  if (g_sm_count[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    g_sm_count[dev] = n;
  }
  return g_sm_count[dev];
}

}  // namespace ts

extern "C" {

const char* ts_status_string(int status) {
  switch (status) {
    case TS_OK: return "TS_OK";
    case TS_ERR_INVALID_ARG: return "TS_ERR_INVALID_ARG";
    case TS_ERR_UNSUPPORTED: return "TS_ERR_UNSUPPORTED";
    case TS_ERR_WORKSPACE: return "TS_ERR_WORKSPACE";
    case TS_ERR_CUDA: return "TS_ERR_CUDA";
    case TS_ERR_CAPACITY: return "TS_ERR_CAPACITY";
    default: return "TS_ERR_UNKNOWN";
  }
}

const char* ts_last_error_detail(void) { return ts::g_detail.c_str(); }

const char* ts_version(void) { return "ts_attn 0.1 (sm_103a)"; }

ts_status ts_read_device_error(const void* workspace, uint32_t* error_bits, void* stream) {
  if (workspace == nullptr || error_bits == nullptr)
    return ts::fail(TS_ERR_INVALID_ARG, "ts_read_device_error: null pointer");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  ts_status st = ts::cuda_check(
      cudaMemcpyAsync(error_bits, workspace, sizeof(uint32_t), cudaMemcpyDeviceToHost, s),
      "ts_read_device_error: copy");
  if (st != TS_OK) return st;
  return ts::cuda_check(cudaStreamSynchronize(s), "ts_read_device_error: sync");
}

}  // extern "C"
