// Status strings, error details, device-property cache and the error-word reader.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <utility>
#include <vector>

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

namespace {
struct TraceRecord {
  const char* kernel;
  cudaEvent_t begin, end;
  int device;
};
std::atomic<bool> g_trace_on{false};
std::mutex g_trace_mutex;
std::vector<TraceRecord> g_trace;                      // recorded, not yet collected
std::vector<std::pair<int, cudaEvent_t>> g_free_events;  // (device, event) for reuse

cudaEvent_t take_event(int device) {  // caller holds g_trace_mutex
  for (size_t i = 0; i < g_free_events.size(); ++i)
    if (g_free_events[i].first == device) {
      cudaEvent_t e = g_free_events[i].second;
      g_free_events.erase(g_free_events.begin() + static_cast<long>(i));
      return e;
    }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}
}  // namespace

LaunchTrace::LaunchTrace(const char* kernel, cudaStream_t stream) : kernel_(kernel), stream_(stream) {
  if (!g_trace_on.load(std::memory_order_relaxed)) return;
  device_ = current_device();
  std::lock_guard<std::mutex> lock(g_trace_mutex);
  begin_ = take_event(device_);
  if (begin_ && cudaEventRecord(begin_, stream_) != cudaSuccess) {
    g_free_events.emplace_back(device_, begin_);
    begin_ = nullptr;
  }
}

LaunchTrace::~LaunchTrace() {
  if (!begin_) return;
  std::lock_guard<std::mutex> lock(g_trace_mutex);
  cudaEvent_t end = take_event(device_);
  if (end && cudaEventRecord(end, stream_) == cudaSuccess) {
    g_trace.push_back({kernel_, begin_, end, device_});
  } else {
    g_free_events.emplace_back(device_, begin_);
    if (end) g_free_events.emplace_back(device_, end);
  }
}

namespace {
std::mutex g_prep_mutex;
std::vector<std::pair<const void*, int>> g_prepared;  // (kernel, device) prepared successfully
}  // namespace

ts_status prepare_once(const void* kernel, ts_status (*prepare)(const void*)) {
  const int dev = current_device();
  std::lock_guard<std::mutex> lock(g_prep_mutex);
  for (const auto& e : g_prepared)
    if (e.first == kernel && e.second == dev) return TS_OK;
  const ts_status st = prepare(kernel);
  if (st == TS_OK) g_prepared.emplace_back(kernel, dev);
  return st;
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

int paged_decode_ctas() {
  if (const char* env = getenv("TS_PAGED_DECODE_CTAS")) {
    const int n = atoi(env);
    if (n > 0 && n <= 65535) return n;
  }
  return device_sm_count();
}

}  // namespace ts

namespace ts {
namespace {
// One stamp per CTA: the SM it runs on, that SM's cycle counter and the
// global nanosecond timer, read back to back by the CTA's first thread.
__global__ void clock_stamp_kernel(unsigned long long* out) {
  if (threadIdx.x != 0) return;
  unsigned int sm;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(sm));
  const unsigned long long clk = clock64();
  const unsigned long long ns = globaltimer_ns();
  out[3 * blockIdx.x] = sm;
  out[3 * blockIdx.x + 1] = clk;
  out[3 * blockIdx.x + 2] = ns;
}
}  // namespace
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

ts_status ts_trace_enable(int32_t on) {
  ts::g_trace_on.store(on != 0);
  return TS_OK;
}

int32_t ts_trace_collect(ts_launch_record* out, int32_t capacity) {
  std::vector<ts::TraceRecord> recs;
  {
    std::lock_guard<std::mutex> lock(ts::g_trace_mutex);
    recs.swap(ts::g_trace);
  }
  int32_t n = 0;
  bool failed = false;
  for (const ts::TraceRecord& r : recs) {
    float ms = 0.f;
    if (cudaEventSynchronize(r.end) != cudaSuccess || cudaEventElapsedTime(&ms, r.begin, r.end) != cudaSuccess)
      failed = true;
    if (out != nullptr && n < capacity) {
      std::memset(out[n].kernel, 0, sizeof(out[n].kernel));
      std::strncpy(out[n].kernel, r.kernel, sizeof(out[n].kernel) - 1);
      out[n].ms = ms;
    }
    ++n;
  }
  {
    std::lock_guard<std::mutex> lock(ts::g_trace_mutex);
    for (const ts::TraceRecord& r : recs) {
      ts::g_free_events.emplace_back(r.device, r.begin);
      ts::g_free_events.emplace_back(r.device, r.end);
    }
  }
  if (failed) {
    ts::fail(TS_ERR_CUDA, "ts_trace_collect: reading an event failed");
    return -1;
  }
  return n;
}

ts_status ts_clock_stamp(void* stamps, int32_t n, void* stream) {
  if (stamps == nullptr || n < 1 || n > 65535)
    return ts::fail(TS_ERR_INVALID_ARG, "ts_clock_stamp: stamps=%p n=%d (n in [1, 65535])", stamps, n);
  if (reinterpret_cast<uintptr_t>(stamps) % 8 != 0)
    return ts::fail(TS_ERR_INVALID_ARG, "ts_clock_stamp: stamps must be 8-byte aligned");
  ts::clock_stamp_kernel<<<n, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<unsigned long long*>(stamps));
  return ts::cuda_check(cudaGetLastError(), "ts_clock_stamp launch");
}

ts_status ts_read_device_error(const void* workspace, uint32_t* error_bits, void* stream) {
  if (error_bits == nullptr)
    return ts::fail(TS_ERR_INVALID_ARG, "ts_read_device_error: null pointer");
  if (workspace == nullptr) {   // the allocation-free entry point's static scratch
    void* scratch = nullptr;
    ts_status st0 = ts::noalloc_scratch_address(&scratch);
    if (st0 != TS_OK) return st0;
    workspace = scratch;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  ts_status st = ts::cuda_check(
      cudaMemcpyAsync(error_bits, workspace, sizeof(uint32_t), cudaMemcpyDeviceToHost, s),
      "ts_read_device_error: copy");
  if (st != TS_OK) return st;
  return ts::cuda_check(cudaStreamSynchronize(s), "ts_read_device_error: sync");
}

}  // extern "C"
