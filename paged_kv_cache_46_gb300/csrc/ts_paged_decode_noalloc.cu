// ts_paged_decode_attn_noalloc: ts_paged_decode_attn for callers that cannot
// allocate device memory.
//
// Some callers have no way to hand this library a workspace: a plugin run by
// a host runtime that passes it only input and output buffers, or a serving
// engine that has already reserved all free HBM for its KV-cache pool and
// whose hot loop must not pay cudaMalloc's latency and implicit device
// synchronisation. This entry point takes the split-KV scratch (error word,
// per-sequence split records, fp32 partial states) from a fixed array that
// lives in the library's own device image instead. It performs no device
// allocation of any kind; the caller still passes every input and output.
//
// Costs and limits:
//   * The array is TS_NOALLOC_SCRATCH_BYTES bytes, and every GPU that loads
//     the library holds one copy of it until the process exits.
//   * All calls on a device share that one array. Calls whose kernels can
//     overlap on the GPU (different streams without ordering between them)
//     race on it and produce wrong results; serialise them.
//   * The array keeps whatever the previous call left. Only the error word
//     must start at zero; it is cleared at the start of every call. The split
//     records and partial states are fully written before they are read.
//   * The first call on each device looks up the array's device address with
//     that device current and caches it; make that first call before any
//     stream capture.
//   * Under CUDA's lazy module loading (the default) the array's memory is
//     committed when its module is first loaded on a device, which is that
//     first call (or ts_read_device_error(NULL, ...)); with eager loading it
//     is committed when the library is loaded. A caller that reserves all
//     free HBM for its KV-cache pool must make the first call before that.
//   * Device-side problems (a page id out of range, a timed-out wait) set
//     bits in the array's error word; ts_read_device_error(NULL, ...) reads
//     it for the current device.
#include <mutex>

#include "ts_common.cuh"

namespace ts {

// Defined in ts_paged_decode.cu.
ts_status launch_paged_decode(const void* q, const void* k_pool, const void* v_pool,
                              const int32_t* block_table, int32_t bt_stride,
                              const int32_t* seq_lens, int32_t B, int32_t H_q, int32_t H_kv,
                              int32_t D, int32_t page_size, int32_t num_pages, float scale,
                              ts_dtype dtype, void* out, float* lse, void* workspace,
                              size_t workspace_bytes, cudaStream_t stream, const char* who);
size_t paged_decode_workspace_bytes(int B, int H_q, int D);
ts_status paged_decode_check_args(const void* q, const void* k_pool, const void* v_pool,
                                  const int32_t* block_table, int32_t bt_stride,
                                  const int32_t* seq_lens, int32_t B, int32_t H_q, int32_t H_kv,
                                  int32_t D, int32_t page_size, int32_t num_pages, float scale,
                                  ts_dtype dtype, void* out, const char* who);

namespace {

constexpr size_t kScratchBytes = TS_NOALLOC_SCRATCH_BYTES;

// Host code must not use this name as a device address: on the host it is
// only a stand-in symbol. Its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};

}  // namespace

// Device address of g_noalloc_scratch on the current device (looked up once).
ts_status noalloc_scratch_address(void** addr) {
  int dev = 0;
  ts_status st = cuda_check(cudaGetDevice(&dev), "ts_paged_decode_attn_noalloc: cudaGetDevice");
  if (st != TS_OK) return st;
  if (dev < 0 || dev >= kMaxDevices)
    return fail(TS_ERR_UNSUPPORTED, "ts_paged_decode_attn_noalloc: device ordinal %d >= %d", dev,
                kMaxDevices);
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    st = cuda_check(cudaGetSymbolAddress(&p, g_noalloc_scratch),
                    "ts_paged_decode_attn_noalloc: cudaGetSymbolAddress of the static scratch");
    if (st != TS_OK) return st;
    if (p == nullptr)
      return fail(TS_ERR_CUDA, "ts_paged_decode_attn_noalloc: static scratch has no device address");
    g_scratch_addr[dev] = p;
  }
  *addr = g_scratch_addr[dev];
  return TS_OK;
}

}  // namespace ts

extern "C" ts_status ts_paged_decode_attn_noalloc(const void* q, const void* k_pool,
                                                  const void* v_pool, const int32_t* block_table,
                                                  int32_t bt_stride, const int32_t* seq_lens,
                                                  int32_t B, int32_t H_q, int32_t H_kv, int32_t D,
                                                  int32_t page_size, int32_t num_pages,
                                                  float scale, ts_dtype dtype, void* out,
                                                  float* lse, void* stream) {
  using namespace ts;
  const char* who = "ts_paged_decode_attn_noalloc";
  if (B == 0) return TS_OK;
  // The arguments and the shape are checked first, so that an unsupported
  // shape is reported as such rather than as a scratch overflow.
  ts_status st = paged_decode_check_args(q, k_pool, v_pool, block_table, bt_stride, seq_lens, B,
                                         H_q, H_kv, D, page_size, num_pages, scale, dtype, out, who);
  if (st != TS_OK) return st;
  const size_t need = paged_decode_workspace_bytes(B, H_q, D);
  if (need == 0) return fail(TS_ERR_CUDA, "%s: cannot size the scratch (SM count query failed)", who);
  if (need > kScratchBytes)
    return fail(TS_ERR_WORKSPACE,
                "%s: B=%d, H_q=%d, D=%d needs %zu bytes of scratch but the static scratch holds %zu "
                "bytes; use ts_paged_decode_attn with a workspace",
                who, B, H_q, D, need, kScratchBytes);
  void* scratch = nullptr;
  st = noalloc_scratch_address(&scratch);
  if (st != TS_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  st = cuda_check(cudaMemsetAsync(scratch, 0, sizeof(uint32_t), s), "clear the scratch error word");
  if (st != TS_OK) return st;
  return launch_paged_decode(q, k_pool, v_pool, block_table, bt_stride, seq_lens, B, H_q, H_kv, D,
                             page_size, num_pages, scale, dtype, out, lse, scratch, kScratchBytes, s,
                             who);
}
