// Shared device and host helpers for the ts_attn library (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ts_attn.h"

namespace ts {

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

// Records a formatted detail message for ts_last_error_detail() and returns s.
ts_status fail(ts_status s, const char* fmt, ...);
// Maps a CUDA error to TS_ERR_CUDA with a detail message (TS_OK if none).
ts_status cuda_check(cudaError_t e, const char* what);

// Device address of the allocation-free entry point's static scratch on the
// current device (looked up once per device; defined beside that entry point).
ts_status noalloc_scratch_address(void** addr);
// SM count of the current device (cached per device).
int device_sm_count();
// CTAs of a persistent grid over the batch's pages: one per SM.
// TS_PAGED_DECODE_CTAS overrides it (tests use it to sweep how sequences are
// cut across CTAs).
int paged_decode_ctas();
// Current device ordinal.
int current_device();

constexpr size_t kWorkspaceAlign = 256;

// Shared-prefix state handed to the paged kernel in cascade mode (device pointers).
struct PrefixInputs {
  const int32_t* group_of;    // [B] group or -1
  const int32_t* prefix_len;  // [groups] shared tokens (whole pages)
  const float* prefix_o;      // [B, H_q, D] normalised prefix output (fp32)
  const float* prefix_lse;    // [B, H_q] prefix LSE (natural log)
  int32_t num_groups;         // entries of prefix_len
};

// Paged split-KV decode (ts_paged_decode.cu); `pre` selects cascade mode.
ts_status launch_paged_decode_impl(const void* q, const void* k_pool, const void* v_pool,
                                   const int32_t* block_table, int32_t bt_stride,
                                   const int32_t* seq_lens, int32_t B, int32_t H_q, int32_t H_kv,
                                   int32_t D, int32_t page_size, int32_t num_pages, float scale,
                                   ts_dtype dtype, void* out, float* lse, void* workspace,
                                   size_t workspace_bytes, cudaStream_t stream, const char* who,
                                   const PrefixInputs* pre);
size_t paged_decode_workspace_bytes(int B, int H_q, int D);
inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Runs `prepare` (function attributes, attribute queries) the first time a
// kernel is launched on a device and remembers a success, so that later calls
// (and calls captured into a CUDA graph) do no attribute work.
ts_status prepare_once(const void* kernel, ts_status (*prepare)(const void*));

// Launch trace: while ts_trace_enable(1) is in force, a LaunchTrace scope
// records one CUDA event on `stream` when it opens and one when it closes
// (put exactly one kernel launch inside); ts_trace_collect reads them back.
class LaunchTrace {
 public:
  LaunchTrace(const char* kernel, cudaStream_t stream);
  ~LaunchTrace();
  LaunchTrace(const LaunchTrace&) = delete;
  LaunchTrace& operator=(const LaunchTrace&) = delete;

 private:
  const char* kernel_;
  cudaStream_t stream_;
  cudaEvent_t begin_ = nullptr;
  int device_ = -1;
};

// ---------------------------------------------------------------------------
// Device side
// ---------------------------------------------------------------------------

// Upper bound on any single pipeline wait. Normal waits last microseconds; on
// expiry the kernel records TS_DEVERR_TIMEOUT and leaves instead of hanging.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Makes mbarrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Orders this thread's generic-proxy shared-memory accesses before later
// async-proxy ones (bulk copies, tensor-core operand reads) after a barrier.
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t tx_bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(tx_bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking test: has the phase with the given parity completed?
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase with the given parity to complete; false on timeout.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
  }
}

// 1-D bulk copy global -> shared (TMA engine), completion counted on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Same, with an L2 cache-policy hint (an evict-first policy for streamed data).
__device__ __forceinline__ void bulk_g2s_hint(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], "
      "%2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Programmatic dependent launch: let the next kernel in the stream start its
// prologue / wait for the previous kernel's results.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_primary() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Named barrier over `nthreads` threads (a multiple of 32).
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// 2^x on the MUFU unit (ex2.approx, flush-to-zero): exp2(-inf) = 0.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Maximum of three floats in one instruction (NaN inputs are ignored, as fmaxf).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// bf16 pair in one 32-bit word -> two floats (exact widening).
__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

__device__ __forceinline__ uint32_t float2_to_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void set_device_error(uint32_t* word, uint32_t bits) {
  if (word != nullptr) atomicOr(word, bits);
}

}  // namespace ts
