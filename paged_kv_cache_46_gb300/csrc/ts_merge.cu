// ts_merge_states: merge two attention states over disjoint key sets by LSE.
//
// TokenSpeed deep dive, section 7 fig. 3 (stage 3 reduces split partials by
// their LSE) and the Tokasaurus blog's shared-prefix attention, where the
// prefix state and the per-sequence state are combined the same way.
//
// Memory-bound elementwise kernel: one warp per row, 16-byte vector loads.
#include <cmath>

#include "ts_common.cuh"

namespace ts {
namespace {

template <typename T>
struct Vec4;  // four elements of T as one load/store
template <>
struct Vec4<float> {
  __device__ static float4 load(const void* p, int64_t i) {
    return reinterpret_cast<const float4*>(p)[i];
  }
  __device__ static void store(void* p, int64_t i, float4 v) { reinterpret_cast<float4*>(p)[i] = v; }
};
template <>
struct Vec4<__nv_bfloat16> {
  __device__ static float4 load(const void* p, int64_t i) {
    const uint2 r = reinterpret_cast<const uint2*>(p)[i];
    const float2 a = bf16x2_to_float2(r.x), b = bf16x2_to_float2(r.y);
    return make_float4(a.x, a.y, b.x, b.y);
  }
  __device__ static void store(void* p, int64_t i, float4 v) {
    uint2 r;
    r.x = float2_to_bf16x2(v.x, v.y);
    r.y = float2_to_bf16x2(v.z, v.w);
    reinterpret_cast<uint2*>(p)[i] = r;
  }
};

template <typename T>
__global__ void __launch_bounds__(256) merge_states_kernel(const void* o_a, const float* lse_a,
                                                           const void* o_b, const float* lse_b,
                                                           void* o_out, float* lse_out,
                                                           int64_t rows, int D) {
  const int64_t row = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const float la = lse_a[row], lb = lse_b[row];
  const float mx = fmaxf(la, lb);
  const bool empty = mx == -INFINITY;
  const float ms = empty ? 0.f : mx;
  const float wa = la == -INFINITY ? 0.f : __expf(la - ms);
  const float wb = lb == -INFINITY ? 0.f : __expf(lb - ms);
  const float wsum = wa + wb;
  const float inv = empty ? 0.f : 1.0f / wsum;
  const float ca = wa * inv, cb = wb * inv;
  const int nvec = D / 4;
  const int64_t base = row * nvec;
  for (int v = lane; v < nvec; v += 32) {
    float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
    if (!empty) {
      const float4 a = Vec4<T>::load(o_a, base + v);
      const float4 b = Vec4<T>::load(o_b, base + v);
      // an empty side contributes nothing, whatever its O holds
      r.x = (wa > 0.f ? ca * a.x : 0.f) + (wb > 0.f ? cb * b.x : 0.f);
      r.y = (wa > 0.f ? ca * a.y : 0.f) + (wb > 0.f ? cb * b.y : 0.f);
      r.z = (wa > 0.f ? ca * a.z : 0.f) + (wb > 0.f ? cb * b.z : 0.f);
      r.w = (wa > 0.f ? ca * a.w : 0.f) + (wb > 0.f ? cb * b.w : 0.f);
    }
    Vec4<T>::store(o_out, base + v, r);
  }
  if (lane == 0 && lse_out) lse_out[row] = empty ? -INFINITY : ms + logf(wsum);
}

}  // namespace
}  // namespace ts

extern "C" ts_status ts_merge_states(const void* o_a, const float* lse_a, const void* o_b,
                                     const float* lse_b, void* o_out, float* lse_out,
                                     int64_t rows, int32_t D, ts_dtype dtype, void* stream) {
  using namespace ts;
  if (rows < 0 || D <= 0 || D > 1024)
    return fail(TS_ERR_INVALID_ARG, "ts_merge_states: bad sizes rows=%lld D=%d",
                static_cast<long long>(rows), D);
  if (dtype != TS_F32 && dtype != TS_BF16)
    return fail(TS_ERR_INVALID_ARG, "ts_merge_states: bad dtype %d", static_cast<int>(dtype));
  if (D % (dtype == TS_F32 ? 4 : 8) != 0)
    return fail(TS_ERR_UNSUPPORTED, "ts_merge_states: D=%d must be a multiple of %d", D,
                dtype == TS_F32 ? 4 : 8);
  if (rows == 0) return TS_OK;
  if (!o_a || !lse_a || !o_b || !lse_b || !o_out)
    return fail(TS_ERR_INVALID_ARG, "ts_merge_states: null pointer");
  for (const void* p : {o_a, o_b, static_cast<const void*>(o_out)})
    if (reinterpret_cast<uintptr_t>(p) % 16 != 0)
      return fail(TS_ERR_INVALID_ARG, "ts_merge_states: state tensors must be 16-byte aligned");
  const int64_t threads = rows * 32;
  const unsigned blocks = static_cast<unsigned>((threads + 255) / 256);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  LaunchTrace trace("merge_states_kernel", s);
  if (dtype == TS_F32)
    merge_states_kernel<float><<<blocks, 256, 0, s>>>(o_a, lse_a, o_b, lse_b, o_out, lse_out, rows, D);
  else
    merge_states_kernel<__nv_bfloat16>
        <<<blocks, 256, 0, s>>>(o_a, lse_a, o_b, lse_b, o_out, lse_out, rows, D);
  return cuda_check(cudaGetLastError(), "ts_merge_states: launch");
}
