// ts_kv_append_fp8: quantize one new token's K and V rows per sequence into an
// fp8 (e4m3fn) paged cache.
//
// Placement as ts_kv_append (SwiftLLM page, section 3.1). Quantization per
// token group, tokenspeed 딥다이브 (fiv.co.kr) section 6-4: a group's scale
// is max(max |x|, 1e-10) / 448 and its codes are e4m3(clamp(x / scale, -448,
// 448)), the scale and the division in float32 rounded to nearest even and the
// cast rounded to nearest even. A token group is one (token, kv head) row of D
// values, so the cache keeps one float32 scale per (page, row, kv head).
//
// One warp per (sequence, kv head, K or V) group: each lane widens D / 32
// elements, a butterfly max gives the group maximum, and each lane writes its
// codes as one 2- or 4-byte store.
#include <cuda_fp8.h>

#include "ts_common.cuh"

namespace ts {
namespace {

constexpr float kE4M3Max = 448.0f;

template <typename T, int D>
__global__ void __launch_bounds__(256) kv_append_fp8_kernel(
    const T* __restrict__ k_new, const T* __restrict__ v_new, uint8_t* __restrict__ k_pool,
    uint8_t* __restrict__ v_pool, float* __restrict__ k_scale, float* __restrict__ v_scale,
    const int32_t* __restrict__ block_table, int32_t bt_stride, const int32_t* __restrict__ positions,
    int32_t B, int32_t H_kv, int32_t page_size, int32_t num_pages) {
  // Programmatic dependent launch as in ts_kv_append.
  pdl_wait_primary();
  pdl_launch_dependents();
  constexpr int kPer = D / 32;  // elements per lane (2 or 4)
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;  // group: (b, head, K or V)
  const int lane = threadIdx.x & 31;
  if (gw >= 2 * B * H_kv) return;
  const bool is_v = gw >= B * H_kv;
  const int bh = is_v ? gw - B * H_kv : gw;
  const int b = bh / H_kv, h = bh % H_kv;
  const int pos = positions[b];
  if (pos < 0) return;
  const int slot = pos / page_size;
  if (slot >= bt_stride) return;
  const int page = block_table[static_cast<int64_t>(b) * bt_stride + slot];
  if (page < 0 || page >= num_pages) return;
  const int row = pos % page_size;
  const T* src = (is_v ? v_new : k_new) + (static_cast<int64_t>(b) * H_kv + h) * D + lane * kPer;
  float x[kPer];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    x[i] = static_cast<float>(src[i]);
    amax = fmaxf(amax, fabsf(x[i]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float scale = __fdiv_rn(fmaxf(amax, 1e-10f), kE4M3Max);
  uint32_t packed = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const float y = fminf(fmaxf(__fdiv_rn(x[i], scale), -kE4M3Max), kE4M3Max);
    const uint32_t c = __nv_cvt_float_to_fp8(y, __NV_SATFINITE, __NV_E4M3);
    packed |= c << (8 * i);
  }
  const int64_t cell = (static_cast<int64_t>(page) * page_size + row) * H_kv + h;
  uint8_t* dst = (is_v ? v_pool : k_pool) + cell * D + lane * kPer;
  if constexpr (kPer == 4)
    *reinterpret_cast<uint32_t*>(dst) = packed;
  else
    *reinterpret_cast<uint16_t*>(dst) = static_cast<uint16_t>(packed);
  if (lane == 0) (is_v ? v_scale : k_scale)[cell] = scale;
}

template <typename T>
ts_status launch(int D, const void* k_new, const void* v_new, void* k_pool, void* v_pool,
                 float* k_scale, float* v_scale, const int32_t* block_table, int32_t bt_stride,
                 const int32_t* positions, int32_t B, int32_t H_kv, int32_t page_size,
                 int32_t num_pages, cudaStream_t stream) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  const long long warps = 2ll * B * H_kv;
  cfg.gridDim = dim3(static_cast<unsigned>((warps + 7) / 8));
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  auto kern = D == 64 ? kv_append_fp8_kernel<T, 64> : kv_append_fp8_kernel<T, 128>;
  LaunchTrace trace("kv_append_fp8_kernel", stream);
  return cuda_check(cudaLaunchKernelEx(&cfg, kern, static_cast<const T*>(k_new), static_cast<const T*>(v_new),
                                       static_cast<uint8_t*>(k_pool), static_cast<uint8_t*>(v_pool), k_scale,
                                       v_scale, block_table, bt_stride, positions, B, H_kv, page_size,
                                       num_pages),
                    "ts_kv_append_fp8: launch");
}

}  // namespace
}  // namespace ts

extern "C" ts_status ts_kv_append_fp8(const void* k_new, const void* v_new, void* k_pool, void* v_pool,
                                      float* k_scale, float* v_scale, const int32_t* block_table,
                                      int32_t bt_stride, const int32_t* positions, int32_t B,
                                      int32_t H_kv, int32_t D, int32_t page_size, int32_t num_pages,
                                      ts_dtype dtype, void* stream) {
  using namespace ts;
  const char* who = "ts_kv_append_fp8";
  if (B < 0 || H_kv <= 0 || D <= 0 || page_size <= 0 || num_pages <= 0 || bt_stride <= 0)
    return fail(TS_ERR_INVALID_ARG, "%s: bad sizes (B=%d H_kv=%d D=%d ps=%d P=%d bt=%d)", who, B, H_kv, D,
                page_size, num_pages, bt_stride);
  if (dtype != TS_F32 && dtype != TS_BF16)
    return fail(TS_ERR_INVALID_ARG, "%s: bad dtype %d", who, static_cast<int>(dtype));
  if (D != 64 && D != 128) return fail(TS_ERR_UNSUPPORTED, "%s: D=%d (supported 64, 128)", who, D);
  if (B == 0) return TS_OK;
  if (!k_new || !v_new || !k_pool || !v_pool || !k_scale || !v_scale || !block_table || !positions)
    return fail(TS_ERR_INVALID_ARG, "%s: null pointer", who);
  for (const void* p : {static_cast<const void*>(k_pool), static_cast<const void*>(v_pool)})
    if (reinterpret_cast<uintptr_t>(p) % 16 != 0)
      return fail(TS_ERR_INVALID_ARG, "%s: pools must be 16-byte aligned", who);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == TS_BF16)
    return launch<__nv_bfloat16>(D, k_new, v_new, k_pool, v_pool, k_scale, v_scale, block_table, bt_stride,
                                 positions, B, H_kv, page_size, num_pages, s);
  return launch<float>(D, k_new, v_new, k_pool, v_pool, k_scale, v_scale, block_table, bt_stride, positions,
                       B, H_kv, page_size, num_pages, s);
}
