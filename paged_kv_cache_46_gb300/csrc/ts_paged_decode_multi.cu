// Instantiations of the paged split-KV decode kernel for several query tokens
// per sequence (ts_paged_decode_multi_attn). They live in their own
// translation unit so that the library's parallel build compiles them beside
// the single-token kernels of ts_paged_decode.cu.
#include "ts_paged_decode_kernel.cuh"

namespace ts {
namespace {

template <typename T, int D>
PagedKernelFn pick_rows(int G) {
  switch (G) {
    case 1: return paged_decode_kernel<T, D, 1, false, true, false>;
    case 2: return paged_decode_kernel<T, D, 2, false, true, false>;
    case 4: return paged_decode_kernel<T, D, 4, false, true, false>;
    case 8: return paged_decode_kernel<T, D, 8, false, true, false>;
    default: return nullptr;
  }
}

}  // namespace

PagedKernelFn pick_paged_multi_kernel(ts_dtype dt, int D, int G) {
  if (dt == TS_BF16) {
    if (D == 64) return pick_rows<__nv_bfloat16, 64>(G);
    if (D == 128) return pick_rows<__nv_bfloat16, 128>(G);
  } else if (dt == TS_F32) {
    if (D == 64) return pick_rows<float, 64>(G);
    if (D == 128) return pick_rows<float, 128>(G);
  }
  return nullptr;
}

}  // namespace ts
