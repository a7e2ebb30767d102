// Instantiations of the paged split-KV decode kernel for a sliding-window KV
// group (ts_paged_decode_window_attn): each sequence attends its last
// `window` tokens. Own translation unit so the parallel build compiles them
// beside the other variants; the whole-context kernels are not affected.
#include "ts_paged_decode_kernel.cuh"

namespace ts {
namespace {

template <typename T, int D>
PagedKernelFn pick_rows(int G) {
  switch (G) {
    case 1: return paged_decode_kernel<T, D, 1, false, false, false, true>;
    case 2: return paged_decode_kernel<T, D, 2, false, false, false, true>;
    case 4: return paged_decode_kernel<T, D, 4, false, false, false, true>;
    case 8: return paged_decode_kernel<T, D, 8, false, false, false, true>;
    default: return nullptr;
  }
}

}  // namespace

PagedKernelFn pick_paged_window_kernel(ts_dtype dt, int D, int G) {
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
