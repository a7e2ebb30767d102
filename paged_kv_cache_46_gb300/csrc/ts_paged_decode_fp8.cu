// Instantiations of the paged split-KV decode kernel for an fp8 (e4m3fn)
// cache (ts_paged_decode_fp8_attn): K/V codes with one float32 scale per
// (page, row, kv head), bf16 queries and output. Own translation unit so the
// parallel build compiles them beside the other variants.
#include "ts_paged_decode_kernel.cuh"

namespace ts {
namespace {

template <int D>
PagedKernelFn pick_rows(int G) {
  switch (G) {
    case 1: return paged_decode_kernel<__nv_bfloat16, D, 1, false, false, true>;
    case 2: return paged_decode_kernel<__nv_bfloat16, D, 2, false, false, true>;
    case 4: return paged_decode_kernel<__nv_bfloat16, D, 4, false, false, true>;
    default: return nullptr;
  }
}

}  // namespace

PagedKernelFn pick_paged_fp8_kernel(int D, int G) {
  if (D == 64) return pick_rows<64>(G);
  if (D == 128) return pick_rows<128>(G);
  return nullptr;
}

}  // namespace ts
