// ts_kv_append: write one new token's K and V per sequence into its page.
//
// SwiftLLM page, section 3.1: a request's KV cache is a list of fixed-size
// blocks handed out on demand and found through its block table, so token
// `pos` lands in page block_table[b][pos / page_size] at row pos % page_size.
//
// One CTA per sequence; the [H_kv, D] row of K and of V is contiguous in both
// the source and the pool (NHD layout), so the copy is a straight 16-byte
// vector copy of row_bytes bytes each.
#include "ts_common.cuh"

namespace ts {
namespace {

__global__ void __launch_bounds__(256) kv_append_kernel(const uint4* __restrict__ k_new,
                                                        const uint4* __restrict__ v_new,
                                                        uint4* __restrict__ k_pool,
                                                        uint4* __restrict__ v_pool,
                                                        const int32_t* __restrict__ block_table,
                                                        int32_t bt_stride,
                                                        const int32_t* __restrict__ positions,
                                                        int32_t page_size, int32_t num_pages,
                                                        int32_t row_vecs) {
  // Programmatic dependent launch: wait for the previous kernel of the stream
  // before reading anything, and let the next one (the attention, which reads
  // only lengths and block tables before its own wait) start its prologue.
  pdl_wait_primary();
  pdl_launch_dependents();
  const int b = blockIdx.x;
  const int pos = positions[b];
  if (pos < 0) return;
  const int slot = pos / page_size;
  if (slot >= bt_stride) return;
  const int page = block_table[static_cast<int64_t>(b) * bt_stride + slot];
  if (page < 0 || page >= num_pages) return;
  const int row = pos % page_size;
  const int64_t dst = (static_cast<int64_t>(page) * page_size + row) * row_vecs;
  const int64_t src = static_cast<int64_t>(b) * row_vecs;
  for (int i = threadIdx.x; i < row_vecs; i += blockDim.x) {
    k_pool[dst + i] = k_new[src + i];
    v_pool[dst + i] = v_new[src + i];
  }
}

}  // namespace
}  // namespace ts

extern "C" ts_status ts_kv_append(const void* k_new, const void* v_new, void* k_pool, void* v_pool,
                                  const int32_t* block_table, int32_t bt_stride,
                                  const int32_t* positions, int32_t B, int32_t H_kv, int32_t D,
                                  int32_t page_size, int32_t num_pages, ts_dtype dtype,
                                  void* stream) {
  using namespace ts;
  if (B < 0 || H_kv <= 0 || D <= 0 || page_size <= 0 || num_pages <= 0 || bt_stride <= 0)
    return fail(TS_ERR_INVALID_ARG, "ts_kv_append: bad sizes (B=%d H_kv=%d D=%d ps=%d P=%d bt=%d)",
                B, H_kv, D, page_size, num_pages, bt_stride);
  if (dtype != TS_F32 && dtype != TS_BF16)
    return fail(TS_ERR_INVALID_ARG, "ts_kv_append: bad dtype %d", static_cast<int>(dtype));
  if (B == 0) return TS_OK;
  if (!k_new || !v_new || !k_pool || !v_pool || !block_table || !positions)
    return fail(TS_ERR_INVALID_ARG, "ts_kv_append: null pointer");
  const size_t esize = dtype == TS_F32 ? 4 : 2;
  const size_t row_bytes = static_cast<size_t>(H_kv) * D * esize;
  if (row_bytes % 16 != 0)
    return fail(TS_ERR_UNSUPPORTED, "ts_kv_append: H_kv*D*elem (%zu B) not a multiple of 16",
                row_bytes);
  for (const void* p : {k_new, v_new, static_cast<const void*>(k_pool),
                        static_cast<const void*>(v_pool)})
    if (reinterpret_cast<uintptr_t>(p) % 16 != 0)
      return fail(TS_ERR_INVALID_ARG, "ts_kv_append: tensors must be 16-byte aligned");
  const int row_vecs = static_cast<int>(row_bytes / 16);
  const int threads = row_vecs >= 256 ? 256 : ((row_vecs + 31) / 32) * 32;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(B);
  cfg.blockDim = dim3(threads);
  cfg.stream = static_cast<cudaStream_t>(stream);
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  LaunchTrace trace("kv_append_kernel", cfg.stream);
  return cuda_check(cudaLaunchKernelEx(&cfg, kv_append_kernel, static_cast<const uint4*>(k_new),
                                       static_cast<const uint4*>(v_new), static_cast<uint4*>(k_pool),
                                       static_cast<uint4*>(v_pool), block_table, bt_stride, positions,
                                       page_size, num_pages, row_vecs),
                    "ts_kv_append: launch");
}
