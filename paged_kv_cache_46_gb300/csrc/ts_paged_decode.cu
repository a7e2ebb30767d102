// ts_paged_decode_attn: GQA decode attention over a paged KV cache.
//
// What it computes (SwiftLLM page, sections 3.1 and 5.1): for each sequence b
// and query head h, softmax(scale * q K_b^T) V_b over the sequence's tokens,
// gathered page by page through its block table.
//
// How (flash-decoding / split-KV, TokenSpeed deep dive, section 7 fig. 3 and
// 7.1: split-KV partial outputs with their LSE, then a second kernel reduces
// the partials by LSE):
//
//   * Persistent grid, one CTA per SM. All pages of the batch, in (sequence,
//     page) order, are cut into gridDim.x equal contiguous ranges, so every
//     SM streams the same number of bytes whatever the length mix. The cut is
//     computed on the device from seq_lens in each CTA's prologue.
//   * Warp specialisation: one producer warp walks the CTA's range and moves
//     each page (all kv heads, K and V, the valid rows only) into a shared-
//     memory stage with two 1-D TMA bulk copies; on a sequence's first page it
//     also copies that sequence's query rows. Completion is tracked by
//     mbarrier transaction counts; consumers release stages on "empty"
//     mbarriers. One consumer warp per kv head reads its rows from the stage.
//   * Inside a consumer warp, LPT lanes share one token (each lane owns DPL
//     dims, 16-byte shared loads), NG token groups run in parallel, and each
//     group keeps its own online-softmax state (m, l, acc) in registers for
//     the g query heads of the kv head, so every K/V element read from shared
//     memory is used g times. Dot products use packed fp32 FMA (FFMA2) and
//     are reduced across the LPT lanes with warp shuffles; softmax runs in
//     the log2 domain (scale * log2 e folded into q).
//   * Several query tokens per sequence (speculative verify, q_len > 1) are
//     folded into the rows of a warp (TokenSpeed deep dive, section 7.2,
//     fold_sq_factor): F tokens x g heads = G rows per kv head, and a
//     sequence becomes q_len / F "virtual sequences" of F tokens each. Row
//     (f, head) of virtual sequence t attends the tokens before position
//     L - q_len + t F + f + 1; only the last F - 1 tokens need a per-row mask.
//   * At the end of a sequence's segment the groups merge by LSE with shuffles
//     and lane group 0 writes either the final output (segment = whole
//     sequence) or an fp32 partial state into one of the CTA's two workspace
//     slots (first / last segment of its range). The merge kernel, launched
//     with programmatic dependent launch, reduces the split sequences.
#include <cstring>

#include "ts_paged_decode_kernel.cuh"

namespace ts {
namespace {

// Reduces the partial states of sequences cut across CTAs, one warp per
// (sequence, query row). Either every row of the batch has a warp (rows of
// sequences written whole by the main kernel are skipped), or, `compact`,
// each CTA of the main kernel has ceil(rows / 8) blocks for the one cut
// sequence whose first part it holds (split_seq): far fewer blocks when the
// batch has many more sequences than CTAs.
// In prefix mode a grouped sequence's shared-prefix state is one more part.
template <typename T, bool kPfx>
__global__ void __launch_bounds__(256) split_merge_kernel(const PagedParams p, int D, int compact) {
  pdl_wait_primary();
  pdl_launch_dependents();  // a following PDL-aware kernel may start its prologue
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  int b, hq;  // virtual sequence, query row
  int2 info;  // {first CTA, (parts << 1) | slot of first part}
  if (compact) {
    const int per_cta = (p.rows + 7) / 8 * 8;  // warps per CTA entry
    const int k = warp / per_cta;
    hq = warp % per_cta;
    if (hq >= p.rows) return;
    const int2 e = p.split_seq[k];
    if (e.x < 0) return;
    b = e.x;
    info = make_int2(k, e.y);
  } else {
    b = warp / p.rows;
    hq = warp % p.rows;
    if (b >= p.B) return;
    info = p.split_info[b];
  }
  const int nparts = info.y >> 1;
  if (nparts <= 1) return;
  const int k0 = info.x, slot0 = info.y & 1;
  const int64_t row = static_cast<int64_t>(b) * p.rows + hq;
  const bool grouped = kPfx && p.group_of[b] >= 0;
  const float lse_pre = grouped ? p.prefix_lse[row] : -INFINITY;
  float mx = lse_pre;
  for (int i = 0; i < nparts; ++i) {
    const int slot = i == 0 ? 2 * k0 + slot0 : 2 * (k0 + i);
    mx = fmaxf(mx, p.part_lse[static_cast<int64_t>(slot) * p.rows + hq]);
  }
  const float ms = mx == -INFINITY ? 0.f : mx;
  float wsum = 0.f;
  for (int d0 = lane * 4; d0 < D; d0 += 128) {
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    wsum = 0.f;
    for (int i = 0; i < nparts; ++i) {
      const int slot = i == 0 ? 2 * k0 + slot0 : 2 * (k0 + i);
      const float w = __expf(p.part_lse[static_cast<int64_t>(slot) * p.rows + hq] - ms);
      const float4 o =
          *reinterpret_cast<const float4*>(p.part_o + (static_cast<int64_t>(slot) * p.rows + hq) * D + d0);
      a.x += w * o.x;
      a.y += w * o.y;
      a.z += w * o.z;
      a.w += w * o.w;
      wsum += w;
    }
    if (grouped && lse_pre != -INFINITY) {
      const float w = __expf(lse_pre - ms);
      const float4 o = *reinterpret_cast<const float4*>(p.prefix_o + row * D + d0);
      a.x += w * o.x;
      a.y += w * o.y;
      a.z += w * o.z;
      a.w += w * o.w;
      wsum += w;
    }
    const float inv = wsum > 0.f ? 1.0f / wsum : 0.f;
    T* out = static_cast<T*>(p.out) + row * D + d0;
    if constexpr (sizeof(T) == 2) {
      uint2 pk;
      pk.x = float2_to_bf16x2(a.x * inv, a.y * inv);
      pk.y = float2_to_bf16x2(a.z * inv, a.w * inv);
      *reinterpret_cast<uint2*>(out) = pk;
    } else {
      *reinterpret_cast<float4*>(out) = make_float4(a.x * inv, a.y * inv, a.z * inv, a.w * inv);
    }
  }
  if (lane == 0 && p.lse) p.lse[row] = wsum > 0.f ? ms + logf(wsum) : -INFINITY;
}

using KernelFn = void (*)(const PagedParams);

template <typename T, int D, bool kPfx>
KernelFn pick_g(int g) {
  switch (g) {
    case 1: return paged_decode_kernel<T, D, 1, kPfx, false, false>;
    case 2: return paged_decode_kernel<T, D, 2, kPfx, false, false>;
    case 4: return paged_decode_kernel<T, D, 4, kPfx, false, false>;
    case 8: return paged_decode_kernel<T, D, 8, kPfx, false, false>;
    default: return nullptr;
  }
}

// The prefix (cascade) variants exist for bf16 only.
KernelFn pick_kernel(ts_dtype dt, int D, int g, bool prefix) {
  if (dt == TS_BF16) {
    if (D == 64) return prefix ? pick_g<__nv_bfloat16, 64, true>(g) : pick_g<__nv_bfloat16, 64, false>(g);
    if (D == 128) return prefix ? pick_g<__nv_bfloat16, 128, true>(g) : pick_g<__nv_bfloat16, 128, false>(g);
  } else if (!prefix) {
    if (D == 64) return pick_g<float, 64, false>(g);
    if (D == 128) return pick_g<float, 128, false>(g);
  }
  return nullptr;
}

constexpr int kSmemBudget = 227 * 1024;

struct WsLayout {
  size_t split_info, split_seq, part_o, part_lse, total;
};

WsLayout workspace_layout(int B, int H_q, int D, int n_ctas) {
  WsLayout w;
  size_t off = kWorkspaceAlign;  // error word + pad
  w.split_info = off;
  off = align_up(off + static_cast<size_t>(B) * sizeof(int2), kWorkspaceAlign);
  w.split_seq = off;
  off = align_up(off + static_cast<size_t>(n_ctas) * sizeof(int2), kWorkspaceAlign);
  w.part_o = off;
  off = align_up(off + static_cast<size_t>(2) * n_ctas * H_q * D * sizeof(float), kWorkspaceAlign);
  w.part_lse = off;
  off = align_up(off + static_cast<size_t>(2) * n_ctas * H_q * sizeof(float), kWorkspaceAlign);
  w.total = off;
  return w;
}

}  // namespace

// Query tokens folded into one warp's rows for q_len tokens and g query heads
// per kv head: the page's fold_sq_factor rule (largest factor F of q_len with
// g F rows in the tile, TokenSpeed deep dive section 7.2) for an 8-row tile,
// restricted to the row counts the kernel is compiled for (g F in 1, 2, 4, 8).
int gqa_fold(int g, int q_len) {
  for (int f = q_len; f >= 1; --f) {
    const int r = g * f;
    if (q_len % f == 0 && r <= 8 && (r & (r - 1)) == 0) return f;
  }
  return 1;
}

// Launches the paged split-KV kernel pair for q_len query tokens per
// sequence; `pre` non-null selects prefix (cascade) mode (q_len 1 only).
// Tensor-core path for several query tokens per sequence (ts_mq_tc.cu).
ts_status launch_fp8_decode_tc(const void* q, const void* k_pool, const void* v_pool, const float* k_scale,
                               const float* v_scale, const int32_t* block_table, int32_t bt_stride,
                               const int32_t* seq_lens, int32_t B, int32_t H_q, int32_t H_kv, int32_t D,
                               int32_t page_size, int32_t num_pages, float scale, void* out, float* lse,
                               uint32_t* err_word, cudaStream_t stream);
ts_status launch_fp8_decode_mma(const void* q, const void* k_pool, const void* v_pool, const float* k_scale,
                                const float* v_scale, const int32_t* block_table, int32_t bt_stride,
                                const int32_t* seq_lens, int32_t B, int32_t H_q, int32_t H_kv, int32_t D,
                                int32_t page_size, int32_t num_pages, float scale, void* out, float* lse,
                                void* workspace, size_t workspace_bytes, cudaStream_t stream);
ts_status launch_multi_query_tc(const void* q, const void* k_pool, const void* v_pool, const int32_t* block_table,
                                int32_t bt_stride, const int32_t* seq_lens, int32_t B, int32_t q_len, int32_t H_q,
                                int32_t H_kv, int32_t D, int32_t page_size, int32_t num_pages, float scale,
                                ts_dtype dtype, void* out, float* lse, uint32_t* err_word, cudaStream_t stream,
                                const int32_t* parents);

// Group scales of an fp8 (e4m3fn) cache, [num_pages, page_size, H_kv] each.
struct Fp8Scales {
  const float* k_scale;
  const float* v_scale;
};

ts_status paged_decode_core(const void* q, const void* k_pool, const void* v_pool,
                            const int32_t* block_table, int32_t bt_stride, const int32_t* seq_lens,
                            int32_t B, int32_t q_len, int32_t H_q, int32_t H_kv, int32_t D,
                            int32_t page_size, int32_t num_pages, float scale, ts_dtype dtype,
                            void* out, float* lse, void* workspace, size_t workspace_bytes,
                            cudaStream_t stream, const char* who, const PrefixInputs* pre,
                            const Fp8Scales* f8 = nullptr, int32_t window = 0,
                            bool check_only = false) {
  if (B < 0 || H_q <= 0 || H_kv <= 0 || D <= 0 || page_size <= 0 || num_pages <= 0 ||
      bt_stride <= 0 || static_cast<long long>(num_pages) * page_size > INT32_MAX)
    return fail(TS_ERR_INVALID_ARG, "%s: bad sizes (B=%d H_q=%d H_kv=%d D=%d ps=%d P=%d bt=%d)",
                who, B, H_q, H_kv, D, page_size, num_pages, bt_stride);
  if (q_len < 1 || (pre != nullptr && q_len != 1) ||
      static_cast<long long>(B) * q_len > INT32_MAX / 2)
    return fail(TS_ERR_INVALID_ARG, "%s: q_len=%d (>= 1; 1 with shared prefixes; B * q_len < 2^30)",
                who, q_len);
  if (H_q % H_kv != 0)
    return fail(TS_ERR_INVALID_ARG, "%s: H_q=%d not a multiple of H_kv=%d", who, H_q, H_kv);
  if (window < 0 || (window > 0 && (q_len != 1 || pre != nullptr || f8 != nullptr)))
    return fail(TS_ERR_INVALID_ARG, "%s: window=%d (>= 1, one query token, no shared prefix, no fp8)", who,
                window);
  if (dtype != TS_F32 && dtype != TS_BF16)
    return fail(TS_ERR_INVALID_ARG, "%s: bad dtype %d", who, static_cast<int>(dtype));
  if (!std::isfinite(scale)) return fail(TS_ERR_INVALID_ARG, "%s: scale not finite", who);
  if (B == 0) return TS_OK;
  if (!q || !k_pool || !v_pool || !block_table || !seq_lens || !out)
    return fail(TS_ERR_INVALID_ARG, "%s: null pointer", who);
  const int g = H_q / H_kv;
  if (H_kv > kMaxConsumerWarps || (H_kv & (H_kv - 1)) != 0)
    return fail(TS_ERR_UNSUPPORTED, "%s: H_kv=%d (supported 1, 2, 4, 8)", who, H_kv);
  if (page_size != 8 && page_size != 16 && page_size != 32)
    return fail(TS_ERR_UNSUPPORTED, "%s: page_size=%d (supported 8, 16, 32)", who, page_size);
  const int fold = (g & (g - 1)) == 0 ? gqa_fold(g, q_len) : 1;
  const int steps = q_len / fold;
  const int Bv = B * steps;           // virtual sequences
  const int rows = fold * H_q;        // query rows of a virtual sequence
  if (f8 != nullptr) {
    if (dtype != TS_BF16 || q_len != 1 || pre != nullptr || g > 4)
      return fail(TS_ERR_UNSUPPORTED, "%s: fp8 cache takes bf16 queries, one per sequence, g <= 4", who);
    if (!f8->k_scale || !f8->v_scale)
      return fail(TS_ERR_INVALID_ARG, "%s: null scale array", who);
    if (reinterpret_cast<uintptr_t>(f8->k_scale) % 16 != 0 ||
        reinterpret_cast<uintptr_t>(f8->v_scale) % 16 != 0)
      return fail(TS_ERR_INVALID_ARG, "%s: scale arrays must be 16-byte aligned", who);
  }
  KernelFn fn = f8 != nullptr ? pick_paged_fp8_kernel(D, g)
                : window > 0  ? pick_paged_window_kernel(dtype, D, g)
                : q_len == 1  ? pick_kernel(dtype, D, g, pre != nullptr)
                              : pick_paged_multi_kernel(dtype, D, g * fold);
  if (!fn)
    return fail(TS_ERR_UNSUPPORTED, "%s: D=%d, group size %d (supported D 64/128, g 1/2/4/8)", who,
                D, g);
  int g_shift = 0;
  while ((1 << g_shift) < g) ++g_shift;
  const size_t es = dtype == TS_F32 ? 4 : 2;
  for (const void* ptr : {q, k_pool, v_pool, static_cast<const void*>(out)})
    if (reinterpret_cast<uintptr_t>(ptr) % 16 != 0)
      return fail(TS_ERR_INVALID_ARG, "%s: q, pools and out must be 16-byte aligned", who);
  const int n_ctas = paged_decode_ctas();
  if (n_ctas <= 0) return fail(TS_ERR_CUDA, "%s: cannot query the SM count", who);
  const WsLayout ws = workspace_layout(Bv, rows, D, n_ctas);
  if (check_only) {
    workspace = nullptr;   // only the argument and support checks below run
  } else if (!workspace || workspace_bytes < ws.total)
    return fail(TS_ERR_WORKSPACE, "%s: workspace %zu B < %zu B needed", who, workspace_bytes,
                ws.total);
  if (reinterpret_cast<uintptr_t>(workspace) % kWorkspaceAlign != 0)
    return fail(TS_ERR_WORKSPACE, "%s: workspace must be 256-byte aligned", who);

  PagedParams prm;
  prm.q = q;
  prm.k_pool = k_pool;
  prm.v_pool = v_pool;
  prm.block_table = block_table;
  prm.seq_lens = seq_lens;
  prm.bt_stride = bt_stride;
  prm.B = Bv;
  prm.H_q = H_q;
  prm.q_len = q_len;
  prm.fold = fold;
  prm.steps = steps;
  prm.rows = rows;
  prm.g_shift = g_shift;
  prm.H_kv = H_kv;
  prm.page_size = page_size;
  prm.num_pages = num_pages;
  prm.scale_log2 = scale * kLog2e;
  prm.out = out;
  prm.lse = lse;
  prm.group_of = pre ? pre->group_of : nullptr;
  prm.prefix_len = pre ? pre->prefix_len : nullptr;
  prm.prefix_o = pre ? pre->prefix_o : nullptr;
  prm.prefix_lse = pre ? pre->prefix_lse : nullptr;
  prm.window = window;
  if (workspace != nullptr) {
    unsigned char* wsb = static_cast<unsigned char*>(workspace);
    prm.err_word = reinterpret_cast<uint32_t*>(wsb);
    prm.split_info = reinterpret_cast<int2*>(wsb + ws.split_info);
    prm.split_seq = reinterpret_cast<int2*>(wsb + ws.split_seq);
    prm.part_o = reinterpret_cast<float*>(wsb + ws.part_o);
    prm.part_lse = reinterpret_cast<float*>(wsb + ws.part_lse);
  }
  const size_t es_kv = f8 != nullptr ? 1 : es;  // K/V element bytes
  prm.row_bytes = static_cast<uint32_t>(H_kv * D * es_kv);
  prm.page_bytes = static_cast<uint32_t>(page_size) * prm.row_bytes;
  prm.q_bytes = static_cast<uint32_t>(rows * D * es);
  prm.k_scale = f8 != nullptr ? f8->k_scale : nullptr;
  prm.v_scale = f8 != nullptr ? f8->v_scale : nullptr;
  // A stage holds chunk_rows token rows of one page (all kv heads, K and V)
  // plus room for one sequence's query rows. Whole pages when two stages fit,
  // else halves, quarters... TS_PAGED_DECODE_CHUNK_ROWS overrides (tuning).
  int chunk_rows = page_size;
  if (const char* env = getenv("TS_PAGED_DECODE_CHUNK_ROWS")) {
    const int v = atoi(env);
    if (v > 0 && v <= page_size) chunk_rows = v;
  }
  // fp8: each stage also holds its rows' K and V group scales
  auto scale_of = [&](int rows) { return f8 != nullptr ? static_cast<uint32_t>(rows * H_kv * 4) : 0u; };
  auto stage_of = [&](int rows) {
    return static_cast<uint32_t>(align_up(2ull * rows * prm.row_bytes + 2ull * scale_of(rows) + prm.q_bytes, 128));
  };
  while (chunk_rows > 1 &&
         (kSmemBudget - kHeaderBytes - align_up(prm.row_bytes, 128)) / stage_of(chunk_rows) < 2)
    chunk_rows = (chunk_rows + 1) / 2;

  prm.chunk_rows = chunk_rows;
  // A sequence's fixed cost (query load, epilogue) measured on GB300 is about
  // what its consumers spend on 16 to 24 token rows; one 16-row page came out
  // best in a sweep of 0..8 units (mixed lengths at head dim 64, Llama-3-8B
  // layer at 128). TS_PAGED_DECODE_SEQ_UNITS overrides (tuning).
  {
    const int rows = 16;
    int units = std::max(1, (rows + page_size / 2) / page_size);
    if (const char* env = getenv("TS_PAGED_DECODE_SEQ_UNITS")) {
      const int v = atoi(env);
      if (v >= 0 && v <= 1024) units = v;
    }
    prm.seq_units = units;
  }
  prm.kv_area = static_cast<uint32_t>(chunk_rows) * prm.row_bytes;
  prm.scale_area = scale_of(chunk_rows);
  if (prm.scale_area % 16 != 0)
    return fail(TS_ERR_UNSUPPORTED, "%s: fp8 stage of %d rows x %d kv heads: scales not a multiple of 16 B",
                who, chunk_rows, H_kv);
  prm.stage_bytes = stage_of(chunk_rows);
  prm.stages_off = static_cast<uint32_t>(kHeaderBytes + align_up(prm.row_bytes, 128));
  const int stages = std::min<int>(kMaxStages, (kSmemBudget - prm.stages_off) / prm.stage_bytes);
  if (stages < 2 || prm.row_bytes > 4096)
    return fail(TS_ERR_UNSUPPORTED, "%s: one token row of K+V plus the query rows (%u B) exceeds the stage budget",
                who, prm.stage_bytes);
  prm.num_stages = stages;
  const size_t smem = prm.stages_off + static_cast<size_t>(stages) * prm.stage_bytes;
  // the prologue's entries: in the stage area, if they fit there
  const uint64_t stage_area = static_cast<uint64_t>(stages) * prm.stage_bytes;
  const uint64_t entries = 8ull * static_cast<uint64_t>(Bv);
  prm.len_scratch_off = entries <= stage_area ? prm.stages_off : 0u;
  // prefix mode: the groups' prefix lengths staged behind the entries
  prm.num_groups = pre ? pre->num_groups : 0;
  {
    const uint64_t at = align_up(entries, 16);
    prm.plen_scratch_off =
        (pre != nullptr && prm.len_scratch_off != 0 && pre->num_groups > 0 &&
         at + 4ull * static_cast<uint64_t>(pre->num_groups) <= stage_area)
            ? prm.stages_off + static_cast<uint32_t>(at)
            : 0u;
  }

  // Once per kernel and device: allow the whole stage budget, and check that
  // the kernel was compiled to launch with kLaunchRegs registers per thread
  // (with fewer, the consumers' setmaxnreg.inc could never be satisfied).
  ts_status st = prepare_once(reinterpret_cast<const void*>(fn), [](const void* k) {
    ts_status s2 = cuda_check(cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBudget),
                              "set smem attribute");
    if (s2 != TS_OK) return s2;
    cudaFuncAttributes fa;
    s2 = cuda_check(cudaFuncGetAttributes(&fa, k), "query kernel attributes");
    if (s2 != TS_OK) return s2;
    if (fa.numRegs < kLaunchRegs)
      return fail(TS_ERR_UNSUPPORTED, "paged decode kernel compiled with %d registers/thread, the register split "
                  "needs %d", fa.numRegs, kLaunchRegs);
    return TS_OK;
  });
  if (st != TS_OK) return st;
  if (smem > static_cast<size_t>(kSmemBudget))
    return fail(TS_ERR_UNSUPPORTED, "%s: shared memory plan %zu B exceeds %d B", who, smem, kSmemBudget);
  if (check_only) return TS_OK;

  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_ctas);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  {
    LaunchTrace trace("paged_decode_kernel", stream);
    st = cuda_check(cudaLaunchKernelEx(&cfg, fn, prm), "paged decode launch");
  }
  if (st != TS_OK) return st;

  const long long warps = static_cast<long long>(Bv) * rows;
  const long long warps_compact = static_cast<long long>(n_ctas) * ((rows + 7) / 8 * 8);
  // the per-CTA grid only where it is several times smaller (the cascade
  // suffix: 16,384 sequences); at a few hundred sequences the plain grid
  // measured as fast
  const int compact = warps_compact * 4 <= warps ? 1 : 0;
  cudaLaunchConfig_t mcfg = {};
  mcfg.gridDim = dim3(static_cast<unsigned>(((compact ? warps_compact : warps) + 7) / 8));
  mcfg.blockDim = dim3(256);
  mcfg.dynamicSmemBytes = 0;
  mcfg.stream = stream;
  mcfg.attrs = attr;
  mcfg.numAttrs = 1;
  LaunchTrace trace("split_merge_kernel", stream);
  if (dtype == TS_BF16)
    st = cuda_check(cudaLaunchKernelEx(&mcfg,
                                       pre ? split_merge_kernel<__nv_bfloat16, true>
                                           : split_merge_kernel<__nv_bfloat16, false>,
                                       prm, D, compact),
                    "split merge launch");
  else
    st = cuda_check(cudaLaunchKernelEx(&mcfg, split_merge_kernel<float, false>, prm, D, compact),
                    "split merge launch");
  return st;
}

ts_status launch_paged_decode_impl(const void* q, const void* k_pool, const void* v_pool,
                                   const int32_t* block_table, int32_t bt_stride,
                                   const int32_t* seq_lens, int32_t B, int32_t H_q, int32_t H_kv,
                                   int32_t D, int32_t page_size, int32_t num_pages, float scale,
                                   ts_dtype dtype, void* out, float* lse, void* workspace,
                                   size_t workspace_bytes, cudaStream_t stream, const char* who,
                                   const PrefixInputs* pre) {
  return paged_decode_core(q, k_pool, v_pool, block_table, bt_stride, seq_lens, B, 1, H_q, H_kv, D,
                           page_size, num_pages, scale, dtype, out, lse, workspace, workspace_bytes,
                           stream, who, pre);
}

ts_status launch_paged_decode_fp8(const void* q, const void* k_pool, const void* v_pool,
                                  const float* k_scale, const float* v_scale,
                                  const int32_t* block_table, int32_t bt_stride, const int32_t* seq_lens,
                                  int32_t B, int32_t H_q, int32_t H_kv, int32_t D, int32_t page_size,
                                  int32_t num_pages, float scale, void* out, float* lse, void* workspace,
                                  size_t workspace_bytes, cudaStream_t stream) {
  const Fp8Scales f8{k_scale, v_scale};
  return paged_decode_core(q, k_pool, v_pool, block_table, bt_stride, seq_lens, B, 1, H_q, H_kv, D,
                           page_size, num_pages, scale, TS_BF16, out, lse, workspace, workspace_bytes,
                           stream, "ts_paged_decode_fp8_attn", nullptr, &f8);
}

ts_status launch_paged_decode(const void* q, const void* k_pool, const void* v_pool,
                              const int32_t* block_table, int32_t bt_stride,
                              const int32_t* seq_lens, int32_t B, int32_t H_q, int32_t H_kv,
                              int32_t D, int32_t page_size, int32_t num_pages, float scale,
                              ts_dtype dtype, void* out, float* lse, void* workspace,
                              size_t workspace_bytes, cudaStream_t stream, const char* who) {
  return launch_paged_decode_impl(q, k_pool, v_pool, block_table, bt_stride, seq_lens, B, H_q,
                                  H_kv, D, page_size, num_pages, scale, dtype, out, lse, workspace,
                                  workspace_bytes, stream, who, nullptr);
}

// Every argument and support check of ts_paged_decode_attn except the
// workspace's; enqueues nothing.
ts_status paged_decode_check_args(const void* q, const void* k_pool, const void* v_pool,
                                  const int32_t* block_table, int32_t bt_stride,
                                  const int32_t* seq_lens, int32_t B, int32_t H_q, int32_t H_kv,
                                  int32_t D, int32_t page_size, int32_t num_pages, float scale,
                                  ts_dtype dtype, void* out, const char* who) {
  return paged_decode_core(q, k_pool, v_pool, block_table, bt_stride, seq_lens, B, 1, H_q, H_kv, D,
                           page_size, num_pages, scale, dtype, out, nullptr, nullptr, 0, nullptr,
                           who, nullptr, nullptr, 0, true);
}

size_t paged_decode_workspace_bytes(int B, int H_q, int D) {
  const int n = paged_decode_ctas();
  if (n <= 0 || B < 0 || H_q <= 0 || D <= 0) return 0;
  return workspace_layout(B, H_q, D, n).total;
}

// Upper bound over the fold: at most B * q_len virtual sequences of at most
// q_len * H_q rows.
size_t paged_decode_multi_workspace_bytes(int B, int q_len, int H_q, int D) {
  const int n = paged_decode_ctas();
  if (n <= 0 || B < 0 || q_len < 1 || H_q <= 0 || D <= 0 ||
      static_cast<long long>(B) * q_len > INT32_MAX / 2)
    return 0;
  return workspace_layout(B * q_len, q_len * H_q, D, n).total;
}

}  // namespace ts

extern "C" size_t ts_paged_decode_workspace_size(int32_t B, int32_t H_q, int32_t D) {
  return ts::paged_decode_workspace_bytes(B, H_q, D);
}

extern "C" ts_status ts_paged_decode_attn(const void* q, const void* k_pool, const void* v_pool,
                                          const int32_t* block_table, int32_t bt_stride,
                                          const int32_t* seq_lens, int32_t B, int32_t H_q,
                                          int32_t H_kv, int32_t D, int32_t page_size,
                                          int32_t num_pages, float scale, ts_dtype dtype,
                                          void* out, float* lse, void* workspace,
                                          size_t workspace_bytes, void* stream) {
  return ts::launch_paged_decode(q, k_pool, v_pool, block_table, bt_stride, seq_lens, B, H_q, H_kv,
                                 D, page_size, num_pages, scale, dtype, out, lse, workspace,
                                 workspace_bytes, static_cast<cudaStream_t>(stream),
                                 "ts_paged_decode_attn");
}

extern "C" ts_status ts_paged_decode_window_attn(const void* q, const void* k_pool, const void* v_pool,
                                                 const int32_t* block_table, int32_t bt_stride,
                                                 const int32_t* seq_lens, int32_t B, int32_t H_q,
                                                 int32_t H_kv, int32_t D, int32_t page_size,
                                                 int32_t num_pages, int32_t window, float scale,
                                                 ts_dtype dtype, void* out, float* lse, void* workspace,
                                                 size_t workspace_bytes, void* stream) {
  const char* who = "ts_paged_decode_window_attn";
  if (window < 1) return ts::fail(TS_ERR_INVALID_ARG, "%s: window=%d (>= 1 token)", who, window);
  return ts::paged_decode_core(q, k_pool, v_pool, block_table, bt_stride, seq_lens, B, 1, H_q, H_kv, D,
                               page_size, num_pages, scale, dtype, out, lse, workspace, workspace_bytes,
                               static_cast<cudaStream_t>(stream), who, nullptr, nullptr, window);
}

extern "C" size_t ts_paged_decode_multi_workspace_size(int32_t B, int32_t q_len, int32_t H_q, int32_t D) {
  return ts::paged_decode_multi_workspace_bytes(B, q_len, H_q, D);
}

extern "C" ts_status ts_paged_decode_multi_attn(const void* q, const void* k_pool, const void* v_pool,
                                                const int32_t* block_table, int32_t bt_stride,
                                                const int32_t* seq_lens, int32_t B, int32_t q_len,
                                                int32_t H_q, int32_t H_kv, int32_t D,
                                                int32_t page_size, int32_t num_pages, float scale,
                                                ts_dtype dtype, void* out, float* lse,
                                                void* workspace, size_t workspace_bytes,
                                                void* stream) {
  // From 8 query rows per kv head (q_len x g) one CTA per (sequence, kv
  // head) runs them on tcgen05 when the shape allows it; the CUDA-core kernel
  // keeps at most 8 rows in registers per pass and is the slower of the two
  // there (Llama-3-8B layer shape, B=64: 2 tokens x 4 heads 140 us against
  // 190 us, 4 x 4 140 us against 367 us). Fewer rows stay on the CUDA-core
  // kernel. TS_MULTI_QUERY_PATH=cuda / =tensor forces one path (tests
  // compare both).
  const char* path = getenv("TS_MULTI_QUERY_PATH");
  const bool force_cuda = path && std::strcmp(path, "cuda") == 0;
  const bool force_tc = path && std::strcmp(path, "tensor") == 0;
  const int rows_per_kv = H_kv > 0 && H_q % H_kv == 0 ? q_len * (H_q / H_kv) : 0;
  if (!force_cuda && (force_tc || rows_per_kv >= 8) && q_len >= 2 && B > 0 && H_q > 0 && H_kv > 0 &&
      H_q % H_kv == 0 && q && k_pool && v_pool &&
      block_table && seq_lens && out && bt_stride > 0 && num_pages > 0 &&
      static_cast<long long>(num_pages) * page_size <= INT32_MAX && std::isfinite(scale) &&
      reinterpret_cast<uintptr_t>(q) % 16 == 0 && reinterpret_cast<uintptr_t>(out) % 16 == 0 &&
      reinterpret_cast<uintptr_t>(k_pool) % 16 == 0 && reinterpret_cast<uintptr_t>(v_pool) % 16 == 0) {
    const size_t need = ts::paged_decode_multi_workspace_bytes(B, q_len, H_q, D);
    if (!workspace || need == 0 || workspace_bytes < need ||
        reinterpret_cast<uintptr_t>(workspace) % ts::kWorkspaceAlign != 0)
      return ts::fail(TS_ERR_WORKSPACE, "ts_paged_decode_multi_attn: workspace %zu B < %zu B needed or misaligned",
                      workspace_bytes, need);
    const ts_status st = ts::launch_multi_query_tc(q, k_pool, v_pool, block_table, bt_stride, seq_lens, B, q_len,
                                                   H_q, H_kv, D, page_size, num_pages, scale, dtype, out, lse,
                                                   static_cast<uint32_t*>(workspace),
                                                   static_cast<cudaStream_t>(stream), nullptr);
    if (st != TS_ERR_UNSUPPORTED) return st;
  }
  return ts::paged_decode_core(q, k_pool, v_pool, block_table, bt_stride, seq_lens, B, q_len, H_q,
                               H_kv, D, page_size, num_pages, scale, dtype, out, lse, workspace,
                               workspace_bytes, static_cast<cudaStream_t>(stream),
                               "ts_paged_decode_multi_attn", nullptr);
}

extern "C" ts_status ts_paged_decode_tree_attn(const void* q, const void* k_pool, const void* v_pool,
                                               const int32_t* block_table, int32_t bt_stride,
                                               const int32_t* seq_lens, const int32_t* parents, int32_t B,
                                               int32_t n, int32_t H_q, int32_t H_kv, int32_t D,
                                               int32_t page_size, int32_t num_pages, float scale,
                                               ts_dtype dtype, void* out, float* lse, void* workspace,
                                               size_t workspace_bytes, void* stream) {
  using namespace ts;
  const char* who = "ts_paged_decode_tree_attn";
  if (B < 0 || n < 1 || H_q <= 0 || H_kv <= 0 || D <= 0 || page_size <= 0 || num_pages <= 0 || bt_stride <= 0 ||
      H_q % H_kv != 0 || static_cast<long long>(num_pages) * page_size > INT32_MAX)
    return fail(TS_ERR_INVALID_ARG, "%s: bad sizes (B=%d n=%d H_q=%d H_kv=%d D=%d ps=%d P=%d bt=%d)", who, B, n,
                H_q, H_kv, D, page_size, num_pages, bt_stride);
  if (dtype != TS_F32 && dtype != TS_BF16)
    return fail(TS_ERR_INVALID_ARG, "%s: bad dtype %d", who, static_cast<int>(dtype));
  if (!std::isfinite(scale)) return fail(TS_ERR_INVALID_ARG, "%s: scale not finite", who);
  if (B == 0) return TS_OK;
  if (!q || !k_pool || !v_pool || !block_table || !seq_lens || !parents || !out)
    return fail(TS_ERR_INVALID_ARG, "%s: null pointer", who);
  for (const void* ptr : {q, k_pool, v_pool, static_cast<const void*>(out)})
    if (reinterpret_cast<uintptr_t>(ptr) % 16 != 0)
      return fail(TS_ERR_INVALID_ARG, "%s: q, pools and out must be 16-byte aligned", who);
  if (!workspace || workspace_bytes < kWorkspaceAlign ||
      reinterpret_cast<uintptr_t>(workspace) % kWorkspaceAlign != 0)
    return fail(TS_ERR_WORKSPACE, "%s: workspace of >= 256 bytes, 256-byte aligned, needed", who);
  const ts_status st = launch_multi_query_tc(q, k_pool, v_pool, block_table, bt_stride, seq_lens, B, n, H_q, H_kv,
                                             D, page_size, num_pages, scale, dtype, out, lse,
                                             static_cast<uint32_t*>(workspace), static_cast<cudaStream_t>(stream),
                                             parents);
  if (st == TS_ERR_UNSUPPORTED)
    return fail(TS_ERR_UNSUPPORTED, "%s: needs bf16, page_size 16, D 64/128, n <= 64, n * H_q / H_kv <= 128 "
                "(got dtype %d, ps %d, D %d, n %d, g %d)", who, static_cast<int>(dtype), page_size, D, n,
                H_q / H_kv);
  return st;
}

extern "C" int32_t ts_fold_sq_factor(int32_t num_heads, int32_t q_len, int32_t tile_rows) {
  if (num_heads <= 0 || q_len <= 0 || tile_rows <= 0) return 0;
  int32_t best = 1;
  for (int32_t f = 1; f <= q_len; ++f)
    if (q_len % f == 0 && static_cast<long long>(num_heads) * f <= tile_rows) best = f;
  return best;
}

extern "C" ts_status ts_paged_decode_fp8_attn(const void* q, const void* k_pool, const void* v_pool,
                                              const float* k_scale, const float* v_scale,
                                              const int32_t* block_table, int32_t bt_stride,
                                              const int32_t* seq_lens, int32_t B, int32_t H_q,
                                              int32_t H_kv, int32_t D, int32_t page_size,
                                              int32_t num_pages, float scale, void* out, float* lse,
                                              void* workspace, size_t workspace_bytes, void* stream) {
  // The CUDA-core split-KV kernel, unless TS_FP8_DECODE_PATH asks for one of
  // the tensor-core kernels (=mma: the code-multiplying one, =tensor: the
  // widening one) and the shape suits it; arguments the tensor-core kernels
  // cannot judge are left to the CUDA-core path's checks.
  if (B > 0 && H_q > 0 && H_kv > 0 && q && k_pool && v_pool && k_scale && v_scale && block_table && seq_lens &&
      out && std::isfinite(scale) && reinterpret_cast<uintptr_t>(q) % 16 == 0 &&
      reinterpret_cast<uintptr_t>(out) % 16 == 0 && reinterpret_cast<uintptr_t>(k_pool) % 16 == 0 &&
      reinterpret_cast<uintptr_t>(v_pool) % 16 == 0 && reinterpret_cast<uintptr_t>(k_scale) % 16 == 0 &&
      reinterpret_cast<uintptr_t>(v_scale) % 16 == 0) {
    const size_t need = ts::paged_decode_workspace_bytes(B, H_q, D);
    if (!workspace || need == 0 || workspace_bytes < need ||
        reinterpret_cast<uintptr_t>(workspace) % ts::kWorkspaceAlign != 0)
      return ts::fail(TS_ERR_WORKSPACE, "ts_paged_decode_fp8_attn: workspace %zu B < %zu B needed or misaligned",
                      workspace_bytes, need);
    ts_status st = ts::launch_fp8_decode_mma(q, k_pool, v_pool, k_scale, v_scale, block_table, bt_stride,
                                             seq_lens, B, H_q, H_kv, D, page_size, num_pages, scale, out, lse,
                                             workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
    if (st != TS_ERR_UNSUPPORTED) return st;
    st = ts::launch_fp8_decode_tc(q, k_pool, v_pool, k_scale, v_scale, block_table, bt_stride, seq_lens, B, H_q,
                                  H_kv, D, page_size, num_pages, scale, out, lse, static_cast<uint32_t*>(workspace),
                                  static_cast<cudaStream_t>(stream));
    if (st != TS_ERR_UNSUPPORTED) return st;
  }
  return ts::launch_paged_decode_fp8(q, k_pool, v_pool, k_scale, v_scale, block_table, bt_stride,
                                     seq_lens, B, H_q, H_kv, D, page_size, num_pages, scale, out, lse,
                                     workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
}
