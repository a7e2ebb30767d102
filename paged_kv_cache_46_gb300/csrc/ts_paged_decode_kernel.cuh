// Device code of the paged split-KV decode kernel, shared by the two
// translation units that instantiate it: ts_paged_decode.cu (one query token
// per sequence, and the shared-prefix mode) and ts_paged_decode_multi.cu
// (several query tokens per sequence). See ts_paged_decode.cu for the design.
#pragma once

#include <cmath>
#include <cstdlib>
#include <type_traits>

#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "ts_common.cuh"

namespace ts {

struct StageDesc {
  int32_t b;         // virtual sequence
  int32_t valid;     // tokens present in this page
  uint32_t flags;    // kFlag*
  int32_t out_slot;  // -1: write the final output; else partial slot index
  int32_t rem;       // tokens from this stage's first row to the virtual sequence's end
};

struct PagedParams {
  const void* q;
  const void* k_pool;
  const void* v_pool;
  const int32_t* block_table;
  const int32_t* seq_lens;
  // B counts virtual sequences: (sequence, step) pairs, `steps` per sequence,
  // each holding `fold` consecutive query tokens (rows = fold * H_q query
  // rows; row f * H_q + head). A warp's G = g * fold rows: g = 2^g_shift.
  int32_t bt_stride, B, H_q, H_kv, page_size, num_pages;
  int32_t q_len, fold, steps, rows, g_shift;
  float scale_log2;  // scale * log2(e)
  void* out;
  float* lse;
  uint32_t* err_word;
  int2* split_info;  // per virtual sequence: {first CTA, (parts << 1) | slot of first part}
  // per CTA: {the cut sequence whose first part it holds (or -1), its
  // (parts << 1) | slot of first part} (its first CTA is this one)
  int2* split_seq;
  float* part_o;     // [2 * gridDim.x, rows, D]
  float* part_lse;   // [2 * gridDim.x, rows]
  // Shared-prefix (cascade) mode: a grouped sequence's own pages start after
  // its group's prefix pages, and the prefix attention state is merged in.
  const int32_t* group_of;    // [B] group or -1
  const int32_t* prefix_len;  // [groups] shared tokens (whole pages)
  const float* prefix_o;      // [B, H_q, D] normalised prefix output (fp32)
  const float* prefix_lse;    // [B, H_q] prefix LSE (natural log)
  int32_t num_stages;
  uint32_t stage_bytes;  // bytes per stage (K rows + V rows + q rows, aligned)
  uint32_t stages_off;   // offset of the first stage in dynamic shared memory
  uint32_t page_bytes;   // bytes of one full page of K (or V), all kv heads
  int32_t chunk_rows;    // token rows per stage (a page, or a contiguous part of one)
  int32_t seq_units;     // work units a sequence costs beyond its pages (its q load and epilogue)
  uint32_t kv_area;      // chunk_rows * row_bytes: K (and V) area of a stage
  uint32_t row_bytes;    // bytes of one token row of K (or V), all kv heads
  uint32_t q_bytes;      // bytes of one virtual sequence's query rows
  // fp8 (e4m3fn) cache: one float32 scale per (page, row, kv head) for K and
  // for V ([num_pages, page_size, H_kv]); a stage holds its rows' scales
  // (scale_area bytes each) after the V rows. nullptr / 0 otherwise.
  const float* k_scale;
  const float* v_scale;
  uint32_t scale_area;
  // Sliding-window KV group (plain decode only): a sequence attends its last
  // `window` tokens; 0 = the whole context.
  int32_t window = 0;
  // Byte offset in dynamic shared memory where the prologue keeps an int2 [B]
  // array of each virtual sequence's (own length, tokens in front of its own
  // pages) while it cuts the batch: the stage area, free until the producer's
  // first copy; 0 = the entries do not fit there (read from global memory).
  uint32_t len_scratch_off = 0;
  // Prefix mode: entries of prefix_len, and where the prologue stages them in
  // the stage area for its gather (0: read from global memory).
  int32_t num_groups = 0;
  uint32_t plen_scratch_off = 0;
};

using PagedKernelFn = void (*)(const PagedParams);
// Kernel for several query tokens per sequence with G rows per kv head
// (defined in ts_paged_decode_multi.cu); nullptr if not compiled.
PagedKernelFn pick_paged_multi_kernel(ts_dtype dt, int D, int G);
// Kernel for an fp8 (e4m3fn) cache with bf16 queries and G rows per kv head
// (defined in ts_paged_decode_fp8.cu); nullptr if not compiled.
PagedKernelFn pick_paged_fp8_kernel(int D, int G);
// Kernel for a sliding-window KV group with G rows per kv head (defined in
// ts_paged_decode_window.cu); nullptr if not compiled.
PagedKernelFn pick_paged_window_kernel(ts_dtype dt, int D, int G);

namespace {

constexpr int kMaxConsumerWarps = 8;
// Three warp groups: group 0 holds the producer (warp 0; warps 1-3 leave after
// the prologue), groups 1-2 hold the consumer warps (warp 4 + kv head).
// Register split: launched at kLaunchRegs per thread; the producer group gives
// registers back (setmaxnreg.dec, RegSplit) and the consumer groups take
// them (setmaxnreg.inc): 128*56 + 256*224 == 384*168, or
// 128*40 + 256*232 == 384*168 for group size 8.
constexpr int kThreads = 384;
constexpr int kFirstConsumerWarp = 4;
constexpr int kLaunchRegs = 168;
// Group size 8 keeps twice the query/accumulator registers per lane pair and
// takes the larger consumer share.
template <int G>
struct RegSplit {
  static constexpr int kProducer = G >= 8 ? 40 : 56;
  static constexpr int kConsumer = G >= 8 ? 232 : 224;
  static_assert(128 * kProducer + 256 * kConsumer <= kThreads * kLaunchRegs,
                "register split exceeds the launch allocation");
};
constexpr int kMaxStages = 8;
constexpr int kHeaderBytes = 1024;
constexpr int kZeroRowOff = kHeaderBytes;  // one zeroed token row (<= 4 KB)
constexpr uint32_t kFlagFirst = 1u, kFlagLast = 2u, kFlagEnd = 4u, kFlagBadPage = 8u;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// Largest score excess over the reference max (log2 units) before the
// accumulators are rescaled: unnormalised weights stay <= 2^8.
constexpr float kRescaleSlack = 8.0f;



template <typename T>
struct Elem;
template <>
struct Elem<float> {
  static constexpr int kVE = 4;  // elements per 16-byte vector
  // Converts word pair w (of a 16-byte vector) to a float2.
  __device__ static __forceinline__ float2 pair(const uint4& v, int w) {
    const uint32_t a = w == 0 ? v.x : v.z;
    const uint32_t b = w == 0 ? v.y : v.w;
    return make_float2(__uint_as_float(a), __uint_as_float(b));
  }
  static constexpr int kPairs = 2;  // float2 pairs per vector
};
template <>
struct Elem<__nv_bfloat16> {
  static constexpr int kVE = 8;
  __device__ static __forceinline__ float2 pair(const uint4& v, int w) {
    const uint32_t x = w == 0 ? v.x : (w == 1 ? v.y : (w == 2 ? v.z : v.w));
    return bf16x2_to_float2(x);
  }
  static constexpr int kPairs = 4;
};
// e4m3fn codes of an fp8 cache: pair w is bytes 2w, 2w+1, widened exactly
// (e4m3 -> f16 -> f32 by the conversion instructions).
template <>
struct Elem<uint8_t> {
  static constexpr int kVE = 16;
  __device__ static __forceinline__ float2 pair(const uint4& v, int w) {
    const uint32_t x = (w >> 1) == 0 ? v.x : ((w >> 1) == 1 ? v.y : ((w >> 1) == 2 ? v.z : v.w));
    const __nv_fp8x2_storage_t c = static_cast<__nv_fp8x2_storage_t>((w & 1) ? (x >> 16) : (x & 0xffffu));
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(c, __NV_E4M3);
    return __half22float2(__half2(h));
  }
  static constexpr int kPairs = 8;
};

__device__ __forceinline__ float lds_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

template <typename T, int D, int G>
struct Cfg {
  static constexpr int kES = sizeof(T);
  static constexpr int kVE = Elem<T>::kVE;
  static constexpr int kDPL = (G <= 4) ? 16 : 8;        // dims per lane
  static constexpr int kNV = kDPL / kVE;                // 16-byte vectors per lane
  static constexpr int kLPT = D / kDPL;                 // lanes per token
  static constexpr int kNG = 32 / kLPT;                 // token groups per warp
  static constexpr int kTPG0 = 16 / kNG;
  static constexpr int kTPG = (kTPG0 * G > 16) ? (16 / G) : kTPG0;  // tokens per group per pass
  static constexpr int kPairsPL = kDPL / 2;             // float2 per lane per head
  static_assert(kLPT >= 2 && kLPT <= 32 && (32 % kLPT) == 0, "lane split");
  static_assert(kTPG >= 1, "tokens per group");
};

// Tokens of sequence b covered by its group's shared prefix (prefix mode).
template <bool kPfx>
__device__ __forceinline__ int prefix_tokens(const PagedParams& p, int b) {
  if constexpr (kPfx) {
    const int g = p.group_of[b];
    return g >= 0 ? p.prefix_len[g] : 0;
  } else {
    return 0;
  }
}

// Sequence (block-table row) of virtual sequence v. Without several query
// tokens (kMulti false) virtual and real sequences coincide.
template <bool kMulti>
__device__ __forceinline__ int real_seq(const PagedParams& p, int v) {
  if constexpr (kMulti) return p.steps == 1 ? v : v / p.steps;
  return v;
}

// Tokens in the whole pages in front of a sliding window (TokenSpeed deep
// dive, section 4.1: a sliding_window KV group; tokenspeed 딥다이브, section
// 6-3: the slots in front of the window hold a placeholder block). Their
// block-table slots are skipped, never read.
template <bool kWin>
__device__ __forceinline__ int window_skip(const PagedParams& p, int v) {
  if constexpr (!kWin) {
    return 0;
  } else {
    const int L = p.seq_lens[v];
    return L > p.window ? (L - p.window) & -p.page_size : 0;  // page_size: a power of two
  }
}

// Own tokens of virtual sequence v: those its last row attends (after the
// shared prefix in prefix mode, where every sequence has one query token).
// With a sliding window: the tokens from the window's first page on (its
// rows in front of the window are not copied).
template <bool kPfx, bool kMulti, bool kWin>
__device__ __forceinline__ int vseq_len(const PagedParams& p, int v) {
  if constexpr (kMulti) {
    const int b = real_seq<kMulti>(p, v);
    return p.seq_lens[b] - p.q_len + (v - b * p.steps + 1) * p.fold;
  } else {
    return p.seq_lens[v] - prefix_tokens<kPfx>(p, v) - window_skip<kWin>(p, v);
  }
}

// vseq_len, also returning the tokens in front of the sequence's own pages
// (its shared prefix, or the whole pages in front of its window).
template <bool kPfx, bool kMulti, bool kWin>
__device__ __forceinline__ int vseq_len_pre(const PagedParams& p, int v, int& pre) {
  if constexpr (kMulti) {
    pre = 0;
    return vseq_len<kPfx, kMulti, kWin>(p, v);
  } else {
    pre = prefix_tokens<kPfx>(p, v) + window_skip<kWin>(p, v);
    return p.seq_lens[v] - pre;
  }
}

// Writes the output of a virtual sequence with no own tokens: O = 0,
// LSE = -inf, or the prefix state alone in prefix mode. All 32 lanes of a
// warp call it together; their stores are coalesced.
template <typename T, bool kPfx>
__device__ void write_empty_sequence(const PagedParams& p, int D, int b, int k, int lane) {
  const bool grouped = kPfx && p.group_of[b] >= 0;
  T* out = static_cast<T*>(p.out) + static_cast<int64_t>(b) * p.rows * D;
  const float* po = grouped ? p.prefix_o + static_cast<int64_t>(b) * p.rows * D : nullptr;
  for (int i = lane; i < p.rows * D; i += 32) out[i] = static_cast<T>(grouped ? po[i] : 0.0f);
  if (p.lse)
    for (int h = lane; h < p.rows; h += 32)
      p.lse[static_cast<int64_t>(b) * p.rows + h] =
          grouped ? p.prefix_lse[static_cast<int64_t>(b) * p.rows + h] : -INFINITY;
  if (lane == 0) p.split_info[b] = make_int2(k, 0);
}

template <typename T, int D, int G, bool kPfx, bool kMulti, bool kFp8, bool kWin = false>
__global__ void __launch_bounds__(kThreads, 1) paged_decode_kernel(const PagedParams p) {
  static_assert(!(kPfx && kMulti), "shared prefixes take one query token per sequence");
  static_assert(!kWin || (!kPfx && !kMulti && !kFp8), "sliding windows: plain decode");
  static_assert(!kFp8 || (G <= 4 && sizeof(T) == 2 && !kPfx), "fp8 cache: bf16 queries, up to 4 rows");
  // K/V element type (the lane split follows it); T is the query / output type
  using KV = std::conditional_t<kFp8, uint8_t, T>;
  using C = Cfg<KV, D, G>;
  extern __shared__ __align__(1024) unsigned char smem[];
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int n_consumer = p.H_kv;  // one consumer warp per kv head
  const int nwarps = blockDim.x >> 5;
  const int k = blockIdx.x;
  const int G_ctas = gridDim.x;
  const int ps = p.page_size;
  const int S = p.num_stages;

  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = reinterpret_cast<uint64_t*>(smem + 64);
  StageDesc* desc = reinterpret_cast<StageDesc*>(smem + 128);
  long long* warp_tot = reinterpret_cast<long long*>(smem + 512);
  int* s_start = reinterpret_cast<int*>(smem + 640);  // b0, p0
  int2* s_pro = p.len_scratch_off != 0 ? reinterpret_cast<int2*>(smem + p.len_scratch_off) : nullptr;
  unsigned char* stages = smem + p.stages_off;

  // Programmatic dependent launch: this kernel may start while the previous
  // kernel of the stream finishes. Until griddepcontrol.wait it only reads
  // seq_lens, the block table and the prefix-group metadata; every other read
  // and every global write comes after the wait.
  pdl_launch_dependents();

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), n_consumer);
    }
    s_start[0] = -1;
    s_start[1] = 0;
    fence_mbar_init();
  }
  // A row of zeros that masked rows of empty units read instead of the stage.
  for (int i = tid; i < static_cast<int>(p.row_bytes / 4); i += blockDim.x)
    reinterpret_cast<uint32_t*>(smem + kZeroRowOff)[i] = 0u;

  // ---- prologue: total pages T and this CTA's range [start, end) ----------
  const int B = p.B;
  const int chunk = (B + blockDim.x - 1) / blockDim.x;
  const int lo = min(B, tid * chunk), hi = min(B, lo + chunk);
  // Work units: a sequence with np > 0 own pages counts np + seq_units, the
  // first seq_units standing for its fixed cost (query load, epilogue); they
  // carry no page. The units of the batch are cut evenly across the CTAs.
  const int A = p.seq_units;
  long long mine = 0;
  bool has_empty = false;
  // More sequences than threads: gather the entries first with consecutive
  // threads on consecutive sequences (coalesced, independent loads), then sum
  // each thread's contiguous chunk from shared memory.
  const bool gathered = s_pro != nullptr && B > static_cast<int>(blockDim.x);
  if (gathered) {
    // prefix mode: the groups' prefix lengths first, so that each sequence's
    // entry needs only independent loads (its length and its group)
    const int* s_plen = nullptr;
    if constexpr (kPfx) {
      if (p.plen_scratch_off != 0) {
        int* w = reinterpret_cast<int*>(smem + p.plen_scratch_off);
        for (int g = tid; g < p.num_groups; g += blockDim.x) w[g] = p.prefix_len[g];
        __syncthreads();
        s_plen = w;
      }
    }
    // eight sequences per thread at a time: all their loads are issued before
    // any entry is stored (stores through a generic pointer would otherwise
    // keep the next loads waiting)
    constexpr int kBatch = 8;
    const int nthr = static_cast<int>(blockDim.x);
    for (int b0 = tid; b0 < B; b0 += kBatch * nthr) {
      int raw[kBatch], grp[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int b = b0 + u * nthr;
        raw[u] = b < B ? p.seq_lens[real_seq<kMulti>(p, b)] : 0;
        grp[u] = (kPfx && b < B) ? p.group_of[b] : -1;
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int b = b0 + u * nthr;
        if (b >= B) break;
        int pre = 0, L;
        if constexpr (kMulti) {
          L = raw[u] - p.q_len + (b - real_seq<kMulti>(p, b) * p.steps + 1) * p.fold;
        } else {
          if constexpr (kPfx) {
            const int g = grp[u];
            pre = g < 0 ? 0 : (s_plen != nullptr ? (g < p.num_groups ? s_plen[g] : 0) : p.prefix_len[g]);
          }
          if constexpr (kWin) pre += raw[u] > p.window ? (raw[u] - p.window) & -p.page_size : 0;
          L = raw[u] - pre;
        }
        s_pro[b] = make_int2(L, pre);
      }
    }
    __syncthreads();
  }
  for (int b = lo; b < hi; ++b) {
    int L;
    if (gathered) {
      L = s_pro[b].x;
    } else {
      int pre;
      L = vseq_len_pre<kPfx, kMulti, kWin>(p, b, pre);
      if (s_pro != nullptr) s_pro[b] = make_int2(L, pre);
    }
    if (L > 0)
      mine += (L + ps - 1) / ps + A;
    else if (b % G_ctas == k)
      has_empty = true;
  }
  // Sequences with no own tokens are written here, after the wait, each by a
  // whole warp: the lanes that found some take turns handing their range to
  // the warp (every thread runs this prologue, so the warps are converged).
  unsigned todo = __ballot_sync(0xffffffffu, has_empty);
  if (todo != 0u) {
    pdl_wait_primary();
    while (todo != 0u) {
      const int src = __ffs(todo) - 1;
      todo &= todo - 1u;
      const int slo = __shfl_sync(0xffffffffu, lo, src), shi = __shfl_sync(0xffffffffu, hi, src);
      for (int b = slo; b < shi; ++b)
        if (vseq_len<kPfx, kMulti, kWin>(p, b) <= 0 && b % G_ctas == k)
          write_empty_sequence<T, kPfx>(p, D, b, k, lane);
    }
  }
  long long incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  long long wbase = 0, total = 0;
  for (int w = 0; w < nwarps; ++w) {
    const long long v = warp_tot[w];
    if (w < warp) wbase += v;
    total += v;
  }
  const long long excl = wbase + incl - mine;
  // Balanced cut: the first (total % G) CTAs take one page more. Non-empty
  // ranges are contiguous, so a sequence's pages always lie in consecutive
  // non-empty CTAs (the merge relies on it).
  const long long q_pages = total / G_ctas, r_pages = total % G_ctas;
  const long long start = k * q_pages + min(static_cast<long long>(k), r_pages);
  const long long end = start + q_pages + (k < r_pages ? 1 : 0);
  if (start < end && excl <= start && start < excl + mine) {
    long long off = excl;
    for (int b = lo; b < hi; ++b) {  // entries this thread wrote, or gathered before a barrier
      const int L = s_pro != nullptr ? s_pro[b].x : vseq_len<kPfx, kMulti, kWin>(p, b);
      const long long np = L > 0 ? (L + ps - 1) / ps + A : 0;
      if (start < off + np) {
        s_start[0] = b;
        s_start[1] = static_cast<int>(start - off);
        break;
      }
      off += np;
    }
  }
  // the stage area's scratch entries are read through the generic proxy; the
  // producer's bulk copies (async proxy) overwrite them after this barrier
  if (s_pro != nullptr) fence_async_smem();
  __syncthreads();

  if (warp < kFirstConsumerWarp) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(RegSplit<G>::kProducer));
    if (warp != 0) return;
    // ======================= producer warp ================================
    int it = 0;
    int ps_stage = 0, ps_phase = 0;  // it % S and (it / S) & 1, kept incrementally
    bool aborted = false;
    if (start < end && s_start[0] >= 0) {
      const uint64_t pol = policy_evict_first();
      // The range is walked in chunks of up to 32 pages of one sequence. The
      // metadata of the next chunk (sequence lengths, 32 lengths per warp load,
      // and the chunk's block-table entries, one per lane) is loaded while the
      // current chunk's pages are issued, so a sequence boundary costs no
      // dependent global-load latency in the copy stream.
      long long g = start;   // global index of the next work unit
      int b = s_start[0];    // sequence of the next unit
      int pg = s_start[1];   // its unit index within the sequence (pages start at unit A;
                             // within a segment pg counts pages)
      bool first_seg = true;
      int seg_left = 0, seg_L = 0, seg_np = 0, seg_pre = 0, seg_slot = -1;
      int wb = b;                                   // lengths window: sequences wb .. wb+31
      auto load_len = [&](int base, int& pre_out) {  // this lane's sequence base+lane
        const int bb = base + lane;
        pre_out = 0;
        if (bb >= B) return -1;
        pre_out = prefix_tokens<kPfx>(p, bb) + window_skip<kWin>(p, bb);
        return max(vseq_len<kPfx, kMulti, kWin>(p, bb), 0);
      };
      int win_pre, nxt_pre;
      int win_len = load_len(wb, win_pre);
      int nxt_len = load_len(wb + 32, nxt_pre);
      // a chunk: `cnt` pages pg0.. of sequence b (own length L), partial slot
      // `slot`, chunk flags, and the split_info value to write (-1: none)
      constexpr int kSegFirst = 1, kSegLast = 2;
      struct Chunk {
        int b, pg0, cnt, L, slot, flags, split;
      };
      // entries past the row (length inconsistent with bt_stride) count as bad pages
      auto load_pid = [&](const Chunk& c, int pre) {
        const int idx = pre / ps + c.pg0 + lane;  // prefix pages come first in the row
        if (lane < c.cnt && idx < p.bt_stride)
          return p.block_table[static_cast<int64_t>(real_seq<kMulti>(p, c.b)) * p.bt_stride + idx];
        return -1;
      };
      // fills c with the next chunk of the range (c.cnt == 0 at its end) and
      // returns this lane's block-table entry of it
      auto next_chunk = [&](Chunk& c) {
        c.cnt = 0;
        if (g >= end) return -1;
        if (seg_left == 0) {
          while (true) {
            if (b >= B) return -1;
            while (b >= wb + 32) {  // slide the lengths window
              win_len = nxt_len;
              win_pre = nxt_pre;
              wb += 32;
              nxt_len = load_len(wb + 32, nxt_pre);
            }
            const int L = __shfl_sync(0xffffffffu, win_len, b - wb);
            const int np = (L + ps - 1) / ps;
            if (np == 0 || pg >= np + A) {
              ++b;
              pg = 0;
              continue;
            }
            if (pg < A) {  // the sequence's overhead units: no page
              const int skip = static_cast<int>(min(static_cast<long long>(A - pg), end - g));
              g += skip;
              pg += skip;
              if (g >= end) return -1;
            }
            pg -= A;  // from here on: page index
            seg_L = L;
            seg_np = np;
            seg_pre = __shfl_sync(0xffffffffu, win_pre, b - wb);
            break;
          }
          const int n_here = static_cast<int>(min(static_cast<long long>(seg_np - pg), end - g));
          const bool complete = (pg == 0) && (n_here == seg_np);
          seg_slot = complete ? -1 : (first_seg ? 2 * k : 2 * k + 1);
          c.split = -1;
          if (pg == 0) {  // the sequence starts here: record how many CTAs hold its pages
            const long long last = g + seg_np - 1;  // global unit of its last page
            const long long big = r_pages * (q_pages + 1);
            const int k1 = static_cast<int>(last < big ? last / (q_pages + 1)
                                                       : r_pages + (last - big) / max(q_pages, 1ll));
            c.split = ((k1 - k + 1) << 1) | (first_seg ? 0 : 1);
          }
          first_seg = false;
          seg_left = n_here;
          c.flags = kSegFirst;
        } else {
          c.flags = 0;
          c.split = -1;
        }
        c.b = b;
        c.pg0 = pg;
        c.cnt = min(32, seg_left);
        c.L = seg_L;
        c.slot = seg_slot;
        seg_left -= c.cnt;
        if (seg_left == 0) c.flags |= kSegLast;
        pg += c.cnt;
        g += c.cnt;
        // inside a segment pg is a page index; a segment ends at the sequence's
        // end (next sequence, unit 0) or at the range's end (walk over)
        if (seg_left == 0 && pg >= seg_np) {
          ++b;
          pg = 0;
        }
        return load_pid(c, seg_pre);
      };
      Chunk cur, nxt;
      int pid = next_chunk(cur);
      pdl_wait_primary();  // the metadata of the first chunk is loaded; copies and writes follow
      // this CTA's split_seq entry: none, unless a cut sequence starts here
      if (lane == 0) p.split_seq[k] = make_int2(-1, 0);
      while (cur.cnt > 0 && !aborted) {
        const int pid_nxt = next_chunk(nxt);
        if (cur.split >= 0 && lane == 0) p.split_info[cur.b] = make_int2(k, cur.split);
        if (cur.split >= 0 && (cur.split >> 1) > 1 && lane == 0) p.split_seq[k] = make_int2(cur.b, cur.split);
        const int np_cur = (cur.L + ps - 1) / ps;
        for (int i = 0; i < cur.cnt; ++i) {
          const int page = __shfl_sync(0xffffffffu, pid, i);
          const int pidx = cur.pg0 + i;
          const bool ok = page >= 0 && page < p.num_pages;
          // rows [lo, rows_end) of the page: a sliding window's first page
          // starts at the window's first token
          const int lo = (kWin && pidx == 0) ? max(0, cur.L - p.window) : 0;
          const int rows_end = ok ? ((pidx == np_cur - 1) ? (cur.L - pidx * ps) : ps) : 0;
          const int rows = kWin ? max(0, rows_end - lo) : rows_end;
          const int nchunks = rows > 0 ? (rows + p.chunk_rows - 1) / p.chunk_rows : 1;
          for (int c = 0; c < nchunks; ++c) {
            if (lane == 0) {
              const int s = ps_stage;
              if (it >= S && !mbar_wait(smem_u32(&empty[s]), ps_phase ^ 1)) {
                set_device_error(p.err_word, TS_DEVERR_TIMEOUT);
                aborted = true;
              } else {
                const int r0 = lo + c * p.chunk_rows;
                const int valid = max(0, min(rows_end - r0, p.chunk_rows));
                uint32_t flags = ((cur.flags & kSegFirst) && i == 0 && c == 0 ? kFlagFirst : 0u) |
                                 ((cur.flags & kSegLast) && i == cur.cnt - 1 && c == nchunks - 1 ? kFlagLast : 0u);
                if (!ok) {
                  flags |= kFlagBadPage;
                  set_device_error(p.err_word, TS_DEVERR_PAGE_RANGE);
                }
                StageDesc d;
                d.b = cur.b;
                d.valid = valid;
                d.flags = flags;
                d.out_slot = cur.slot;
                d.rem = cur.L - (pidx * ps + r0);
                desc[s] = d;
                const uint32_t bytes = static_cast<uint32_t>(valid) * p.row_bytes;
                const uint32_t qb = (flags & kFlagFirst) ? p.q_bytes : 0u;
                // fp8: the scales of the stage's chunk_rows rows (whole, in bounds
                // of the page even past the valid rows)
                const uint32_t sb = (kFp8 && bytes) ? p.scale_area : 0u;
                const uint32_t full_bar = smem_u32(&full[s]);
                mbar_arrive_expect_tx(full_bar, 2 * bytes + 2 * sb + qb);
                const uint32_t st = smem_u32(stages + static_cast<size_t>(s) * p.stage_bytes);
                if (bytes) {
                  const size_t off = static_cast<size_t>(page) * p.page_bytes +
                                     static_cast<size_t>(r0) * p.row_bytes;
                  bulk_g2s_hint(st, static_cast<const char*>(p.k_pool) + off, bytes, full_bar, pol);
                  bulk_g2s_hint(st + p.kv_area, static_cast<const char*>(p.v_pool) + off, bytes,
                                full_bar, pol);
                  if (sb) {
                    const size_t so = (static_cast<size_t>(page) * ps + r0) * p.H_kv;
                    bulk_g2s_hint(st + 2 * p.kv_area, p.k_scale + so, sb, full_bar, pol);
                    bulk_g2s_hint(st + 2 * p.kv_area + sb, p.v_scale + so, sb, full_bar, pol);
                  }
                }
                if (qb)
                  bulk_g2s(st + 2 * (p.kv_area + (kFp8 ? p.scale_area : 0u)),
                           static_cast<const char*>(p.q) + static_cast<size_t>(cur.b) * p.q_bytes, qb,
                           full_bar);
              }
            }
            aborted = __shfl_sync(0xffffffffu, aborted, 0);
            if (aborted) break;
            ++it;
            if (++ps_stage == S) {
              ps_stage = 0;
              ps_phase ^= 1;
            }
          }
          if (aborted) break;
        }
        cur = nxt;
        pid = pid_nxt;
      }
    } else if (lane == 0) {
      pdl_wait_primary();  // before the write
      p.split_seq[k] = make_int2(-1, 0);  // an empty range holds no cut sequence
    }
    if (lane == 0) {
      if (!aborted) {
        const int s = it % S;
        if (it >= S && !mbar_wait(smem_u32(&empty[s]), ((it / S) & 1) ^ 1)) {
          set_device_error(p.err_word, TS_DEVERR_TIMEOUT);
          aborted = true;
        } else {
          desc[s].flags = kFlagEnd;
          mbar_arrive(smem_u32(&full[s]));
        }
      }
      if (aborted) {
        // Let any copy already issued land before the CTA's shared memory is released.
        for (int j = max(0, it - S); j < it; ++j)
          mbar_wait(smem_u32(&full[j % S]), (j / S) & 1);
      }
    }
    return;
  }
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(RegSplit<G>::kConsumer));
  if (warp - kFirstConsumerWarp >= n_consumer) return;
  pdl_wait_primary();  // before the consumers' global reads (prefix state) and writes

  // ========================= consumer warps ================================
  const int h = warp - kFirstConsumerWarp;  // kv head of this warp
  const int j = lane / C::kLPT;
  const int l = lane % C::kLPT;
  const int tokens_per_pass = C::kNG * C::kTPG;
  const int npass = (p.chunk_rows + tokens_per_pass - 1) / tokens_per_pass;

  int dim_off[C::kNV];
  uint32_t lane_off[C::kNV];  // byte offset of this lane's vectors within a token row
#pragma unroll
  for (int v = 0; v < C::kNV; ++v) {
    dim_off[v] = v * (D / C::kNV) + C::kVE * l;
    lane_off[v] = static_cast<uint32_t>((h * D + dim_off[v]) * C::kES);
  }
  const uint32_t zero_row = smem_u32(smem + kZeroRowOff);
  const uint32_t row_stride = p.row_bytes;
  // Query row (within its virtual sequence) of warp row hh: folded token
  // hh >> g_shift, head h * g + (hh & (g - 1)).
  const int gs = kMulti ? p.g_shift : 0;
  auto qrow = [&](int hh) {
    if constexpr (kMulti) return (hh >> gs) * p.H_q + (h << gs) + (hh & ((1 << gs) - 1));
    return h * G + hh;
  };

  float2 qv[G][C::kPairsPL];
  float2 acc[G][C::kPairsPL];
  float m[G], lsum[G];

  int it = 0, s = 0, phase = 0;  // s = it % S, phase = (it / S) & 1
  while (true) {
    if (!mbar_wait(smem_u32(&full[s]), phase)) {
      set_device_error(p.err_word, TS_DEVERR_TIMEOUT);
      break;
    }
    const StageDesc d = desc[s];
    if (d.flags & kFlagEnd) break;
    const uint32_t st = smem_u32(stages + static_cast<size_t>(s) * p.stage_bytes);
    const uint32_t kbase = st, vbase = st + p.kv_area;
    const uint32_t sarea = kFp8 ? p.scale_area : 0u;
    const uint32_t ksbase = st + 2 * p.kv_area, vsbase = ksbase + sarea;  // fp8 scales
    const uint32_t qbase = st + 2 * (p.kv_area + sarea);

    if (d.flags & kFlagFirst) {
      // the lane's query dims are those of its K/V vectors; a K/V vector of
      // fp8 codes spans two 16-byte vectors of bf16 queries
      constexpr int kQV = C::kVE / Elem<T>::kVE;
#pragma unroll
      for (int hh = 0; hh < G; ++hh) {
        m[hh] = -INFINITY;
        lsum[hh] = 0.f;
#pragma unroll
        for (int v = 0; v < C::kNV; ++v) {
#pragma unroll
          for (int u = 0; u < kQV; ++u) {
            const uint4 raw =
                lds128(qbase + (qrow(hh) * D + dim_off[v] + u * Elem<T>::kVE) * static_cast<int>(sizeof(T)));
#pragma unroll
            for (int w = 0; w < Elem<T>::kPairs; ++w) {
              const float2 f = Elem<T>::pair(raw, w);
              const int x = v * Elem<KV>::kPairs + u * Elem<T>::kPairs + w;
              qv[hh][x] = make_float2(f.x * p.scale_log2, f.y * p.scale_log2);
              acc[hh][x] = make_float2(0.f, 0.f);
            }
          }
        }
      }
    }

    const int valid = d.valid;
    // Folded query tokens: warp row hh attends the stage's rows before
    // lim(hh) = rem - (fold - 1) + (hh >> g_shift) (>= valid unless the stage
    // holds one of the virtual sequence's last fold - 1 tokens).
    const int lim0 = kMulti ? d.rem - p.fold + 1 : valid;
    // A full stage (every row valid, passes cover it exactly) needs no row
    // clamping and no score masking: the common case gets its own copy.
    auto run_passes = [&](auto full_tag) {
    constexpr bool kFull = decltype(full_tag)::value;
    for (int pass = 0; pass < npass; ++pass) {
      const int t0 = pass * tokens_per_pass + j * C::kTPG;
      // Rows past `valid` read the last valid row (their scores are masked and
      // their weights are 0); a unit with no valid row reads the zero row. So the
      // token loop has no branches and its dependency chains interleave freely.
      float sc[C::kTPG][G];
      // V rows are read together with the K rows, so their shared-memory
      // latency hides behind the scores and the softmax
      uint4 vv[C::kTPG][C::kNV];
      uint32_t row_off[C::kTPG];
#pragma unroll
      for (int i = 0; i < C::kTPG; ++i)
        row_off[i] = kFull ? (t0 + i) * row_stride
                           : (valid > 0 ? min(t0 + i, valid - 1) * row_stride : 0xffffffffu);
#pragma unroll
      for (int i = 0; i < C::kTPG; ++i) {
        const uint32_t ra = row_off[i] != 0xffffffffu ? vbase + row_off[i] : zero_row;
#pragma unroll
        for (int v = 0; v < C::kNV; ++v) vv[i][v] = lds128(ra + lane_off[v]);
      }
#pragma unroll
      for (int i = 0; i < C::kTPG; ++i) {
        const uint32_t ra = row_off[i] != 0xffffffffu ? kbase + row_off[i] : zero_row;
        uint4 kv[C::kNV];
#pragma unroll
        for (int v = 0; v < C::kNV; ++v) kv[v] = lds128(ra + lane_off[v]);
        float2 kf[C::kPairsPL];  // the row widened once, used by all G heads
#pragma unroll
        for (int v = 0; v < C::kNV; ++v)
#pragma unroll
          for (int w = 0; w < Elem<KV>::kPairs; ++w) kf[v * Elem<KV>::kPairs + w] = Elem<KV>::pair(kv[v], w);
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
          float2 a = make_float2(0.f, 0.f);
#pragma unroll
          for (int x = 0; x < C::kPairsPL; ++x) a = __ffma2_rn(qv[hh][x], kf[x], a);
          sc[i][hh] = a.x + a.y;
        }
      }
#pragma unroll
      for (int o = 1; o < C::kLPT; o <<= 1)
#pragma unroll
        for (int i = 0; i < C::kTPG; ++i)
#pragma unroll
          for (int hh = 0; hh < G; ++hh) sc[i][hh] += __shfl_xor_sync(0xffffffffu, sc[i][hh], o);
      // fp8 cache: token i's scores take its K row's group scale, and its
      // softmax weight its V row's (0 for rows past the valid ones, whose
      // scale slots may hold anything)
      float vsc[C::kTPG];
      if constexpr (kFp8) {
#pragma unroll
        for (int i = 0; i < C::kTPG; ++i) {
          const int rix = kFull ? t0 + i : min(t0 + i, max(valid - 1, 0));
          const uint32_t so = static_cast<uint32_t>((rix * p.H_kv + h) * 4);
          const float ks = lds_f32(ksbase + so);
          vsc[i] = (kFull || t0 + i < valid) ? lds_f32(vsbase + so) : 0.f;
#pragma unroll
          for (int hh = 0; hh < G; ++hh) sc[i][hh] *= ks;
        }
      }
#pragma unroll
      for (int i = 0; i < C::kTPG; ++i) {
        const bool in = kFull || t0 + i < valid;
#pragma unroll
        for (int hh = 0; hh < G; ++hh)
          sc[i][hh] = (in && (kFull || !kMulti || t0 + i < lim0 + (hh >> gs))) ? sc[i][hh] : -INFINITY;
      }

      // Online softmax with a lazily moved reference max: m[] only moves when a
      // score exceeds it by more than kRescaleSlack (log2 units), so p <= 2^slack
      // and the accumulators are rescaled only a few times per sequence. The
      // decision is made warp-uniform so the rescale branch never diverges.
      float mx[G];
      bool need = false;
#pragma unroll
      for (int hh = 0; hh < G; ++hh) {
        mx[hh] = sc[0][hh];
#pragma unroll
        for (int i = 1; i < C::kTPG; ++i) mx[hh] = fmaxf(mx[hh], sc[i][hh]);
        need |= mx[hh] > m[hh] + kRescaleSlack;
      }
      if (__any_sync(0xffffffffu, need)) {
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
          const float mnew = fmaxf(m[hh], mx[hh]);
          const float alpha = m[hh] == -INFINITY ? 0.f : fast_exp2(m[hh] - mnew);
          m[hh] = mnew;
          lsum[hh] *= alpha;
          const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
          for (int x = 0; x < C::kPairsPL; ++x) acc[hh][x] = __fmul2_rn(acc[hh][x], a2);
        }
      }
      float pr[C::kTPG][G];
#pragma unroll
      for (int hh = 0; hh < G; ++hh) {
        const float msafe = m[hh] == -INFINITY ? 0.f : m[hh];
        float ls = lsum[hh];
#pragma unroll
        for (int i = 0; i < C::kTPG; ++i) {
          pr[i][hh] = fast_exp2(sc[i][hh] - msafe);
          ls += pr[i][hh];
        }
        lsum[hh] = ls;
      }
#pragma unroll
      for (int i = 0; i < C::kTPG; ++i) {
        float2 vf[C::kPairsPL];
#pragma unroll
        for (int v = 0; v < C::kNV; ++v)
#pragma unroll
          for (int w = 0; w < Elem<KV>::kPairs; ++w) vf[v * Elem<KV>::kPairs + w] = Elem<KV>::pair(vv[i][v], w);
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
          const float pw = kFp8 ? pr[i][hh] * vsc[i] : pr[i][hh];
          const float2 p2 = make_float2(pw, pw);
#pragma unroll
          for (int x = 0; x < C::kPairsPL; ++x) acc[hh][x] = __ffma2_rn(p2, vf[x], acc[hh][x]);
        }
      }
    }
    };
    if (valid == p.chunk_rows && p.chunk_rows % tokens_per_pass == 0 && lim0 >= valid)
      run_passes(std::integral_constant<bool, true>());
    else
      run_passes(std::integral_constant<bool, false>());

    if (d.flags & kFlagLast) {
      // Merge the NG token groups of this warp (lanes with equal l hold the
      // same dims of different token groups) by LSE, as a reduce-scatter:
      // weights first (group max M, w_j = 2^(m_j - M), total l), then each
      // butterfly step hands half of the still-shared values to the partner,
      // so after log2(NG) steps every lane owns NT/NG finished values and
      // all 32 lanes write the output.
      constexpr int P = C::kPairsPL;     // float2 per lane per head
      constexpr int NT = G * P;          // float2 per lane
      constexpr int NF = NT / C::kNG;    // float2 each lane owns at the end
      static_assert(NT % C::kNG == 0 && NF >= 1, "reduce-scatter split");
      static_assert((G & (G - 1)) == 0, "heads per kv head: a power of two");
      float M[G], Lt[G];
      float2 r[NT];
#pragma unroll
      for (int hh = 0; hh < G; ++hh) {
        float mx = m[hh];
#pragma unroll
        for (int o = C::kLPT; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        const float ms = mx == -INFINITY ? 0.f : mx;
        const float w = fast_exp2(m[hh] - ms);  // 0 for a group that saw no token
        float lw = lsum[hh] * w;
#pragma unroll
        for (int o = C::kLPT; o < 32; o <<= 1) lw += __shfl_xor_sync(0xffffffffu, lw, o);
        M[hh] = mx;
        Lt[hh] = lw;
        const float2 w2 = make_float2(w, w);
#pragma unroll
        for (int x = 0; x < P; ++x) r[hh * P + x] = __fmul2_rn(acc[hh][x], w2);
      }
      int own = 0;  // flattened index (head * P + pair) of r[0] after the steps
#pragma unroll
      for (int st = 0; (C::kLPT << st) < 32; ++st) {
        const int o = C::kLPT << st;
        const int half = (NT >> st) / 2;
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
          const float2 send = up ? r[i] : r[i + half];
          const float2 keep = up ? r[i + half] : r[i];
          float2 recv;
          recv.x = __shfl_xor_sync(0xffffffffu, send.x, o);
          recv.y = __shfl_xor_sync(0xffffffffu, send.y, o);
          r[i] = make_float2(keep.x + recv.x, keep.y + recv.y);
        }
        own += up ? half : 0;
      }
      // r[i] now holds flattened value own + i: head (own + i) / P, pair
      // (own + i) % P of this lane's dims. Finish them per whole 16-byte
      // vector when the share allows it.
      constexpr int U = (NF % Elem<T>::kPairs == 0) ? Elem<T>::kPairs : 1;
      auto pick = [&](const float (&a)[G], int hh) {
        float v = a[0];
#pragma unroll
        for (int q = 1; q < G; ++q) v = hh == q ? a[q] : v;
        return v;
      };
      bool grouped = false;
      if constexpr (kPfx) grouped = p.group_of[d.b] >= 0;
      const int64_t row0 = static_cast<int64_t>(d.b) * p.rows;  // first query row of the virtual sequence
      // normaliser c_s of the own-token state and weight c_p of the prefix
      // state (0 outside prefix mode), and the row's final LSE (log2 units)
      auto finish = [&](int hh, float& cs, float& cp, float& lse2) {
        const float Mh = pick(M, hh), Lh = pick(Lt, hh);
        cs = Lh > 0.f ? __fdividef(1.0f, Lh) : 0.f;
        cp = 0.f;
        lse2 = Lh > 0.f ? Mh + __log2f(Lh) : -INFINITY;
        if (kPfx && grouped && d.out_slot < 0) {
          const float lp2 = p.prefix_lse[row0 + qrow(hh)] * kLog2e;
          const float Mx = fmaxf(lse2, lp2);
          const float ws = lse2 == -INFINITY ? 0.f : fast_exp2(lse2 - Mx);
          const float wp = lp2 == -INFINITY ? 0.f : fast_exp2(lp2 - Mx);
          const float den = ws + wp;
          const float iden = den > 0.f ? __fdividef(1.0f, den) : 0.f;
          cs *= ws * iden;
          cp = wp * iden;
          lse2 = den > 0.f ? Mx + __log2f(den) : -INFINITY;
        }
      };
#pragma unroll
      for (int c = 0; c < NF; c += U) {
        const int xf = own + c;
        const int hh = xf / P, x = xf % P;
        const int dim = (x / Elem<KV>::kPairs) * (D / C::kNV) + C::kVE * l + 2 * (x % Elem<KV>::kPairs);
        float cs, cp, lse2;
        finish(hh, cs, cp, lse2);
        float2 val[U];
#pragma unroll
        for (int u = 0; u < U; ++u) val[u] = make_float2(r[c + u].x * cs, r[c + u].y * cs);
        if (d.out_slot < 0) {
          if (cp != 0.f) {
            const float* po = p.prefix_o + (row0 + qrow(hh)) * D + dim;
#pragma unroll
            for (int u = 0; u < U; ++u) {
              const float2 pv = *reinterpret_cast<const float2*>(po + 2 * u);
              val[u] = make_float2(val[u].x + pv.x * cp, val[u].y + pv.y * cp);
            }
          }
          T* o = static_cast<T*>(p.out) + (row0 + qrow(hh)) * D + dim;
          if constexpr (sizeof(T) == 2) {
            if constexpr (U == 4) {
              *reinterpret_cast<uint4*>(o) =
                  make_uint4(float2_to_bf16x2(val[0].x, val[0].y), float2_to_bf16x2(val[1].x, val[1].y),
                             float2_to_bf16x2(val[2].x, val[2].y), float2_to_bf16x2(val[3].x, val[3].y));
            } else {
#pragma unroll
              for (int u = 0; u < U; ++u)
                *reinterpret_cast<uint32_t*>(o + 2 * u) = float2_to_bf16x2(val[u].x, val[u].y);
            }
          } else {
            if constexpr (U == 2) {
              *reinterpret_cast<float4*>(o) = make_float4(val[0].x, val[0].y, val[1].x, val[1].y);
            } else {
#pragma unroll
              for (int u = 0; u < U; ++u) *reinterpret_cast<float2*>(o + 2 * u) = val[u];
            }
          }
        } else {
          float* o = p.part_o + (static_cast<int64_t>(d.out_slot) * p.rows + qrow(hh)) * D + dim;
          if constexpr (U % 2 == 0) {
#pragma unroll
            for (int u = 0; u < U; u += 2)
              *reinterpret_cast<float4*>(o + 2 * u) = make_float4(val[u].x, val[u].y, val[u + 1].x, val[u + 1].y);
          } else {
#pragma unroll
            for (int u = 0; u < U; ++u) *reinterpret_cast<float2*>(o + 2 * u) = val[u];
          }
        }
      }
      {  // lane q < G writes head q's LSE (every lane computes one, no divergence)
        const int q = lane & (G - 1);
        float cs, cp, lse2;
        finish(q, cs, cp, lse2);
        if (lane < G) {
          if (d.out_slot < 0) {
            if (p.lse) p.lse[row0 + qrow(q)] = lse2 * kLn2;
          } else {
            p.part_lse[static_cast<int64_t>(d.out_slot) * p.rows + qrow(q)] = lse2 * kLn2;
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
    ++it;
    if (++s == S) {
      s = 0;
      phase ^= 1;
    }
  }
}

}  // namespace
}  // namespace ts
