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
//   * At the end of a sequence's segment the groups merge by LSE with shuffles
//     and lane group 0 writes either the final output (segment = whole
//     sequence) or an fp32 partial state into one of the CTA's two workspace
//     slots (first / last segment of its range). The merge kernel, launched
//     with programmatic dependent launch, reduces the split sequences.
#include <cmath>
#include <cstdlib>

#include "ts_common.cuh"

namespace ts {
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

struct StageDesc {
  int32_t b;         // sequence
  int32_t valid;     // tokens present in this page
  uint32_t flags;    // kFlag*
  int32_t out_slot;  // -1: write the final output; else partial slot index
};

struct PagedParams {
  const void* q;
  const void* k_pool;
  const void* v_pool;
  const int32_t* block_table;
  const int32_t* seq_lens;
  int32_t bt_stride, B, H_q, H_kv, page_size, num_pages;
  float scale_log2;  // scale * log2(e)
  void* out;
  float* lse;
  uint32_t* err_word;
  int2* split_info;  // per sequence: {first CTA, (parts << 1) | slot of first part}
  float* part_o;     // [2 * gridDim.x, H_q, D]
  float* part_lse;   // [2 * gridDim.x, H_q]
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
  uint32_t kv_area;      // chunk_rows * row_bytes: K (and V) area of a stage
  uint32_t row_bytes;    // bytes of one token row of K (or V), all kv heads
  uint32_t q_bytes;      // bytes of one sequence's query rows
};

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

// Writes the output of a sequence with no own tokens: O = 0, LSE = -inf, or
// the prefix state alone in prefix mode.
template <typename T, bool kPfx>
__device__ void write_empty_sequence(const PagedParams& p, int D, int b, int k) {
  const bool grouped = kPfx && p.group_of[b] >= 0;
  T* out = static_cast<T*>(p.out) + static_cast<int64_t>(b) * p.H_q * D;
  const float* po = grouped ? p.prefix_o + static_cast<int64_t>(b) * p.H_q * D : nullptr;
  for (int i = 0; i < p.H_q * D; ++i) out[i] = static_cast<T>(grouped ? po[i] : 0.0f);
  if (p.lse)
    for (int h = 0; h < p.H_q; ++h)
      p.lse[static_cast<int64_t>(b) * p.H_q + h] =
          grouped ? p.prefix_lse[static_cast<int64_t>(b) * p.H_q + h] : -INFINITY;
  p.split_info[b] = make_int2(k, 0);
}

template <typename T, int D, int G, bool kPfx>
__global__ void __launch_bounds__(kThreads, 1) paged_decode_kernel(const PagedParams p) {
  using C = Cfg<T, D, G>;
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
  unsigned char* stages = smem + p.stages_off;

  pdl_wait_primary();
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
  long long mine = 0;
  for (int b = lo; b < hi; ++b) {
    const int L = p.seq_lens[b] - prefix_tokens<kPfx>(p, b);
    if (L > 0)
      mine += (L + ps - 1) / ps;
    else if (b % G_ctas == k)
      write_empty_sequence<T, kPfx>(p, D, b, k);
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
    for (int b = lo; b < hi; ++b) {
      const int L = p.seq_lens[b] - prefix_tokens<kPfx>(p, b);
      const long long np = L > 0 ? (L + ps - 1) / ps : 0;
      if (start < off + np) {
        s_start[0] = b;
        s_start[1] = static_cast<int>(start - off);
        break;
      }
      off += np;
    }
  }
  __syncthreads();

  if (warp < kFirstConsumerWarp) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(RegSplit<G>::kProducer));
    if (warp != 0) return;
    // ======================= producer warp ================================
    int it = 0;
    bool aborted = false;
    if (start < end && s_start[0] >= 0) {
      const uint64_t pol = policy_evict_first();
      long long g = start;
      int b = s_start[0];
      int pg = s_start[1];
      bool first_seg = true;
      while (g < end && !aborted && b < B) {
        const int pre = prefix_tokens<kPfx>(p, b);
        const int L = max(p.seq_lens[b] - pre, 0);
        const int np = (L + ps - 1) / ps;
        if (np == 0 || pg >= np) {
          ++b;
          pg = 0;
          continue;
        }
        const int n_here = static_cast<int>(min(static_cast<long long>(np - pg), end - g));
        const bool complete = (pg == 0) && (n_here == np);
        const int out_slot = complete ? -1 : (first_seg ? 2 * k : 2 * k + 1);
        if (pg == 0 && lane == 0) {
          const long long last = g + np - 1;  // global index of the sequence's last page
          const long long big = r_pages * (q_pages + 1);
          const int k1 = static_cast<int>(last < big ? last / (q_pages + 1)
                                                     : r_pages + (last - big) / max(q_pages, 1ll));
          const int nparts = k1 - k + 1;
          p.split_info[b] = make_int2(k, (nparts << 1) | (first_seg ? 0 : 1));
        }
        const int pre_pages = pre / ps;  // prefix pages come first in the row
        const int32_t* bt_row = p.block_table + static_cast<int64_t>(b) * p.bt_stride + pre_pages + pg;
        for (int base = 0; base < n_here && !aborted; base += 32) {
          const int cnt = min(32, n_here - base);
          // entries past the row (length inconsistent with bt_stride) count as bad pages
          int pid = -1;
          if (lane < cnt && pre_pages + pg + base + lane < p.bt_stride) pid = bt_row[base + lane];
          for (int i = 0; i < cnt; ++i) {
            const int page = __shfl_sync(0xffffffffu, pid, i);
            const int pidx = pg + base + i;
            const bool ok = page >= 0 && page < p.num_pages;
            const int rows = ok ? ((pidx == np - 1) ? (L - pidx * ps) : ps) : 0;
            const int nchunks = rows > 0 ? (rows + p.chunk_rows - 1) / p.chunk_rows : 1;
            for (int c = 0; c < nchunks; ++c) {
              if (lane == 0) {
                const int s = it % S;
                if (it >= S && !mbar_wait(smem_u32(&empty[s]), ((it / S) & 1) ^ 1)) {
                  set_device_error(p.err_word, TS_DEVERR_TIMEOUT);
                  aborted = true;
                } else {
                  const int r0 = c * p.chunk_rows;
                  const int valid = max(0, min(rows - r0, p.chunk_rows));
                  uint32_t flags = (base + i == 0 && c == 0 ? kFlagFirst : 0u) |
                                   (base + i == n_here - 1 && c == nchunks - 1 ? kFlagLast : 0u);
                  if (!ok) {
                    flags |= kFlagBadPage;
                    set_device_error(p.err_word, TS_DEVERR_PAGE_RANGE);
                  }
                  StageDesc d;
                  d.b = b;
                  d.valid = valid;
                  d.flags = flags;
                  d.out_slot = out_slot;
                  desc[s] = d;
                  const uint32_t bytes = static_cast<uint32_t>(valid) * p.row_bytes;
                  const uint32_t qb = (flags & kFlagFirst) ? p.q_bytes : 0u;
                  const uint32_t full_bar = smem_u32(&full[s]);
                  mbar_arrive_expect_tx(full_bar, 2 * bytes + qb);
                  const uint32_t st = smem_u32(stages + static_cast<size_t>(s) * p.stage_bytes);
                  if (bytes) {
                    const size_t off = static_cast<size_t>(page) * p.page_bytes +
                                       static_cast<size_t>(r0) * p.row_bytes;
                    bulk_g2s_hint(st, static_cast<const char*>(p.k_pool) + off, bytes, full_bar, pol);
                    bulk_g2s_hint(st + p.kv_area, static_cast<const char*>(p.v_pool) + off, bytes,
                                  full_bar, pol);
                  }
                  if (qb)
                    bulk_g2s(st + 2 * p.kv_area,
                             static_cast<const char*>(p.q) + static_cast<size_t>(b) * p.q_bytes, qb,
                             full_bar);
                }
              }
              aborted = __shfl_sync(0xffffffffu, aborted, 0);
              if (aborted) break;
              ++it;
            }
            if (aborted) break;
          }
        }
        g += n_here;
        pg += n_here;
        if (pg >= np) {
          ++b;
          pg = 0;
        }
        first_seg = false;
      }
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

  // ========================= consumer warps ================================
  const int h = warp - kFirstConsumerWarp;  // kv head of this warp
  const int j = lane / C::kLPT;
  const int l = lane % C::kLPT;
  const int tokens_per_pass = C::kNG * C::kTPG;
  const int npass = (p.chunk_rows + tokens_per_pass - 1) / tokens_per_pass;
  const int H_kv = p.H_kv;

  int dim_off[C::kNV];
  uint32_t lane_off[C::kNV];  // byte offset of this lane's vectors within a token row
#pragma unroll
  for (int v = 0; v < C::kNV; ++v) {
    dim_off[v] = v * (D / C::kNV) + C::kVE * l;
    lane_off[v] = static_cast<uint32_t>((h * D + dim_off[v]) * C::kES);
  }
  const uint32_t zero_row = smem_u32(smem + kZeroRowOff);
  const uint32_t row_stride = p.row_bytes;

  float2 qv[G][C::kPairsPL];
  float2 acc[G][C::kPairsPL];
  float m[G], lsum[G];

  int it = 0;
  while (true) {
    const int s = it % S;
    if (!mbar_wait(smem_u32(&full[s]), (it / S) & 1)) {
      set_device_error(p.err_word, TS_DEVERR_TIMEOUT);
      break;
    }
    const StageDesc d = desc[s];
    if (d.flags & kFlagEnd) break;
    const uint32_t st = smem_u32(stages + static_cast<size_t>(s) * p.stage_bytes);
    const uint32_t kbase = st, vbase = st + p.kv_area, qbase = st + 2 * p.kv_area;

    if (d.flags & kFlagFirst) {
#pragma unroll
      for (int hh = 0; hh < G; ++hh) {
        m[hh] = -INFINITY;
        lsum[hh] = 0.f;
#pragma unroll
        for (int v = 0; v < C::kNV; ++v) {
          const uint4 raw =
              lds128(qbase + ((h * G + hh) * D + dim_off[v]) * C::kES);
#pragma unroll
          for (int w = 0; w < Elem<T>::kPairs; ++w) {
            const float2 f = Elem<T>::pair(raw, w);
            qv[hh][v * Elem<T>::kPairs + w] = make_float2(f.x * p.scale_log2, f.y * p.scale_log2);
            acc[hh][v * Elem<T>::kPairs + w] = make_float2(0.f, 0.f);
          }
        }
      }
    }

    const int valid = d.valid;
    for (int pass = 0; pass < npass; ++pass) {
      const int t0 = pass * tokens_per_pass + j * C::kTPG;
      // Rows past `valid` read the last valid row (their scores are masked and
      // their weights are 0); a unit with no valid row reads the zero row. So the
      // token loop has no branches and its dependency chains interleave freely.
      float sc[C::kTPG][G];
#pragma unroll
      for (int i = 0; i < C::kTPG; ++i) {
        const int t = t0 + i;
        const uint32_t ra = valid > 0 ? kbase + min(t, valid - 1) * row_stride : zero_row;
        uint4 kv[C::kNV];
#pragma unroll
        for (int v = 0; v < C::kNV; ++v) kv[v] = lds128(ra + lane_off[v]);
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
          float2 a = make_float2(0.f, 0.f);
#pragma unroll
          for (int v = 0; v < C::kNV; ++v)
#pragma unroll
            for (int w = 0; w < Elem<T>::kPairs; ++w)
              a = __ffma2_rn(qv[hh][v * Elem<T>::kPairs + w], Elem<T>::pair(kv[v], w), a);
          sc[i][hh] = a.x + a.y;
        }
      }
#pragma unroll
      for (int o = 1; o < C::kLPT; o <<= 1)
#pragma unroll
        for (int i = 0; i < C::kTPG; ++i)
#pragma unroll
          for (int hh = 0; hh < G; ++hh) sc[i][hh] += __shfl_xor_sync(0xffffffffu, sc[i][hh], o);
#pragma unroll
      for (int i = 0; i < C::kTPG; ++i) {
        const bool in = t0 + i < valid;
#pragma unroll
        for (int hh = 0; hh < G; ++hh) sc[i][hh] = in ? sc[i][hh] : -INFINITY;
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
        const int t = t0 + i;
        const uint32_t ra = valid > 0 ? vbase + min(t, valid - 1) * row_stride : zero_row;
        uint4 vv[C::kNV];
#pragma unroll
        for (int v = 0; v < C::kNV; ++v) vv[v] = lds128(ra + lane_off[v]);
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
          const float2 p2 = make_float2(pr[i][hh], pr[i][hh]);
#pragma unroll
          for (int v = 0; v < C::kNV; ++v)
#pragma unroll
            for (int w = 0; w < Elem<T>::kPairs; ++w)
              acc[hh][v * Elem<T>::kPairs + w] =
                  __ffma2_rn(p2, Elem<T>::pair(vv[v], w), acc[hh][v * Elem<T>::kPairs + w]);
        }
      }
    }

    if (d.flags & kFlagLast) {
      // Merge the NG token groups of this warp by LSE (lanes with equal l).
#pragma unroll
      for (int o = C::kLPT; o < 32; o <<= 1) {
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
          const float mo = __shfl_xor_sync(0xffffffffu, m[hh], o);
          const float lo_ = __shfl_xor_sync(0xffffffffu, lsum[hh], o);
          const float mn = fmaxf(m[hh], mo);
          const float ms = mn == -INFINITY ? 0.f : mn;
          const float wa = fast_exp2(m[hh] - ms), wb = fast_exp2(mo - ms);
          lsum[hh] = lsum[hh] * wa + lo_ * wb;
          m[hh] = mn;
          const float2 wa2 = make_float2(wa, wa), wb2 = make_float2(wb, wb);
#pragma unroll
          for (int x = 0; x < C::kPairsPL; ++x) {
            float2 other;
            other.x = __shfl_xor_sync(0xffffffffu, acc[hh][x].x, o);
            other.y = __shfl_xor_sync(0xffffffffu, acc[hh][x].y, o);
            acc[hh][x] = __ffma2_rn(acc[hh][x], wa2, __fmul2_rn(other, wb2));
          }
        }
      }
      if (j == 0) {
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
          const int hq = h * G + hh;
          const float ls = lsum[hh];
          float inv = ls > 0.f ? 1.0f / ls : 0.f;
          float lse2 = ls > 0.f ? m[hh] + log2f(ls) : -INFINITY;
          if (d.out_slot < 0) {
            T* o = static_cast<T*>(p.out) + (static_cast<int64_t>(d.b) * p.H_q + hq) * D;
            if constexpr (kPfx) {
              if (p.group_of[d.b] >= 0) {
                // merge the shared-prefix state: weights by LSE (log2 domain)
                const int64_t row = static_cast<int64_t>(d.b) * p.H_q + hq;
                const float lp2 = p.prefix_lse[row] * kLog2e;
                const float M = fmaxf(lse2, lp2);
                const float ws = lse2 == -INFINITY ? 0.f : fast_exp2(lse2 - M);
                const float wp = lp2 == -INFINITY ? 0.f : fast_exp2(lp2 - M);
                const float den = ws + wp;
                const float cs = den > 0.f ? inv * ws / den : 0.f;
                const float cp = den > 0.f ? wp / den : 0.f;
                const float* po = p.prefix_o + row * D;
#pragma unroll
                for (int v = 0; v < C::kNV; ++v)
#pragma unroll
                  for (int w = 0; w < Elem<T>::kPairs; ++w) {
                    const float2 pv2 = *reinterpret_cast<const float2*>(po + dim_off[v] + 2 * w);
                    float2& a = acc[hh][v * Elem<T>::kPairs + w];
                    a = make_float2(a.x * cs + pv2.x * cp, a.y * cs + pv2.y * cp);
                  }
                inv = 1.0f;  // the merged rows are already normalised
                lse2 = den > 0.f ? M + log2f(den) : -INFINITY;
              }
            }
#pragma unroll
            for (int v = 0; v < C::kNV; ++v) {
              if constexpr (sizeof(T) == 2) {
                uint4 pk;
                const float2* a = &acc[hh][v * 4];
                pk.x = float2_to_bf16x2(a[0].x * inv, a[0].y * inv);
                pk.y = float2_to_bf16x2(a[1].x * inv, a[1].y * inv);
                pk.z = float2_to_bf16x2(a[2].x * inv, a[2].y * inv);
                pk.w = float2_to_bf16x2(a[3].x * inv, a[3].y * inv);
                *reinterpret_cast<uint4*>(o + dim_off[v]) = pk;
              } else {
                const float2* a = &acc[hh][v * 2];
                *reinterpret_cast<float4*>(o + dim_off[v]) =
                    make_float4(a[0].x * inv, a[0].y * inv, a[1].x * inv, a[1].y * inv);
              }
            }
            if (l == 0 && p.lse) p.lse[static_cast<int64_t>(d.b) * p.H_q + hq] = lse2 * kLn2;
          } else {
            float* o = p.part_o + (static_cast<int64_t>(d.out_slot) * p.H_q + hq) * D;
#pragma unroll
            for (int v = 0; v < C::kNV; ++v) {
#pragma unroll
              for (int w = 0; w < Elem<T>::kPairs; w += 2) {
                const float2 a0 = acc[hh][v * Elem<T>::kPairs + w];
                const float2 a1 = acc[hh][v * Elem<T>::kPairs + w + 1];
                *reinterpret_cast<float4*>(o + dim_off[v] + 2 * w) =
                    make_float4(a0.x * inv, a0.y * inv, a1.x * inv, a1.y * inv);
              }
            }
            if (l == 0) p.part_lse[static_cast<int64_t>(d.out_slot) * p.H_q + hq] = lse2 * kLn2;
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
    ++it;
  }
}

// Reduces the partial states of sequences cut across CTAs (one warp per
// (sequence, query head)); sequences written whole by the main kernel are
// skipped.
// In prefix mode a grouped sequence's shared-prefix state is one more part.
template <typename T, bool kPfx>
__global__ void __launch_bounds__(256) split_merge_kernel(const PagedParams p, int D) {
  pdl_wait_primary();
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int b = warp / p.H_q, hq = warp % p.H_q;
  if (b >= p.B) return;
  const int2 info = p.split_info[b];
  const int nparts = info.y >> 1;
  if (nparts <= 1) return;
  const int k0 = info.x, slot0 = info.y & 1;
  const int64_t row = static_cast<int64_t>(b) * p.H_q + hq;
  const bool grouped = kPfx && p.group_of[b] >= 0;
  const float lse_pre = grouped ? p.prefix_lse[row] : -INFINITY;
  float mx = lse_pre;
  for (int i = 0; i < nparts; ++i) {
    const int slot = i == 0 ? 2 * k0 + slot0 : 2 * (k0 + i);
    mx = fmaxf(mx, p.part_lse[static_cast<int64_t>(slot) * p.H_q + hq]);
  }
  const float ms = mx == -INFINITY ? 0.f : mx;
  float wsum = 0.f;
  for (int d0 = lane * 4; d0 < D; d0 += 128) {
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    wsum = 0.f;
    for (int i = 0; i < nparts; ++i) {
      const int slot = i == 0 ? 2 * k0 + slot0 : 2 * (k0 + i);
      const float w = __expf(p.part_lse[static_cast<int64_t>(slot) * p.H_q + hq] - ms);
      const float4 o =
          *reinterpret_cast<const float4*>(p.part_o + (static_cast<int64_t>(slot) * p.H_q + hq) * D + d0);
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
    T* out = static_cast<T*>(p.out) + (static_cast<int64_t>(b) * p.H_q + hq) * D + d0;
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
    case 1: return paged_decode_kernel<T, D, 1, kPfx>;
    case 2: return paged_decode_kernel<T, D, 2, kPfx>;
    case 4: return paged_decode_kernel<T, D, 4, kPfx>;
    case 8: return paged_decode_kernel<T, D, 8, kPfx>;
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

// CTAs of the persistent grid: one per SM. TS_PAGED_DECODE_CTAS overrides it
// (tests use it to sweep how sequences are cut across CTAs).
int paged_decode_ctas() {
  if (const char* env = getenv("TS_PAGED_DECODE_CTAS")) {
    const int n = atoi(env);
    if (n > 0 && n <= 65535) return n;
  }
  return device_sm_count();
}

struct WsLayout {
  size_t split_info, part_o, part_lse, total;
};

WsLayout workspace_layout(int B, int H_q, int D, int n_ctas) {
  WsLayout w;
  size_t off = kWorkspaceAlign;  // error word + pad
  w.split_info = off;
  off = align_up(off + static_cast<size_t>(B) * sizeof(int2), kWorkspaceAlign);
  w.part_o = off;
  off = align_up(off + static_cast<size_t>(2) * n_ctas * H_q * D * sizeof(float), kWorkspaceAlign);
  w.part_lse = off;
  off = align_up(off + static_cast<size_t>(2) * n_ctas * H_q * sizeof(float), kWorkspaceAlign);
  w.total = off;
  return w;
}

}  // namespace

// Launches the paged split-KV kernel pair; `pre` non-null selects prefix
// (cascade) mode.
ts_status launch_paged_decode_impl(const void* q, const void* k_pool, const void* v_pool,
                                   const int32_t* block_table, int32_t bt_stride,
                                   const int32_t* seq_lens, int32_t B, int32_t H_q, int32_t H_kv,
                                   int32_t D, int32_t page_size, int32_t num_pages, float scale,
                                   ts_dtype dtype, void* out, float* lse, void* workspace,
                                   size_t workspace_bytes, cudaStream_t stream, const char* who,
                                   const PrefixInputs* pre) {
  if (B < 0 || H_q <= 0 || H_kv <= 0 || D <= 0 || page_size <= 0 || num_pages <= 0 ||
      bt_stride <= 0)
    return fail(TS_ERR_INVALID_ARG, "%s: bad sizes (B=%d H_q=%d H_kv=%d D=%d ps=%d P=%d bt=%d)",
                who, B, H_q, H_kv, D, page_size, num_pages, bt_stride);
  if (H_q % H_kv != 0)
    return fail(TS_ERR_INVALID_ARG, "%s: H_q=%d not a multiple of H_kv=%d", who, H_q, H_kv);
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
  KernelFn fn = pick_kernel(dtype, D, g, pre != nullptr);
  if (!fn)
    return fail(TS_ERR_UNSUPPORTED, "%s: D=%d, group size %d (supported D 64/128, g 1/2/4/8)", who,
                D, g);
  const size_t es = dtype == TS_F32 ? 4 : 2;
  for (const void* ptr : {q, k_pool, v_pool, static_cast<const void*>(out)})
    if (reinterpret_cast<uintptr_t>(ptr) % 16 != 0)
      return fail(TS_ERR_INVALID_ARG, "%s: q, pools and out must be 16-byte aligned", who);
  const int n_ctas = paged_decode_ctas();
  if (n_ctas <= 0) return fail(TS_ERR_CUDA, "%s: cannot query the SM count", who);
  const WsLayout ws = workspace_layout(B, H_q, D, n_ctas);
  if (!workspace || workspace_bytes < ws.total)
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
  prm.B = B;
  prm.H_q = H_q;
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
  unsigned char* wsb = static_cast<unsigned char*>(workspace);
  prm.err_word = reinterpret_cast<uint32_t*>(wsb);
  prm.split_info = reinterpret_cast<int2*>(wsb + ws.split_info);
  prm.part_o = reinterpret_cast<float*>(wsb + ws.part_o);
  prm.part_lse = reinterpret_cast<float*>(wsb + ws.part_lse);
  prm.row_bytes = static_cast<uint32_t>(H_kv * D * es);
  prm.page_bytes = static_cast<uint32_t>(page_size) * prm.row_bytes;
  prm.q_bytes = static_cast<uint32_t>(H_q * D * es);
  // A stage holds chunk_rows token rows of one page (all kv heads, K and V)
  // plus room for one sequence's query rows. Whole pages when two stages fit,
  // else halves, quarters... TS_PAGED_DECODE_CHUNK_ROWS overrides (tuning).
  int chunk_rows = page_size;
  if (const char* env = getenv("TS_PAGED_DECODE_CHUNK_ROWS")) {
    const int v = atoi(env);
    if (v > 0 && v <= page_size) chunk_rows = v;
  }
  auto stage_of = [&](int rows) {
    return static_cast<uint32_t>(align_up(2ull * rows * prm.row_bytes + prm.q_bytes, 128));
  };
  while (chunk_rows > 1 &&
         (kSmemBudget - kHeaderBytes - align_up(prm.row_bytes, 128)) / stage_of(chunk_rows) < 2)
    chunk_rows = (chunk_rows + 1) / 2;
  prm.chunk_rows = chunk_rows;
  prm.kv_area = static_cast<uint32_t>(chunk_rows) * prm.row_bytes;
  prm.stage_bytes = stage_of(chunk_rows);
  prm.stages_off = static_cast<uint32_t>(kHeaderBytes + align_up(prm.row_bytes, 128));
  const int stages = std::min<int>(kMaxStages, (kSmemBudget - prm.stages_off) / prm.stage_bytes);
  if (stages < 2 || prm.row_bytes > 4096)
    return fail(TS_ERR_UNSUPPORTED, "%s: one token row of K+V plus the query rows (%u B) exceeds the stage budget",
                who, prm.stage_bytes);
  prm.num_stages = stages;
  const size_t smem = prm.stages_off + static_cast<size_t>(stages) * prm.stage_bytes;

  ts_status st = cuda_check(
      cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)),
      "set smem attribute");
  if (st != TS_OK) return st;
  // The producer/consumer register split assumes the kernel was compiled to
  // launch with kLaunchRegs registers per thread; with fewer, the consumers'
  // setmaxnreg.inc could never be satisfied. Refuse to launch in that case.
  cudaFuncAttributes fa;
  st = cuda_check(cudaFuncGetAttributes(&fa, fn), "query kernel attributes");
  if (st != TS_OK) return st;
  if (fa.numRegs < kLaunchRegs)
    return fail(TS_ERR_UNSUPPORTED, "%s: kernel compiled with %d registers/thread, the register split needs %d",
                who, fa.numRegs, kLaunchRegs);

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

  const long long warps = static_cast<long long>(B) * H_q;
  cudaLaunchConfig_t mcfg = {};
  mcfg.gridDim = dim3(static_cast<unsigned>((warps + 7) / 8));
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
                                       prm, D),
                    "split merge launch");
  else
    st = cuda_check(cudaLaunchKernelEx(&mcfg, split_merge_kernel<float, false>, prm, D),
                    "split merge launch");
  return st;
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

size_t paged_decode_workspace_bytes(int B, int H_q, int D) {
  const int n = paged_decode_ctas();
  if (n <= 0 || B < 0 || H_q <= 0 || D <= 0) return 0;
  return workspace_layout(B, H_q, D, n).total;
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
