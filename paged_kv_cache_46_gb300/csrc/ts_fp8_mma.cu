// Tensor-core decode over an fp8 (e4m3fn) KV cache that multiplies the cached
// codes as they are, for the Llama-3-8B layer shape (32 query heads over 8 kv
// heads, head dim 128, 16-token pages); ts_paged_decode_fp8_attn runs it when
// TS_FP8_DECODE_PATH=mma asks for it.
//
// tokenspeed 딥다이브 (fiv.co.kr), section 6-4: a cached row is its e4m3 codes
// times its token group's float32 scale. The products are tcgen05
// kind::f8f6f4 with K = 32, reading the codes where the TMA lands them:
//
// - A tile is one page of every kv head: 8 heads x 16 tokens = 128 keys
//   (N = 128), landing head by head as 128-byte rows (128-byte swizzle).
// - The 128 rows (TMEM lanes) are the 32 query heads, four lanes each: the
//   head's query split into three e4m3 terms (hi, then the rounding of what
//   hi leaves, then of what both leave: within max(2^-12 |x|, 2^-10) of the
//   scaled value, below bf16's own rounding for the elements that carry the
//   score) and a zero lane. The query is first scaled by a
//   power of two that brings its largest element to [2^7, 2^8).
//   S = Q K^T takes the terms from TMEM and the key codes from shared
//   memory. The head's four lanes split the tile's 16 keys of its kv head:
//   a reduce-scatter sums the three partial scores, four keys per lane.
// - Scores take the key row's scale. P follows the same three-term split,
//   of p x the value row's scale x a power-of-two gain that brings the
//   tile's largest value scale to [2^7, 2^8); with the running maximum
//   allowed to lag by at most 0.5 (log2 units), the terms stay below 448.
//   O += P V reads the value codes from shared memory (MN-major). P is zero
//   outside a head's own kv head (block-diagonal), so the heads sharing a
//   page do not mix. O is rescaled when the maximum or the gain moves.
// - Per page: 4 score and 4 value products against 32 KB of codes. S and P
//   are double-buffered in TMEM, so S(j + 1) runs while the softmax works on
//   tile j.
//
// Work split: the batch's pages are cut into equal contiguous ranges, one
// per CTA (persistent, one CTA per SM). A sequence cut across CTAs leaves
// float32 partial states (O / l and the LSE, one slot per CTA and end of its
// range); the CTA that arrives last on the sequence's counter merges them by
// LSE in slot order, so the result does not depend on which CTA finishes
// last. Counters carry the launch's epoch and the merging CTA clears them.
//
// Roles (320 threads): warps 0-3 softmax (thread = TMEM lane = query head
// tid / 4, term tid % 4; the head's four lanes split each tile's 16 keys),
// warp 4 TMA producer, warp 5 TMEM allocator and (lane 0) MMA issuer, warps
// 6-9 segment epilogues (O read out, outputs or partial states and the
// merge) and the query terms, which they prepare a segment ahead (two Q
// buffers in TMEM).
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <atomic>
#include <cmath>
#include <cstdlib>
#include <cstring>

#include "ts_tcgen05.cuh"

namespace ts {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

namespace {

constexpr int kPS = 16;                   // tokens per page
constexpr int kD = 128;                   // head dim (codes per row)
constexpr int kHkv = 8;
constexpr int kG = 4;                     // query heads per kv head
constexpr int kHq = kHkv * kG;            // 32
constexpr int kKeys = kHkv * kPS;         // keys per tile (one page of every kv head)
constexpr int kThreads = 320;
constexpr int kStages = 6;
constexpr int kTile = kKeys * kD;         // 16 KB of K (or V) codes
constexpr int kScaleBytes = kPS * kHkv * 4;   // a page's K (or V) scale rows
constexpr int kStage = 2 * kTile + 2 * kScaleBytes;  // codes K, V; scales K, V (1024-aligned)
constexpr int kMaxB = 4096;
constexpr int kOffPre = kStages * kStage;                 // [B + 1] page prefix sums
constexpr int kOffBar = kOffPre + (kMaxB + 4) * 4;
constexpr int kOffMisc = kOffBar + 256;                   // TMEM base, arrival, scan totals
constexpr int kOffQs = kOffMisc + 64;                     // [2][32] score factors
constexpr int kOffStats = kOffQs + 2 * kHq * 4;           // [2][32][3] segment statistics
constexpr int kSmem = kOffStats + 2 * kHq * 3 * 4;
// TMEM columns: Q terms [0, 64) (two segments), P [64, 128) (two tiles),
// S [128, 384) (two tiles), O [384, 512)
constexpr uint32_t kTQ = 0, kTP = 64, kTS = 128, kTO = 384, kTCols = 512;
constexpr float kSlack = 0.5f;            // lag of the running maximum (log2 units)
constexpr float kLog2eC = 1.4426950408889634f;
constexpr float kLn2C = 0.6931471805599453f;
constexpr int kCasLimit = 1 << 20;
static_assert(kStage % 1024 == 0 && kTile % 1024 == 0, "swizzled tiles 1024-byte aligned");
static_assert(kOffBar % 8 == 0, "mbarriers 8-byte aligned");
static_assert(kSmem <= 227 * 1024, "shared memory budget");

struct MmaParams {
  const __nv_bfloat16* q;        // [B, 32, 128]
  __nv_bfloat16* out;            // [B, 32, 128]
  float* lse;                    // [B, 32] or nullptr
  const int32_t* block_table;    // [B, bt_stride]
  const int32_t* seq_lens;       // [B]
  const float* k_scale;          // [num_pages, 16, 8]
  const float* v_scale;
  int32_t B, bt_stride, num_pages;
  float scale_log2;
  uint32_t* err_word;
  unsigned long long* counters;  // [B]: epoch << 32 | parts arrived
  float* part_o;                 // [2 * gridDim.x][32][128]: O / l of a cut sequence's part
  float* part_lse;               // [2 * gridDim.x][32]: its LSE (log2 units)
  uint32_t epoch;
};

// 2^e as a float, for e in [-126, 127].
__device__ __forceinline__ float pow2i(int e) { return __uint_as_float(static_cast<uint32_t>(127 + e) << 23); }

// floor(log2 x) of a positive normal float.
__device__ __forceinline__ int ilog2f(float x) { return static_cast<int>((__float_as_uint(x) >> 23) & 0xffu) - 127; }

// Two floats -> two e4m3 codes (round to nearest even, saturating), low byte first.
__device__ __forceinline__ uint32_t to_e4m3x2(float a, float b) {
  return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3));
}

// Two e4m3 codes (low byte first) -> their exact values.
__device__ __forceinline__ float2 from_e4m3x2(uint32_t c) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(c & 0xffffu), __NV_E4M3);
  return __half22float2(__half2(h));
}

// The three-term e4m3 split of (a, b): hi = e4m3(x), mid = e4m3(x - hi),
// lo = e4m3(x - hi - mid); the differences are exact in float32. Two codes
// per term, low byte first.
__device__ __forceinline__ void e4m3_terms(float a, float b, uint32_t& hi, uint32_t& mid, uint32_t& lo) {
  hi = to_e4m3x2(a, b);
  const float2 h = from_e4m3x2(hi);
  const float ra = a - h.x, rb = b - h.y;
  mid = to_e4m3x2(ra, rb);
  const float2 md = from_e4m3x2(mid);
  lo = to_e4m3x2(ra - md.x, rb - md.y);
}

// t[i] for a run-time i in 0 .. 3, by selects (indexing a register array at
// run time would move it to local memory).
__device__ __forceinline__ uint32_t pick4(const uint32_t (&t)[4], int i) {
  return i == 0 ? t[0] : (i == 1 ? t[1] : (i == 2 ? t[2] : t[3]));
}

// Counts this CTA's arrival on a counter tagged with the launch's epoch (a
// count left by another launch reads as none) and returns the count with it;
// 0 if the compare-and-swap kept failing.
__device__ __forceinline__ int arrive_count(unsigned long long* cnt, uint32_t epoch) {
  unsigned long long old = *reinterpret_cast<volatile unsigned long long*>(cnt);
  for (int i = 0; i < kCasLimit; ++i) {
    const unsigned long long nw = static_cast<uint32_t>(old >> 32) == epoch
                                      ? old + 1ull
                                      : ((static_cast<unsigned long long>(epoch) << 32) | 1ull);
    const unsigned long long prev = atomicCAS(cnt, old, nw);
    if (prev == old) return static_cast<int>(nw & 0xffffffffull);
    old = prev;
  }
  return 0;
}

__global__ void __launch_bounds__(kThreads, 1) fp8_mma_kernel(const MmaParams p, const __grid_constant__ CUtensorMap kmap,
                                                               const __grid_constant__ CUtensorMap vmap) {
  extern __shared__ __align__(1024) unsigned char smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  pdl_launch_dependents();
  if ((smem_u32(smem) & 1023u) != 0) {
    if (tid == 0) set_device_error(p.err_word, TS_DEVERR_SMEM_ALIGN);
    return;
  }
  int* pre = reinterpret_cast<int*>(smem + kOffPre);
  const uint32_t bars = smem_u32(smem + kOffBar);
  auto b_full = [&](int s) { return bars + 8u * s; };                       // stage landed
  auto b_empty = [&](int s) { return bars + 8u * (kStages + s); };          // stage consumed
  auto b_sfull = [&](int u) { return bars + 8u * (2 * kStages + u); };     // S buffer u written
  auto b_sfree = [&](int u) { return bars + 8u * (2 * kStages + 2 + u); }; // S buffer u read
  auto b_pfull = [&](int u) { return bars + 8u * (2 * kStages + 4 + u); };  // P buffer u written
  auto b_pvdone = [&](int u) { return bars + 8u * (2 * kStages + 6 + u); }; // P V of P buffer u done
  auto b_qready = [&](int u) { return bars + 8u * (2 * kStages + 8 + u); }; // Q buffer u holds its segment
  const uint32_t b_ofull = bars + 8u * (2 * kStages + 10);                  // O final for a segment
  const uint32_t b_ofree = bars + 8u * (2 * kStages + 11);                  // O read out
  auto b_segdone = [&](int u) { return bars + 8u * (2 * kStages + 12 + u); };  // segment statistics written
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  int* arrived = reinterpret_cast<int*>(smem + kOffMisc + 4);
  int* wsum = reinterpret_cast<int*>(smem + kOffMisc + 16);
  float* qscale = reinterpret_cast<float*>(smem + kOffQs);   // [2][32]: a head's score factor
  float* stats = reinterpret_cast<float*>(smem + kOffStats); // [2][32][3]: m, l, gain exponent

  // ---- prologue: pages per sequence and their prefix sums (lengths and
  // block tables are read before the wait; the pools, scales and queries
  // may belong to the previous kernel) ----
  const int B = p.B;
  auto pages_of = [&](int b) {
    const int len = p.seq_lens[b];
    return len > 0 ? min((len + kPS - 1) / kPS, p.bt_stride) : 0;
  };
  {
    const int chunk = (B + kThreads - 1) / kThreads;
    const int c0 = min(B, tid * chunk), c1 = min(B, c0 + chunk);
    int sum = 0;
    for (int b = c0; b < c1; ++b) sum += pages_of(b);
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) wsum[warp] = incl;
    if (tid == 0) {
      for (int i = 0; i < kStages; ++i) {
        mbar_init(b_full(i), 1);
        mbar_init(b_empty(i), 1);
      }
      for (int u = 0; u < 2; ++u) {
        mbar_init(b_sfull(u), 1);
        mbar_init(b_sfree(u), 4);
        mbar_init(b_pfull(u), 4);
        mbar_init(b_pvdone(u), 1);
        mbar_init(b_qready(u), 4);
        mbar_init(b_segdone(u), 4);
      }
      mbar_init(b_ofull, 1);
      mbar_init(b_ofree, 4);
      fence_mbar_init();
    }
    __syncthreads();
    int off = 0;
    for (int w = 0; w < warp; ++w) off += wsum[w];
    int run = off + incl - sum;
    for (int b = c0; b < c1; ++b) {
      pre[b] = run;
      run += pages_of(b);
    }
    if (tid == kThreads - 1) pre[B] = off + incl;
  }
  if (warp == 5) tmem_alloc(smem_u32(tmem_slot), kTCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int total = pre[B];
  const int n = min(static_cast<int>(gridDim.x), total);   // CTAs with pages
  const int c = static_cast<int>(blockIdx.x);
  const int lo = c < n ? static_cast<int>(static_cast<long long>(c) * total / n) : 0;
  const int hi = c < n ? static_cast<int>(static_cast<long long>(c + 1) * total / n) : 0;
  const int n_tiles = hi - lo;
  // the sequence holding global page x < total (skipping empty sequences)
  auto seq_of = [&](int x) {
    int a = 0, z = B - 1;
    while (a < z) {
      const int mid = (a + z + 1) >> 1;
      if (pre[mid] <= x) a = mid;
      else z = mid - 1;
    }
    return a;
  };
  // the CTA whose range holds global page x
  auto owner = [&](int x) { return static_cast<int>((static_cast<long long>(x + 1) * n - 1) / total); };

  bool ok = true;
  if (warp == 4) {
    // ---------------- TMA producer: lane i resolves the page of tile j0 + i ----
    if (n_tiles > 0) {
      pdl_wait_primary();
      const int oob = p.num_pages * kPS;  // a row past the pool: the box is zero-filled
      for (int j0 = 0; j0 < n_tiles && ok; j0 += 32) {
        int row = oob, sp = 0;  // a bad page id: zero codes, and page 0's scales (a valid address)
        if (j0 + lane < n_tiles) {
          const int x = lo + j0 + lane, b = seq_of(x);
          const int page = p.block_table[static_cast<int64_t>(b) * p.bt_stride + (x - pre[b])];
          if (page >= 0 && page < p.num_pages) {
            row = page * kPS;
            sp = page;
          } else {
            set_device_error(p.err_word, TS_DEVERR_PAGE_RANGE);
          }
        }
        const int cnt = min(32, n_tiles - j0);
        for (int i = 0; i < cnt; ++i) {
          const int rw = __shfl_sync(0xffffffffu, row, i);
          const int pg = __shfl_sync(0xffffffffu, sp, i);
          const int j = j0 + i, s = j % kStages;
          if (lane == 0) {
            if (j >= kStages) ok = mbar_wait(b_empty(s), ((j / kStages) - 1) & 1);
            if (ok) {
              const uint32_t st = smem_u32(smem + s * kStage);
              mbar_arrive_expect_tx(b_full(s), 2 * kTile + 2 * kScaleBytes);
              tma_load_3d(st, &kmap, 0, rw, 0, b_full(s));
              tma_load_3d(st + kTile, &vmap, 0, rw, 0, b_full(s));
              const int64_t so = static_cast<int64_t>(pg) * kPS * kHkv;
              bulk_g2s(st + 2 * kTile, p.k_scale + so, kScaleBytes, b_full(s));
              bulk_g2s(st + 2 * kTile + kScaleBytes, p.v_scale + so, kScaleBytes, b_full(s));
            }
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) break;
        }
      }
      if (!ok && lane == 0) set_device_error(p.err_word, TS_DEVERR_TIMEOUT);
    }
  } else if (warp == 5) {
    // ---------------- MMA issuer ----------------
    // Blocking order: S(j + 1) once tile j + 1 has landed and the softmax
    // has read S(j - 1) (two S buffers), then P V(j) once P(j) is written.
    // No wait here depends on a product not yet issued.
    if (lane == 0 && n_tiles > 0) {
      constexpr uint32_t iS = idesc_e4m3(128, kKeys, 0);
      constexpr uint32_t iO = idesc_e4m3(128, kD, 1);
      // segment boundaries followed incrementally (one search per segment)
      auto seg_end = [&](int j) { return min(n_tiles, pre[seq_of(lo + j) + 1] - lo); };
      int s_seg = 0, s_next = seg_end(0);  // the S pointer's segment; first tile of the next
      auto issue_s = [&](int js) {
        const int s = js % kStages;
        if (!mbar_wait(b_full(s), (js / kStages) & 1)) return false;
        if (js >= 2 && !mbar_wait(b_sfree(js & 1), ((js >> 1) - 1) & 1)) return false;
        const bool first = js == 0 || js == s_next;
        if (js > 0 && first) {
          ++s_seg;
          s_next = seg_end(js);
        }
        if (first && !mbar_wait(b_qready(s_seg & 1), (s_seg >> 1) & 1)) return false;
        tc_fence_after();
        const uint32_t sK = smem_u32(smem + s * kStage);
        // S = Q K^T: K-steps of 32 dims (32 bytes of each 128-byte key row)
#pragma unroll
        for (int i = 0; i < kD / 32; ++i)
          mma_e4m3_tmem_a(tmem + kTS + (js & 1) * kKeys, tmem + kTQ + (s_seg & 1) * 32 + i * 8,
                          desc_sw128(sK + i * 32), iS, i > 0 ? 1u : 0u);
        mma_commit(b_sfull(js & 1));
        return true;
      };
      ok = issue_s(0);
      int j_seg = -1, j_next = 0;  // the P V pointer's segment; first tile of the next
      for (int j = 0; j < n_tiles && ok; ++j) {
        const bool j_starts = j == j_next;
        if (j_starts) {
          ++j_seg;
          j_next = seg_end(j);
        }
        const bool j_ends = j + 1 == j_next;
        if (j + 1 < n_tiles) {
          ok = issue_s(j + 1);
          if (!ok) break;
        }
        // P V(j) once P(j) is written and, for a segment's first tile, O has
        // been read out for the segment before
        ok = mbar_wait(b_pfull(j & 1), (j >> 1) & 1);
        if (ok && j_starts && j_seg >= 1) ok = mbar_wait(b_ofree, (j_seg - 1) & 1);
        if (!ok) break;
        tc_fence_after();
        const int s = j % kStages;
        const uint32_t sV = smem_u32(smem + s * kStage + kTile);
        // O += P V: V MN-major (a key row of 128 codes per 128-byte row), K-steps of 32 keys
#pragma unroll
        for (int ks = 0; ks < kKeys / 32; ++ks)
          mma_e4m3_tmem_a(tmem + kTO, tmem + kTP + (j & 1) * 32 + ks * 8,
                          desc_sw128(sV + ks * 4096, kTile, 1024), iO, (ks > 0 || !j_starts) ? 1u : 0u);
        mma_commit(b_pvdone(j & 1));
        mma_commit(b_empty(s));
        if (j_ends) mma_commit(b_ofull);
      }
      if (!ok) set_device_error(p.err_word, TS_DEVERR_TIMEOUT);
    }
  } else if (warp < 4) {
    // ---------------- softmax: thread = TMEM lane (query head h, term k) ----------------
    // The head's four lanes split a tile's 16 keys (of its kv head): lane k
    // takes keys 4k .. 4k + 3, each summed over the head's three terms.
    const int h = tid >> 2, k = tid & 3, kvh = h / kG;
    const bool upper = (lane >> 4) != 0;  // the warp's second kv head (kv heads 2 warp, 2 warp + 1)
    const uint32_t trow = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    {
      // P is zero outside a row's own kv head: both buffers cleared once
      uint32_t z[16];
#pragma unroll
      for (int x = 0; x < 16; ++x) z[x] = 0u;
#pragma unroll
      for (int cc = 0; cc < 64; cc += 16) tmem_st16(trow + kTP + cc, z);
      tmem_wait_st();
    }
    int seg = 0;
    for (int j = 0; j < n_tiles && ok; ++seg) {
      const int j_seg = j;
      const int b = seq_of(lo + j);
      const int j_end = min(n_tiles, pre[b + 1] - lo);
      const int L = p.seq_lens[b];
      // the head's score factor, written with the segment's Q terms
      ok = mbar_wait(b_qready(seg & 1), (seg >> 1) & 1);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      const float sl = qscale[(seg & 1) * kHq + h];
      float m = -INFINITY, l = 0.f;  // l: this lane's keys' share of the row sum
      int gexp = 0;
      for (; j < j_end && ok; ++j) {
        const int pi = lo + j - pre[b];
        const int valid = min(kPS, L - pi * kPS);  // keys of this page in the sequence
        const int u = j & 1, s = j % kStages;
        ok = mbar_wait(b_sfull(u), (j >> 1) & 1);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t ua[16], ub[16];
        tmem_ld16(trow + kTS + u * kKeys + (2 * warp) * kPS, ua);
        tmem_ld16(trow + kTS + u * kKeys + (2 * warp + 1) * kPS, ub);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(b_sfree(u));
        // reduce-scatter over the head's four lanes: lane k ends with keys 4k .. 4k + 3
        const bool k1 = (k >> 1) != 0, k0 = (k & 1) != 0;
        float half8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint32_t lo8 = upper ? ub[i] : ua[i], hi8 = upper ? ub[8 + i] : ua[8 + i];
          const float mine = __uint_as_float(k1 ? hi8 : lo8), give = __uint_as_float(k1 ? lo8 : hi8);
          half8[i] = mine + __shfl_xor_sync(0xffffffffu, give, 2);
        }
        float sc[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float give = k0 ? half8[i] : half8[4 + i];
          sc[i] = (k0 ? half8[4 + i] : half8[i]) + __shfl_xor_sync(0xffffffffu, give, 1);
        }
        // the stage's scale rows [16 tokens][8 kv heads] landed with its codes
        ok = mbar_wait(b_full(s), (j / kStages) & 1);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        const float* ksr = reinterpret_cast<const float*>(smem + s * kStage + 2 * kTile);
        const float* vsr = ksr + kPS * kHkv;
        float vs[4];
        float mx = -INFINITY, vmax = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int t = 4 * k + i;
          const bool in = t < valid;  // rows past the sequence: masked (their codes and scales may be anything)
          vs[i] = in ? vsr[t * kHkv + kvh] : 0.f;
          sc[i] = in ? sc[i] * ksr[t * kHkv + kvh] * sl : -INFINITY;
          mx = fmaxf(mx, sc[i]);
          vmax = fmaxf(vmax, vs[i]);
        }
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, 1));
        vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, 2));
        // gain 2^ge: the tile's largest value scale times it lies in [2^7, 2^8)
        const int ge = vmax >= 1.17549435e-38f ? min(126, max(-126, 7 - ilog2f(vmax))) : 126;
        const bool first = j == j_seg;
        const float m_new = first || mx > m + kSlack ? mx : m;
        const int g_new = first ? ge : min(gexp, ge);
        const bool need = !first && (m_new != m || g_new != gexp);
        if (__any_sync(0xffffffffu, need)) {
          // O holds P V of the earlier tiles: rescale it once the last is done
          ok = mbar_wait(b_pvdone((j - 1) & 1), ((j - 1) >> 1) & 1);
          if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const float alpha = need ? fast_exp2(m - m_new) * pow2i(max(-126, g_new - gexp)) : 1.f;
          const uint32_t to = trow + kTO;
#pragma unroll
          for (int c0 = 0; c0 < kD; c0 += 16) {
            uint32_t o[16];
            tmem_ld16(to + c0, o);
            tmem_wait_ld();
#pragma unroll
            for (int x = 0; x < 16; ++x) o[x] = __float_as_uint(__uint_as_float(o[x]) * alpha);
            tmem_st16(to + c0, o);
          }
          tmem_wait_st();
        }
        if (!first) l *= fast_exp2(m - m_new);
        m = m_new;
        gexp = g_new;
        const float gain = pow2i(gexp);
        float pv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float pr = fast_exp2(sc[i] - m);  // masked keys: 0
          l += pr;
          pv[i] = pr * vs[i] * gain;
        }
        // the three terms of this lane's four probabilities, then each lane
        // collects its own term of all 16 (lane k's keys from lane k)
        uint32_t tw[4];
        {
          uint32_t h0, m0, l0, h1, m1, l1;
          e4m3_terms(pv[0], pv[1], h0, m0, l0);
          e4m3_terms(pv[2], pv[3], h1, m1, l1);
          tw[0] = h0 | (h1 << 16);
          tw[1] = m0 | (m1 << 16);
          tw[2] = l0 | (l1 << 16);
          tw[3] = 0u;
        }
        uint32_t got[4];  // got[r]: lane k ^ r's keys in this lane's term (r = 0: its own)
        got[0] = pick4(tw, k);
#pragma unroll
        for (int r = 1; r < 4; ++r) got[r] = __shfl_xor_sync(0xffffffffu, pick4(tw, k ^ r), r);  // partner keeps term k ^ r
        uint32_t w[4];  // w[x]: keys 4x .. 4x + 3 in this lane's term
#pragma unroll
        for (int x = 0; x < 4; ++x) w[x] = pick4(got, x ^ k);
        // P(j)'s buffer was last read by P V(j - 2)
        if (j >= 2) {
          ok = mbar_wait(b_pvdone(u), ((j - 2) >> 1) & 1);
          if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        uint32_t pw[8];
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          pw[x] = upper ? 0u : w[x];
          pw[4 + x] = upper ? w[x] : 0u;
        }
        tmem_st8(trow + kTP + u * 32 + (2 * warp) * 4, pw);
        tmem_wait_st();
        // the last page's value rows past the sequence may hold NaN codes, and
        // 0 x NaN is NaN in the product: zero them (row tid = kv head tid / 16, token tid % 16)
        if (valid < kPS) {
          if ((tid & (kPS - 1)) >= valid) {
            uint4* vr = reinterpret_cast<uint4*>(smem + s * kStage + kTile + tid * 128);
#pragma unroll
            for (int x = 0; x < 8; ++x) vr[x] = make_uint4(0u, 0u, 0u, 0u);
          }
          fence_async_smem();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(b_pfull(u));
      }
      if (!ok) break;
      // the segment's statistics for the epilogue: m, the row sum, the gain
      l += __shfl_xor_sync(0xffffffffu, l, 1);
      l += __shfl_xor_sync(0xffffffffu, l, 2);
      if (k == 0) {
        float* st = stats + ((seg & 1) * kHq + h) * 3;
        st[0] = m;
        st[1] = l;
        st[2] = __int_as_float(gexp);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(b_segdone(seg & 1));
    }
    if (!ok) set_device_error(p.err_word, TS_DEVERR_TIMEOUT);
  } else {
    // ---------------- epilogue and query terms: TMEM lane r = (head, term) ----------------
    const int qw = warp & 3;
    const int r = qw * 32 + lane, h = r >> 2, term = r & 3;
    const int et = tid - 192;  // 0 .. 127
    const uint32_t trow = tmem + (static_cast<uint32_t>(qw * 32) << 16);
    pdl_wait_primary();
    // sequences without a key: O = 0, LSE = -inf
    for (int b = c; b < B; b += gridDim.x) {
      if (pre[b + 1] != pre[b]) continue;
      uint4* dst = reinterpret_cast<uint4*>(p.out + (static_cast<int64_t>(b) * kHq + h) * kD + term * 32);
#pragma unroll
      for (int x = 0; x < 4; ++x) dst[x] = make_uint4(0u, 0u, 0u, 0u);
      if (term == 0 && p.lse) p.lse[static_cast<int64_t>(b) * kHq + h] = -INFINITY;
    }
    // Q terms of sequence b's head h into Q buffer u (this lane's term of all
    // 128 elements), the head scaled by 2^e into [2^7, 2^8); its score factor
    // into qscale. The head's four lanes split the row (32 elements each),
    // compute all three terms of their share and exchange them.
    auto write_q = [&](int b, int u) {
      const uint4* src = reinterpret_cast<const uint4*>(p.q + (static_cast<int64_t>(b) * kHq + h) * kD + term * 32);
      uint4 raw[4];
      float amax = 0.f;
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        raw[v] = src[v];
        const uint32_t w4[4] = {raw[v].x, raw[v].y, raw[v].z, raw[v].w};
#pragma unroll
        for (int q2 = 0; q2 < 4; ++q2) {
          const float2 f = bf16x2_to_float2(w4[q2]);
          amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
        }
      }
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
      const int e = amax >= 1.17549435e-38f ? min(126, max(-126, 7 - ilog2f(amax))) : 0;
      const float up = pow2i(e);
      if (term == 0) qscale[u * kHq + h] = p.scale_log2 * pow2i(-e);
      // tw[i][t]: term t of this lane's elements 32 term + 4 i .. + 3 (t = 3: zero)
      uint32_t tw[8][4];
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const uint32_t w4[4] = {raw[v].x, raw[v].y, raw[v].z, raw[v].w};
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const float2 f0 = bf16x2_to_float2(w4[2 * half]), f1 = bf16x2_to_float2(w4[2 * half + 1]);
          uint32_t h0, m0, l0, h1, m1, l1;
          e4m3_terms(f0.x * up, f0.y * up, h0, m0, l0);
          e4m3_terms(f1.x * up, f1.y * up, h1, m1, l1);
          uint32_t (&t4)[4] = tw[2 * v + half];
          t4[0] = h0 | (h1 << 16);
          t4[1] = m0 | (m1 << 16);
          t4[2] = l0 | (l1 << 16);
          t4[3] = 0u;
        }
      }
      // words[8 x + i]: elements 32 x + 4 i .. + 3 in this lane's term (from lane x of the head)
      uint32_t words[32];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        uint32_t got[4];
        got[0] = pick4(tw[i], term);
#pragma unroll
        for (int r = 1; r < 4; ++r) got[r] = __shfl_xor_sync(0xffffffffu, pick4(tw[i], term ^ r), r);
#pragma unroll
        for (int x = 0; x < 4; ++x) words[8 * x + i] = pick4(got, x ^ term);
      }
      tmem_st16(trow + kTQ + u * 32, *reinterpret_cast<const uint32_t(*)[16]>(&words[0]));
      tmem_st16(trow + kTQ + u * 32 + 16, *reinterpret_cast<const uint32_t(*)[16]>(&words[16]));
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_qready(u));
    };
    // segments in order: sequence, first tile; the first two get their Q terms now
    int js0 = 0, js1 = n_tiles;  // first tiles of segments k and k + 1 ...
    auto next_start = [&](int j) { return j < n_tiles ? min(n_tiles, pre[seq_of(lo + j) + 1] - lo) : n_tiles; };
    if (n_tiles > 0) {
      write_q(seq_of(lo), 0);
      js1 = next_start(0);
      if (js1 < n_tiles) write_q(seq_of(lo + js1), 1);
    }
    for (int seg = 0; js0 < n_tiles && ok; ++seg) {
      const int b = seq_of(lo + js0);
      const int j_end = js1;
      const int js2 = next_start(js1);  // first tile of segment seg + 2
      ok = mbar_wait(b_segdone(seg & 1), (seg >> 1) & 1) && mbar_wait(b_ofull, seg & 1);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float* st = stats + ((seg & 1) * kHq + h) * 3;
      const float m = st[0], l = st[1];
      const int gexp = __float_as_int(st[2]);
      const float inv = l > 0.f ? 1.0f / (l * pow2i(gexp)) : 0.f;
      const float lse2 = l > 0.f ? m + log2f(l) : -INFINITY;
      // reduce-scatter of the four lanes' O rows: term t keeps dims [32 t, 32 t + 32)
      const bool b1 = (term >> 1) != 0, b0 = (term & 1) != 0;
      const uint32_t to = trow + kTO;
      float own[32];
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int cq = half * 16;
        uint32_t r0[16], r1[16], r2[16], r3[16];
        tmem_ld16(to + cq, r0);
        tmem_ld16(to + 32 + cq, r1);
        tmem_ld16(to + 64 + cq, r2);
        tmem_ld16(to + 96 + cq, r3);
        tmem_wait_ld();
        float ka[16], kb[16];
#pragma unroll
        for (int x = 0; x < 16; ++x) {
          const float s0 = __uint_as_float(b1 ? r0[x] : r2[x]), s1 = __uint_as_float(b1 ? r1[x] : r3[x]);
          ka[x] = __uint_as_float(b1 ? r2[x] : r0[x]) + __shfl_xor_sync(0xffffffffu, s0, 2);
          kb[x] = __uint_as_float(b1 ? r3[x] : r1[x]) + __shfl_xor_sync(0xffffffffu, s1, 2);
        }
#pragma unroll
        for (int x = 0; x < 16; ++x) {
          const float snd = b0 ? ka[x] : kb[x];
          own[cq + x] = (b0 ? kb[x] : ka[x]) + __shfl_xor_sync(0xffffffffu, snd, 1);
        }
      }
      // O read out: the next segment's first P V may overwrite it (the
      // statistics buffer is rewritten two segments on)
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_ofree);
      // own[x] is dim 32 term + x
      const int64_t orow = static_cast<int64_t>(b) * kHq + h;
      const int np = pre[b + 1] - pre[b];
      const bool whole = lo + js0 == pre[b] && j_end - js0 == np;
      if (whole) {
        uint4* dst = reinterpret_cast<uint4*>(p.out + orow * kD + term * 32);
#pragma unroll
        for (int x = 0; x < 32; x += 8)
          dst[x / 8] = make_uint4(float2_to_bf16x2(own[x] * inv, own[x + 1] * inv),
                                  float2_to_bf16x2(own[x + 2] * inv, own[x + 3] * inv),
                                  float2_to_bf16x2(own[x + 4] * inv, own[x + 5] * inv),
                                  float2_to_bf16x2(own[x + 6] * inv, own[x + 7] * inv));
        if (term == 0 && p.lse) p.lse[orow] = lse2 == -INFINITY ? -INFINITY : lse2 * kLn2C;
      } else {
        // a part of a cut sequence: its state in this CTA's slot (first or last segment)
        const int slot = 2 * c + (js0 == 0 ? 0 : 1);
        float4* dst = reinterpret_cast<float4*>(p.part_o + (static_cast<int64_t>(slot) * kHq + h) * kD + term * 32);
#pragma unroll
        for (int x = 0; x < 32; x += 4)
          dst[x / 4] = make_float4(own[x] * inv, own[x + 1] * inv, own[x + 2] * inv, own[x + 3] * inv);
        if (term == 0) p.part_lse[static_cast<int64_t>(slot) * kHq + h] = lse2;
        __threadfence();
        named_bar_sync(1, 128);
        const int c0 = owner(pre[b]), c1 = owner(pre[b + 1] - 1);
        if (et == 0) {
          unsigned long long* cnt = p.counters + b;
          const int k = arrive_count(cnt, p.epoch);
          const bool last = k == c1 - c0 + 1;
          if (k == 0) set_device_error(p.err_word, TS_DEVERR_TIMEOUT);
          // the last arrival is the last use of the counter in this launch:
          // cleared, so that a replay with the same epoch starts from zero
          if (last) atomicExch(cnt, 0ull);
          __threadfence();
          *arrived = last ? 1 : 0;
        }
        named_bar_sync(1, 128);
        if (*arrived) {
          __threadfence();
          // merge the parts in slot order: CTA c0's slot is its last segment's
          // unless its range starts at the sequence's first page
          const int lo0 = static_cast<int>(static_cast<long long>(c0) * total / n);
          float mx = -INFINITY;
          for (int cc = c0; cc <= c1; ++cc) {
            const int sl2 = 2 * cc + ((cc == c0 && lo0 < pre[b]) ? 1 : 0);
            mx = fmaxf(mx, __ldcg(p.part_lse + static_cast<int64_t>(sl2) * kHq + h));
          }
          float acc[32];
#pragma unroll
          for (int x = 0; x < 32; ++x) acc[x] = 0.f;
          float den = 0.f;
          for (int cc = c0; cc <= c1; ++cc) {
            const int sl2 = 2 * cc + ((cc == c0 && lo0 < pre[b]) ? 1 : 0);
            const float lk = __ldcg(p.part_lse + static_cast<int64_t>(sl2) * kHq + h);
            const float wk = lk == -INFINITY ? 0.f : fast_exp2(lk - mx);
            den += wk;
            const float4* src =
                reinterpret_cast<const float4*>(p.part_o + (static_cast<int64_t>(sl2) * kHq + h) * kD + term * 32);
#pragma unroll
            for (int x = 0; x < 32; x += 4) {
              const float4 v = __ldcg(src + x / 4);
              acc[x] += wk * v.x;
              acc[x + 1] += wk * v.y;
              acc[x + 2] += wk * v.z;
              acc[x + 3] += wk * v.w;
            }
          }
          const float idn = den > 0.f ? 1.0f / den : 0.f;
          uint4* dst = reinterpret_cast<uint4*>(p.out + orow * kD + term * 32);
#pragma unroll
          for (int x = 0; x < 32; x += 8)
            dst[x / 8] = make_uint4(float2_to_bf16x2(acc[x] * idn, acc[x + 1] * idn),
                                    float2_to_bf16x2(acc[x + 2] * idn, acc[x + 3] * idn),
                                    float2_to_bf16x2(acc[x + 4] * idn, acc[x + 5] * idn),
                                    float2_to_bf16x2(acc[x + 6] * idn, acc[x + 7] * idn));
          if (term == 0 && p.lse) p.lse[orow] = den > 0.f ? (mx + log2f(den)) * kLn2C : -INFINITY;
        }
      }
      // the Q terms of the segment after next go into this segment's Q buffer
      // (all of this segment's S products are done: its last P V is)
      if (js2 < n_tiles) write_q(seq_of(lo + js2), seg & 1);
      js0 = js1;
      js1 = js2;
    }
    if (!ok) set_device_error(p.err_word, TS_DEVERR_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, kTCols);
  }
}

// 3-D map over an fp8 pool [P * 16 rows][8 kv heads][128] bytes taken as
// (byte, pool row, kv head): a box is one page (16 rows) of all 8 heads,
// landing head by head, [8][16][128]; 128-byte swizzle, zero fill.
ts_status make_map(CUtensorMap* map, const void* pool, int num_pages) {
  auto fn = tensor_map_encoder();
  if (!fn) return fail(TS_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(num_pages) * kPS,
                        static_cast<cuuint64_t>(kHkv)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(kHkv) * kD, static_cast<cuuint64_t>(kD)};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(kD), kPS, static_cast<cuuint32_t>(kHkv)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult res = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(pool), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (res != CUDA_SUCCESS) return fail(TS_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(res));
  return TS_OK;
}

// Workspace after the error word: counters [B], part LSEs [2 n][32], part
// states [2 n][32][128], each 256-byte aligned.
struct MmaWorkspace {
  size_t counters, part_lse, part_o, total;
};
MmaWorkspace mma_workspace(int B, int n) {
  MmaWorkspace w;
  w.counters = kWorkspaceAlign;
  w.part_lse = align_up(w.counters + sizeof(unsigned long long) * static_cast<size_t>(B), kWorkspaceAlign);
  w.part_o = align_up(w.part_lse + sizeof(float) * 2 * static_cast<size_t>(n) * kHq, kWorkspaceAlign);
  w.total = align_up(w.part_o + sizeof(float) * 2 * static_cast<size_t>(n) * kHq * kD, kWorkspaceAlign);
  return w;
}

}  // namespace

// Runs the code-multiplying tensor-core kernel when TS_FP8_DECODE_PATH=mma
// asks for it, the shape is the one it is built for (bf16 queries, 32 query
// heads over 8 kv heads, head dim 128, page 16, at most 4096 sequences) and
// the workspace holds its partial states; TS_ERR_UNSUPPORTED otherwise, with
// nothing enqueued, so that the caller takes another path. Not the default:
// on the Llama-3-8B layer shape it measures 112.8 us against the CUDA-core
// kernel's 106.6 us.
ts_status launch_fp8_decode_mma(const void* q, const void* k_pool, const void* v_pool, const float* k_scale,
                                const float* v_scale, const int32_t* block_table, int32_t bt_stride,
                                const int32_t* seq_lens, int32_t B, int32_t H_q, int32_t H_kv, int32_t D,
                                int32_t page_size, int32_t num_pages, float scale, void* out, float* lse,
                                void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  const char* path = getenv("TS_FP8_DECODE_PATH");
  if (!path || std::strcmp(path, "mma") != 0) return TS_ERR_UNSUPPORTED;
  if (B <= 0 || B > kMaxB || H_q != kHq || H_kv != kHkv || D != kD || page_size != kPS || num_pages <= 0 ||
      bt_stride <= 0 || static_cast<long long>(num_pages) * kPS > INT32_MAX)
    return TS_ERR_UNSUPPORTED;
  const int n = paged_decode_ctas();
  if (n <= 0) return TS_ERR_UNSUPPORTED;
  const MmaWorkspace w = mma_workspace(B, n);
  if (workspace_bytes < w.total) return TS_ERR_UNSUPPORTED;
  unsigned char* wsb = static_cast<unsigned char*>(workspace);
  MmaParams prm;
  prm.q = static_cast<const __nv_bfloat16*>(q);
  prm.out = static_cast<__nv_bfloat16*>(out);
  prm.lse = lse;
  prm.block_table = block_table;
  prm.seq_lens = seq_lens;
  prm.k_scale = k_scale;
  prm.v_scale = v_scale;
  prm.B = B;
  prm.bt_stride = bt_stride;
  prm.num_pages = num_pages;
  prm.scale_log2 = scale * kLog2eC;
  prm.err_word = static_cast<uint32_t*>(workspace);
  prm.counters = reinterpret_cast<unsigned long long*>(wsb + w.counters);
  prm.part_lse = reinterpret_cast<float*>(wsb + w.part_lse);
  prm.part_o = reinterpret_cast<float*>(wsb + w.part_o);
  // a launch's epoch: distinct between launches, top bit set (no count or
  // index another kernel leaves in the workspace looks like one)
  static std::atomic<uint32_t> launches{0};
  prm.epoch = ((launches.fetch_add(1) + 1u) * 2654435761u) | 0x80000000u;
  CUtensorMap kmap, vmap;
  ts_status st = make_map(&kmap, k_pool, num_pages);
  if (st != TS_OK) return st;
  st = make_map(&vmap, v_pool, num_pages);
  if (st != TS_OK) return st;
  st = prepare_once(reinterpret_cast<const void*>(fp8_mma_kernel), [](const void* k) {
    ts_status s2 = cuda_check(cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem),
                              "fp8 tensor-core smem attribute");
    if (s2 != TS_OK) return s2;
    return cuda_check(cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout,
                                           static_cast<int>(cudaSharedmemCarveoutMaxShared)),
                      "fp8 tensor-core carveout attribute");
  });
  if (st != TS_OK) return st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(n));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  LaunchTrace trace("fp8_mma_kernel", stream);
  return cuda_check(cudaLaunchKernelEx(&cfg, fp8_mma_kernel, prm, kmap, vmap), "fp8 tensor-core launch");
}

}  // namespace ts
