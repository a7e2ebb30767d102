// ts_mla_paged_decode: absorbed multi-head latent attention (MLA) decode.
//
// TokenSpeed deep dive (wth2jhl.online), section 7 fig. 3 and 7.1: MLA decode
// as split-KV partial attention with an LSE per row, then a reduction. Every
// one of the 128 query heads attends the one shared latent head: scores over
// the 576-wide latent row (512 latent + 64 rope), values = its first 512 dims.
//
// Design for sm_103a. The 128 heads x 64 tokens of a page form an M=128,
// N=64 tensor-core product, but an fp32 accumulator of 128 x 512 would fill
// all 512 TMEM columns. So a thread-block cluster of two CTAs (two SMs) shares
// each page and splits the latent by columns:
//   CTA 0: Q[:, 0:288]  . K[:, 0:288]^T   and O[:, 0:256]   += P V[:, 0:256]
//   CTA 1: Q[:, 288:576] . K[:, 288:576]^T and O[:, 256:512] += P V[:, 256:512]
// Each CTA loads five 64-column atoms of the latent: CTA 0 atoms 0-4, CTA 1
// atoms 4-8. Atom 4 is loaded by both (the pair reads it at once, so the
// second read hits L2), and each takes half of its 16-column steps, so both
// issue 18 score products per page. Splitting at 256 would leave CTA 1 with 20
// and CTA 0 with 16, and the tensor-core issue rate bounds the kernel. The
// two partial score tiles are swapped through distributed shared memory and
// summed, so both CTAs hold the same full scores and the same softmax. Q (the MMA's A operand) and P live in TMEM, which keeps the
// small-N products from re-reading A from shared memory:
//   TMEM columns: Q [0,160)  S [160,224)  P [224,256)  O [256,512).
// Pages of the whole batch are cut into equal contiguous ranges, one per
// cluster; a sequence cut across clusters leaves fp32 partial states that a
// second kernel merges by LSE.
//
// Roles (384 threads): warp 0 TMA producer, warp 1 MMA issuer, warp 2 TMEM
// allocator, warps 4-11 softmax / epilogue (one head row and half of the
// tile's tokens per thread). Four K/V stages keep three pages in flight.
//
// Several query tokens per sequence (section 7.2, fold_sq_factor): with H
// heads and q_len tokens, F = the largest factor of q_len with H * F <= 128
// tokens are folded into the 128 rows of a tile (row r = token r / H of the
// step, head r % H), and the q_len / F steps of a sequence are separate
// "virtual sequences" of the cut. With q laid out [B, q_len, H, 576], the
// rows of virtual sequence v are the contiguous rows v * 128 .. v * 128 + 127,
// and likewise for O and LSE. Row r of step st attends keys up to
// L - q_len + st * F + r / H (causal among the new tokens).
#include <cmath>

#include "ts_tcgen05.cuh"

namespace ts {
namespace {

constexpr int kH = 128, kDqk = 576, kDv = 512, kPS = 64, kTok = 64, kTokHalf = kTok / 2;
constexpr int kAtomBytes = kTok * 128;  // 64 tokens x 64 bf16 = 8 KB (128-byte rows)
constexpr int kStages = 4;
constexpr int kStageBytes = 5 * kAtomBytes;
constexpr uint32_t kTQ = 0, kTS = 160, kTP = 224, kTO = 256, kTCols = 512;
constexpr int kThreadsMla = 384;
constexpr float kLog2eM = 1.4426950408889634f;
constexpr float kLn2M = 0.6931471805599453f;
constexpr float kSlackM = 8.0f;

// Shared memory map (from a 1024-aligned base).
constexpr int kOffStages = 0;
// Score exchange buffers hold one 32 x 32 fp32 block per softmax warp (its
// rows, its half of the tokens), 128-byte rows with the 16-byte chunks
// swizzled by row, so that one bulk copy moves a warp's block.
constexpr int kWarpX = 32 * kTokHalf * 4;                       // 4 KB
constexpr int kXBufBytes = 8 * kWarpX;                          // a tile's 128 x 64 scores
constexpr int kOffX = kOffStages + kStages * kStageBytes;       // score exchange, 2 tiles
constexpr int kOffRed = kOffX + 2 * kXBufBytes;                 // pair exchange: [2][2][128] floats
constexpr int kOffBars = kOffRed + 2 * 2 * kH * 4;              // 36 mbarriers
constexpr int kOffMisc = kOffBars + 36 * 8;
constexpr int kSmemMla = kOffMisc + 192;
static_assert(kSmemMla <= 232448, "shared memory of one CTA");

struct MlaParams {
  const __nv_bfloat16* q;   // [B, 128, 576]
  const int32_t* block_table;
  const int32_t* seq_lens;
  int32_t bt_stride, B, num_pages;
  float scale_log2;
  __nv_bfloat16* out;       // [B, 128, 512]
  float* lse;               // [B, 128] or null
  uint32_t* err_word;
  int2* split_info;         // per sequence: {first pair, (parts << 1) | slot of first part}
  float* part_o;            // [2 * pairs, 128, 512]
  float* part_lse;          // [2 * pairs, 128]
  // query tokens per sequence, tokens folded per tile, steps = q_len / fold,
  // log2 of the head count (B above counts virtual sequences: B_seq * steps)
  int32_t q_len, fold, steps, h_shift;
};

// Context length of virtual sequence v (the length of its sequence).
__device__ __forceinline__ int vlen(const int32_t* lens, int steps, int v) {
  return max(lens[steps == 1 ? v : v / steps], 0);
}

struct Tile {
  int b, pidx, rem, out_slot;  // rem: the sequence's tokens from this tile's first on
  bool first, last;
  __device__ int valid() const { return min(rem, kTok); }
};

// Deterministic walk over a cluster's page range (identical in every role).
struct Walker {
  const int32_t* lens;
  int B, k, steps;
  long long g, end, q_pages, r_pages, total;
  int b, pg, np, L, seg_left, out_slot;
  bool first_seg;

  __device__ void init(const MlaParams& p, int k_, long long start, long long end_, int b0, int p0,
                       long long qp, long long rp, long long tot) {
    lens = p.seq_lens;
    B = p.B;
    steps = p.steps;
    k = k_;
    g = start;
    end = end_;
    q_pages = qp;
    r_pages = rp;
    total = tot;
    b = b0;
    pg = p0;
    seg_left = 0;
    first_seg = true;
    np = 0;
    L = 0;
    if (b >= 0 && b < B) load();
  }
  __device__ void load() {
    L = vlen(lens, steps, b);
    np = (L + kPS - 1) / kPS;
  }
  // Next tile; false at the end of the range. `n_here` and the sequence's
  // first/last global page are returned for split bookkeeping.
  __device__ bool next(Tile& t, int* n_here_out = nullptr, long long* first_pg_out = nullptr) {
    if (g >= end || b < 0) return false;
    if (seg_left == 0) {
      while (b < B && (np == 0 || pg >= np)) {
        ++b;
        pg = 0;
        if (b < B) load();
      }
      if (b >= B) return false;
      const int n_here = static_cast<int>(min(static_cast<long long>(np - pg), end - g));
      const bool complete = (pg == 0) && (n_here == np);
      out_slot = complete ? -1 : (first_seg ? 2 * k : 2 * k + 1);
      seg_left = n_here;
      if (n_here_out) *n_here_out = n_here;
      if (first_pg_out) *first_pg_out = g - pg;
      t.first = true;
    } else {
      t.first = false;
      if (n_here_out) *n_here_out = 0;
    }
    t.b = b;
    t.pidx = pg;
    t.rem = L - pg * kPS;
    t.out_slot = out_slot;
    t.last = (seg_left == 1);
    ++g;
    ++pg;
    --seg_left;
    if (seg_left == 0) first_seg = false;
    return true;
  }
};

__global__ void __launch_bounds__(kThreadsMla, 1) mla_decode_kernel(const MlaParams p,
                                                                    const __grid_constant__ CUtensorMap kvmap) {
  // The whole 227 KB is in use, with no room to realign: the swizzled tiles
  // need a 1024-byte aligned base, which the declaration asks for and the
  // check below confirms (both CTAs of a cluster see the same offset).
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = smem_raw;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if ((smem_u32(smem) & 1023u) != 0) {
    if (tid == 0) set_device_error(p.err_word, TS_DEVERR_SMEM_ALIGN);
    return;
  }
  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  const int pair = blockIdx.x >> 1;
  const int n_pairs = gridDim.x >> 1;
  const int n_atoms = 5;                     // latent atoms this CTA loads
  const int atom0 = rank == 0 ? 0 : 4;       // first latent atom
  const int q_words = 160;                   // TMEM columns of this CTA's Q part
  // the shared atom 4 (stage atom 4 of CTA 0, 0 of CTA 1): CTA 0 takes its
  // 16-column steps 0-1, CTA 1 steps 2-3
  const int shared_atom = rank == 0 ? 4 : 0, shared_ks0 = rank == 0 ? 0 : 2;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBars);
  // [0,4) kv_full  [4,8) kv_empty  8 s_full  9 s_free  10 p_full  11 pv_done
  // 12 q_ready  [16,32) xfull[buf][w]: the peer's half rows for softmax warp w
  // landed in inbound buffer buf  [32,36) pair[q]: both softmax warps of TMEM
  // lane quarter q posted their value
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  long long* scratch = reinterpret_cast<long long*>(smem + kOffMisc + 16);  // warp sums (12)
  int* s_start = reinterpret_cast<int*>(smem + kOffMisc + 16 + 8 * (kThreadsMla / 32));
  const uint32_t x_peer = map_to_cta(smem_u32(smem + kOffX), peer);

  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(bar(i), 1);
      mbar_init(bar(4 + i), 1);
    }
    mbar_init(bar(8), 1);
    mbar_init(bar(9), 8);
    mbar_init(bar(10), 8);
    mbar_init(bar(11), 1);
    mbar_init(bar(12), 8);
    for (int i = 16; i < 32; ++i) mbar_init(bar(i), 1);
    for (int q = 0; q < 4; ++q) mbar_init(bar(32 + q), 2);
    s_start[0] = -1;
    s_start[1] = 0;
    fence_mbar_init();
  }

  // ---- range of this cluster: balanced cut of all pages ----------------------
  const int B = p.B;
  const int chunk = (B + kThreadsMla - 1) / kThreadsMla;
  const int lo = min(B, tid * chunk), hi = min(B, lo + chunk);
  long long mine = 0;
  bool has_empty = false;
  for (int b = lo; b < hi; ++b) {
    const int L = vlen(p.seq_lens, p.steps, b);
    if (L > 0)
      mine += (L + kPS - 1) / kPS;
    else if (b % n_pairs == pair && rank == 0)
      has_empty = true;
  }
  // Sequences with no tokens: O = 0, LSE = -inf, each written by a whole warp
  // (the lanes that found some hand their range to the warp in turn).
  unsigned todo = __ballot_sync(0xffffffffu, has_empty);
  while (todo != 0u) {
    const int src = __ffs(todo) - 1;
    todo &= todo - 1u;
    const int slo = __shfl_sync(0xffffffffu, lo, src), shi = __shfl_sync(0xffffffffu, hi, src);
    for (int b = slo; b < shi; ++b) {
      if (vlen(p.seq_lens, p.steps, b) > 0 || b % n_pairs != pair) continue;
      uint4* o4 = reinterpret_cast<uint4*>(p.out + static_cast<int64_t>(b) * kH * kDv);
      for (int i = lane; i < kH * kDv / 8; i += 32) o4[i] = make_uint4(0u, 0u, 0u, 0u);
      if (p.lse)
        for (int h = lane; h < kH; h += 32) p.lse[static_cast<int64_t>(b) * kH + h] = -INFINITY;
      if (lane == 0) p.split_info[b] = make_int2(pair, 0);
    }
  }
  long long incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) scratch[warp] = incl;
  __syncthreads();
  long long wbase = 0, total = 0;
  for (int w = 0; w < kThreadsMla / 32; ++w) {
    if (w < warp) wbase += scratch[w];
    total += scratch[w];
  }
  const long long excl = wbase + incl - mine;
  const long long q_pages = total / n_pairs, r_pages = total % n_pairs;
  const long long start = pair * q_pages + min(static_cast<long long>(pair), r_pages);
  const long long end = start + q_pages + (pair < r_pages ? 1 : 0);
  if (start < end && excl <= start && start < excl + mine) {
    long long off = excl;
    for (int b = lo; b < hi; ++b) {
      const int L = vlen(p.seq_lens, p.steps, b);
      const long long np = L > 0 ? (L + kPS - 1) / kPS : 0;
      if (start < off + np) {
        s_start[0] = b;
        s_start[1] = static_cast<int>(start - off);
        break;
      }
      off += np;
    }
  }
  if (warp == 2) tmem_alloc(smem_u32(tmem_slot), kTCols);
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the peer's barriers are initialised before any remote arrive
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const bool have_work = start < end && s_start[0] >= 0;
  bool ok = true;

  if (have_work && warp == 0 && lane == 0) {
    // ---------------- TMA producer ----------------
    Walker w;
    w.init(p, pair, start, end, s_start[0], s_start[1], q_pages, r_pages, total);
    Tile t;
    int n_here = 0;
    long long first_pg = 0;
    auto page_of = [&](const Tile& x) {
      // the block table has one row per sequence, not per virtual sequence
      const int seq = p.steps == 1 ? x.b : x.b / p.steps;
      return x.pidx < p.bt_stride ? p.block_table[static_cast<int64_t>(seq) * p.bt_stride + x.pidx] : -1;
    };
    // the page id of the next tile is loaded one tile ahead
    Walker wa = w;
    Tile ta;
    int page_next = wa.next(ta) ? page_of(ta) : -1;
    for (int j = 0; ok && w.next(t, &n_here, &first_pg); ++j) {
      const int page = page_next;
      page_next = wa.next(ta) ? page_of(ta) : -1;
      if (t.first && t.pidx == 0 && rank == 0) {
        const long long last_pg = first_pg + (w.np - 1);
        const long long big = r_pages * (q_pages + 1);
        const int k1 = static_cast<int>(last_pg < big ? last_pg / (q_pages + 1)
                                                      : r_pages + (last_pg - big) / max(q_pages, 1ll));
        p.split_info[t.b] = make_int2(pair, ((k1 - pair + 1) << 1) | (first_pg == start ? 0 : 1));
      }
      const int s = j % kStages;
      if (j >= kStages && !mbar_wait(bar(4 + s), ((j / kStages) & 1) ^ 1)) {
        ok = false;
        break;
      }
      int row = p.num_pages * kPS;  // past the pool: zero fill
      if (page >= 0 && page < p.num_pages)
        row = page * kPS;
      else
        set_device_error(p.err_word, TS_DEVERR_PAGE_RANGE);
      mbar_arrive_expect_tx(bar(s), n_atoms * kAtomBytes);
      const uint32_t st = smem_u32(smem + kOffStages + s * kStageBytes);
      for (int a = 0; a < n_atoms; ++a) tma_load_2d(st + a * kAtomBytes, &kvmap, (atom0 + a) * 64, row, bar(s));
    }
    if (!ok) set_device_error(p.err_word, TS_DEVERR_TIMEOUT);
  } else if (have_work && warp == 1 && lane == 0) {
    // ---------------- MMA issuer ----------------
    constexpr uint32_t iS = idesc_bf16(kH, kTok, 0);
    constexpr uint32_t iO = idesc_bf16(kH, 256, 1);
    Walker w;
    w.init(p, pair, start, end, s_start[0], s_start[1], q_pages, r_pages, total);
    auto issue_s = [&](int j) {
      const int s = j % kStages;
      if (!mbar_wait(bar(s), (j / kStages) & 1)) return false;
      tc_fence_after();
      const uint32_t st = smem_u32(smem + kOffStages + s * kStageBytes);
      // the first product issued (atom 0, step 0 on CTA 0; step 2 on CTA 1)
      // overwrites S, the others accumulate
#pragma unroll
      for (int a = 0; a < 5; ++a)
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          if (a != shared_atom || (ks >> 1) == (shared_ks0 >> 1))
            mma_bf16_tmem_a(tmem + kTS, tmem + kTQ + a * 32 + ks * 8, desc_sw128(st + a * kAtomBytes + ks * 32),
                            iS, (a == 0 && ks == shared_ks0) ? 0u : 1u);
      mma_commit(bar(8));
      return true;
    };
    // S runs two tiles ahead of P V: the softmax reads S(j+1) (freeing the S
    // columns, and reloading Q when tile j+2 starts a sequence) before it
    // writes P(j), so S(j+2) is issued ahead of PV(j).
    Tile cur, nxt, nn;
    bool has_cur = w.next(cur);
    bool has_nxt = has_cur && w.next(nxt);
    ok = mbar_wait(bar(12), 0) && (!has_cur || issue_s(0));
    if (ok && has_nxt) ok = mbar_wait(bar(9), 0) && issue_s(1);
    for (int j = 0; ok && has_cur; ++j) {
      const bool has_nn = has_nxt && w.next(nn);
      if (has_nn) {
        ok = mbar_wait(bar(9), (j + 1) & 1) && issue_s(j + 2);
        if (!ok) break;
      }
      ok = mbar_wait(bar(10), j & 1);
      if (!ok) break;
      tc_fence_after();
      const int s = j % kStages;
      const uint32_t st = smem_u32(smem + kOffStages + s * kStageBytes);
      // O[:, 0:256] += P V: V is MN-major over four 64-column atoms (LBO = atom stride)
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16_tmem_a(tmem + kTO, tmem + kTP + ks * 8, desc_sw128(st + ks * 2048, kAtomBytes, 1024), iO,
                        !(cur.first && ks == 0));
      mma_commit(bar(11));
      mma_commit(bar(4 + s));
      cur = nxt;
      has_cur = has_nxt;
      nxt = nn;
      has_nxt = has_nn;
    }
    if (!ok) set_device_error(p.err_word, TS_DEVERR_TIMEOUT);
  } else if (have_work && warp >= 4) {
    // ---------------- softmax / epilogue -------------------------------------
    // Eight warps: warp w reads TMEM lane quarter w % 4 (head rows 32(w%4) ..
    // +31, one row per thread) and handles one half of the columns: tokens
    // 32 hf .. 32 hf + 31 of each tile and O columns 128 hf .. 128 hf + 127 of
    // this CTA's 256. The two warps of a quarter agree on the row maximum (and
    // at the end on the row sum) through pair_exchange.
    const int sw = warp - 4;                  // softmax warp 0..7
    const int quarter = warp & 3, hf = sw >> 2;
    const int h = quarter * 32 + lane;        // head row
    const uint32_t trow = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const int dim0 = (rank == 0 ? 0 : 256) + hf * 128;  // first output column of this thread
    const int q_half = q_words / 2;           // TMEM columns of Q this warp loads
    Walker w;
    w.init(p, pair, start, end, s_start[0], s_start[1], q_pages, r_pages, total);
    auto load_q = [&](int b) {
      const uint4* src = reinterpret_cast<const uint4*>(
          p.q + (static_cast<int64_t>(b) * kH + h) * kDqk + atom0 * 64 + hf * q_half * 2);
#pragma unroll 1
      for (int c0 = 0; c0 < q_half; c0 += 16) {
        uint32_t u[16];
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          const uint4 v = src[c0 / 4 + x];
          u[4 * x] = v.x;
          u[4 * x + 1] = v.y;
          u[4 * x + 2] = v.z;
          u[4 * x + 3] = v.w;
        }
        tmem_st16(trow + kTQ + hf * q_half + c0, u);
      }
      tmem_wait_st();
    };
    // Swap one float per row with the other warp of this quarter (bounded
    // wait on the pair's mbarrier; the two warps make the same calls in the
    // same order, so the phase counter nx agrees).
    float* const red = reinterpret_cast<float*>(smem + kOffRed);
    int nx = 0;
    auto pair_exchange = [&](float v, float& other) {
      const int slot = nx & 1;
      red[(slot * 2 + hf) * kH + h] = v;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(32 + quarter));
      const bool got = __all_sync(0xffffffffu, mbar_wait(bar(32 + quarter), slot));
      other = red[(slot * 2 + (hf ^ 1)) * kH + h];
      ++nx;
      return got;
    };
    auto epilogue = [&](const Tile& t, float m, float l_half) {
      float l_other = 0.f;
      if (!pair_exchange(l_half, l_other)) return false;
      const float l = l_half + l_other;
      const float inv = l > 0.f ? 1.0f / l : 0.f;
      for (int c0 = 0; c0 < 128; c0 += 16) {
        uint32_t u[16];
        tmem_ld16(trow + kTO + hf * 128 + c0, u);
        tmem_wait_ld();
        if (t.out_slot < 0) {
          uint4* dst = reinterpret_cast<uint4*>(p.out + (static_cast<int64_t>(t.b) * kH + h) * kDv + dim0 + c0);
#pragma unroll
          for (int x = 0; x < 2; ++x) {
            uint4 pk;
            pk.x = float2_to_bf16x2(__uint_as_float(u[8 * x]) * inv, __uint_as_float(u[8 * x + 1]) * inv);
            pk.y = float2_to_bf16x2(__uint_as_float(u[8 * x + 2]) * inv, __uint_as_float(u[8 * x + 3]) * inv);
            pk.z = float2_to_bf16x2(__uint_as_float(u[8 * x + 4]) * inv, __uint_as_float(u[8 * x + 5]) * inv);
            pk.w = float2_to_bf16x2(__uint_as_float(u[8 * x + 6]) * inv, __uint_as_float(u[8 * x + 7]) * inv);
            dst[x] = pk;
          }
        } else {
          float4* dst = reinterpret_cast<float4*>(p.part_o + (static_cast<int64_t>(t.out_slot) * kH + h) * kDv + dim0 + c0);
#pragma unroll
          for (int x = 0; x < 4; ++x)
            dst[x] = make_float4(__uint_as_float(u[4 * x]) * inv, __uint_as_float(u[4 * x + 1]) * inv,
                                 __uint_as_float(u[4 * x + 2]) * inv, __uint_as_float(u[4 * x + 3]) * inv);
        }
      }
      const float lse = l > 0.f ? (m + log2f(l)) * kLn2M : -INFINITY;
      if (rank == 0 && hf == 0) {
        if (t.out_slot < 0) {
          if (p.lse) p.lse[static_cast<int64_t>(t.b) * kH + h] = lse;
        } else {
          p.part_lse[static_cast<int64_t>(t.out_slot) * kH + h] = lse;
        }
      }
      return true;
    };
    // Score exchange, pipelined one tile ahead: this warp reads its block of
    // S(j+1) from TMEM and sends it with one bulk copy into the peer's buffer
    // X[(j+1) % 2], completing on the peer's xfull[(j+1) % 2][sw], before the
    // softmax of tile j, so the transfer hides behind that math. The thread
    // keeps its own partial scores in registers. The copy's source is this
    // CTA's X[j % 2], whose inbound scores of tile j were just read. Both
    // directions of reuse are ordered by the copies themselves: the peer sends
    // its copy j+2 (into X[j % 2] here) only after it saw copy j+1 land, i.e.
    // after that copy finished reading X[j % 2].
    auto xoff = [&](int c) {  // 16-byte chunk c (0..7) of this thread's row in a warp block
      return static_cast<uint32_t>(sw * kWarpX + lane * (kTokHalf * 4) + ((c ^ (lane & 7)) << 4));
    };
    float mine[kTokHalf];
    auto send_next = [&](int jn, bool reload_q, int qb) {
      if (!__all_sync(0xffffffffu, mbar_wait(bar(8), jn & 1))) return false;
      tc_fence_after();
      {
        uint32_t u[2][16];
        tmem_ld16(trow + kTS + hf * kTokHalf, u[0]);
        tmem_ld16(trow + kTS + hf * kTokHalf + 16, u[1]);
        tmem_wait_ld();
#pragma unroll
        for (int x = 0; x < kTokHalf; ++x) mine[x] = __uint_as_float(u[x / 16][x % 16]);
      }
      if (reload_q) load_q(qb);  // S(jn) is read: Q may change for S(jn+1)
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(9));
      const int src = (jn + 1) & 1, dst = jn & 1;
#pragma unroll
      for (int c = 0; c < kTokHalf / 4; ++c)
        *reinterpret_cast<float4*>(smem + kOffX + src * kXBufBytes + xoff(c)) =
            make_float4(mine[4 * c], mine[4 * c + 1], mine[4 * c + 2], mine[4 * c + 3]);
      fence_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(16 + 8 * dst + sw), kWarpX);
        bulk_s2s_cluster(x_peer + dst * kXBufBytes + sw * kWarpX,
                         smem_u32(smem + kOffX + src * kXBufBytes + sw * kWarpX), kWarpX,
                         map_to_cta(bar(16 + 8 * dst + sw), peer));
      }
      return true;
    };
    Tile cur, nxt, nn, prev;
    bool has_cur = w.next(cur);
    if (has_cur) load_q(cur.b);
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(12));
    bool has_nxt = has_cur && w.next(nxt);
    if (has_cur) ok = send_next(0, has_nxt && nxt.first, nxt.b);
    float m = -INFINITY, l = 0.f;  // running max (log2 units) and this half's running sum
    bool prev_last = false;
    int n_tiles = 0;
    for (int j = 0; ok && has_cur; ++j) {
      const bool has_nn = has_nxt && w.next(nn);
      // full scores of tile j: this thread's partial + the peer's
      const int xb = j & 1;
      ok = mbar_wait(bar(16 + 8 * xb + sw), (j >> 1) & 1);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      float s[kTokHalf];
#pragma unroll
      for (int c = 0; c < kTokHalf / 4; ++c) {
        const float4 o = *reinterpret_cast<const float4*>(smem + kOffX + xb * kXBufBytes + xoff(c));
        s[4 * c] = mine[4 * c] + o.x;
        s[4 * c + 1] = mine[4 * c + 1] + o.y;
        s[4 * c + 2] = mine[4 * c + 2] + o.z;
        s[4 * c + 3] = mine[4 * c + 3] + o.w;
      }
      if (has_nxt && !send_next(j + 1, has_nn && nn.first, nn.b)) { ok = false; break; }
      // keys of this tile the row may see: the sequence's valid rows, and with
      // several query tokens only those up to the row's own position
      int lim = cur.rem;
      if (p.q_len > 1) lim -= p.q_len - 1 - ((cur.b % p.steps) * p.fold + (h >> p.h_shift));
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < kTokHalf; ++c) {
        s[c] = hf * kTokHalf + c < lim ? s[c] * p.scale_log2 : -INFINITY;
        mx = fmaxf(mx, s[c]);
      }
      {
        float mo;
        if (!pair_exchange(mx, mo)) { ok = false; break; }
        mx = fmaxf(mx, mo);
      }
      // PV(j-1) done: P and O are free; finish the previous sequence if it ended
      if (j > 0) {
        ok = mbar_wait(bar(11), (j - 1) & 1);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
        if (prev_last && !epilogue(prev, m, l)) { ok = false; break; }
      }
      if (cur.first) {
        m = mx;
        l = 0.f;
      } else if (__any_sync(0xffffffffu, mx > m + kSlackM)) {
        // both warps of the quarter see the same row maxima: same decision
        const float mnew = fmaxf(m, mx);
        const float alpha = m == -INFINITY ? 0.f : fast_exp2(m - mnew);
        m = mnew;
        l *= alpha;
        for (int c0 = 0; c0 < 128; c0 += 16) {
          uint32_t u[16];
          tmem_ld16(trow + kTO + hf * 128 + c0, u);
          tmem_wait_ld();
#pragma unroll
          for (int x = 0; x < 16; ++x) u[x] = __float_as_uint(__uint_as_float(u[x]) * alpha);
          tmem_st16(trow + kTO + hf * 128 + c0, u);
        }
        tmem_wait_st();
      }
      const float ms = m == -INFINITY ? 0.f : m;
      float ls = 0.f;
      {
        uint32_t u[16];
#pragma unroll
        for (int x = 0; x < 16; ++x) {
          const float e0 = fast_exp2(s[2 * x] - ms);
          const float e1 = fast_exp2(s[2 * x + 1] - ms);
          ls += e0 + e1;
          u[x] = float2_to_bf16x2(e0, e1);
        }
        tmem_st16(trow + kTP + hf * 16, u);
      }
      tmem_wait_st();
      l += ls;
      const int valid = cur.valid();
      if (valid < kTok) {
        // rows past the sequence's end hold whatever the pool has there (NaN
        // sentinels included): zero them so 0-weight rows stay 0 in P V
        const int sj = j % kStages;
        ok = mbar_wait(bar(sj), (j / kStages) & 1);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        unsigned char* st = smem + kOffStages + sj * kStageBytes;
        for (int i = sw * 32 + lane; i < (kTok - valid) * 4 * 8; i += 8 * 32) {
          const int row = valid + i / 32, a = (i / 8) & 3, c = i & 7;
          *reinterpret_cast<uint4*>(st + a * kAtomBytes + row * 128 + c * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_async_smem();  // each warp's zeros reach the MMA before its p_full arrive
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(10));
      prev = cur;
      prev_last = cur.last;
      cur = nxt;
      has_cur = has_nxt;
      nxt = nn;
      has_nxt = has_nn;
      n_tiles = j + 1;
    }
    if (ok && prev_last) {
      // the last tile's PV, then the last sequence's epilogue
      ok = mbar_wait(bar(11), (n_tiles - 1) & 1);
      if (__all_sync(0xffffffffu, ok)) {
        tc_fence_after();
        ok = epilogue(prev, m, l);
      } else {
        ok = false;
      }
    }
    if (!ok) set_device_error(p.err_word, TS_DEVERR_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no CTA leaves while its peer may still touch its shared memory
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, kTCols);
  }
}

// Merges the parts of split sequences: one warp per (sequence, head), 16 dims per lane.
__global__ void __launch_bounds__(256) mla_merge_kernel(const MlaParams p) {
  pdl_wait_primary();
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int b = warp / kH, h = warp % kH;
  if (b >= p.B) return;
  const int2 info = p.split_info[b];
  const int nparts = info.y >> 1;
  if (nparts <= 1) return;
  const int k0 = info.x, slot0 = info.y & 1;
  auto slot_of = [&](int i) { return i == 0 ? 2 * k0 + slot0 : 2 * (k0 + i); };
  float mx = -INFINITY;
  for (int i = 0; i < nparts; ++i) mx = fmaxf(mx, p.part_lse[static_cast<int64_t>(slot_of(i)) * kH + h]);
  const float ms = mx == -INFINITY ? 0.f : mx;
  float acc[16];
#pragma unroll
  for (int x = 0; x < 16; ++x) acc[x] = 0.f;
  float wsum = 0.f;
  for (int i = 0; i < nparts; ++i) {
    const int slot = slot_of(i);
    const float w = __expf(p.part_lse[static_cast<int64_t>(slot) * kH + h] - ms);
    wsum += w;
    const float4* src = reinterpret_cast<const float4*>(p.part_o + (static_cast<int64_t>(slot) * kH + h) * kDv);
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const float4 o = src[lane + 32 * x];
      acc[4 * x] += w * o.x;
      acc[4 * x + 1] += w * o.y;
      acc[4 * x + 2] += w * o.z;
      acc[4 * x + 3] += w * o.w;
    }
  }
  const float inv = wsum > 0.f ? 1.0f / wsum : 0.f;
  __nv_bfloat16* out = p.out + (static_cast<int64_t>(b) * kH + h) * kDv;
#pragma unroll
  for (int x = 0; x < 4; ++x) {
    uint2 pk;
    pk.x = float2_to_bf16x2(acc[4 * x] * inv, acc[4 * x + 1] * inv);
    pk.y = float2_to_bf16x2(acc[4 * x + 2] * inv, acc[4 * x + 3] * inv);
    *reinterpret_cast<uint2*>(out + (lane + 32 * x) * 4) = pk;
  }
  if (lane == 0 && p.lse) p.lse[static_cast<int64_t>(b) * kH + h] = wsum > 0.f ? ms + logf(wsum) : -INFINITY;
}

struct MlaWs {
  size_t split_info, part_o, part_lse, total;
};

MlaWs mla_layout(int B, int n_pairs) {
  MlaWs w;
  size_t off = kWorkspaceAlign;
  w.split_info = off;
  off = align_up(off + static_cast<size_t>(B) * sizeof(int2), kWorkspaceAlign);
  w.part_o = off;
  off = align_up(off + static_cast<size_t>(2) * n_pairs * kH * kDv * sizeof(float), kWorkspaceAlign);
  w.part_lse = off;
  off = align_up(off + static_cast<size_t>(2) * n_pairs * kH * sizeof(float), kWorkspaceAlign);
  w.total = off;
  return w;
}

int mla_pairs() {
  if (const char* env = getenv("TS_MLA_CLUSTERS")) {
    const int n = atoi(env);
    if (n > 0 && n <= 4096) return n;
  }
  return device_sm_count() / 2;
}

}  // namespace
}  // namespace ts

namespace ts {
namespace {

// Tokens folded into the 128 rows of a tile (TokenSpeed deep dive, section
// 7.2): the largest F with q_len % F == 0 and H * F <= 128. 0 if H * F != 128
// (the kernel needs full tiles).
int mla_fold(int H, int q_len) {
  if (H <= 0 || q_len <= 0 || H > kH) return 0;
  int best = 1;
  for (int f = 1; f <= q_len; ++f)
    if (q_len % f == 0 && H * f <= kH) best = f;
  return H * best == kH ? best : 0;
}

ts_status mla_launch(const void* q, const void* kv_pool, const int32_t* block_table, int32_t bt_stride,
                     const int32_t* seq_lens, int32_t B, int32_t q_len, int32_t H, int32_t D_qk,
                     int32_t D_v, int32_t page_size, int32_t num_pages, float scale, void* out, float* lse,
                     void* workspace, size_t workspace_bytes, void* stream, const char* who) {
  if (B < 0 || q_len < 1 || num_pages <= 0 || bt_stride <= 0 ||
      static_cast<long long>(num_pages) * page_size > INT32_MAX ||
      static_cast<long long>(B) * q_len > INT32_MAX / kH)
    return fail(TS_ERR_INVALID_ARG, "%s: bad sizes (B=%d q_len=%d P=%d bt=%d)", who, B, q_len, num_pages,
                bt_stride);
  const int fold = mla_fold(H, q_len);
  if (fold == 0 || D_qk != kDqk || D_v != kDv || page_size != kPS)
    return fail(TS_ERR_UNSUPPORTED,
                "%s: needs H * fold_sq_factor(H, q_len) == 128 (H=%d, q_len=%d), D_qk=576, D_v=512, "
                "page_size=64 (got %d, %d, %d)", who, H, q_len, D_qk, D_v, page_size);
  if (!std::isfinite(scale)) return fail(TS_ERR_INVALID_ARG, "%s: scale not finite", who);
  if (B == 0) return TS_OK;
  if (!q || !kv_pool || !block_table || !seq_lens || !out)
    return fail(TS_ERR_INVALID_ARG, "%s: null pointer", who);
  for (const void* ptr : {q, kv_pool, static_cast<const void*>(out)})
    if (reinterpret_cast<uintptr_t>(ptr) % 16 != 0)
      return fail(TS_ERR_INVALID_ARG, "%s: q, kv_pool and out must be 16-byte aligned", who);
  const int steps = q_len / fold;
  const int Bv = B * steps;
  const int pairs = mla_pairs();
  if (pairs <= 0) return fail(TS_ERR_CUDA, "%s: cannot query the SM count", who);
  const MlaWs ws = mla_layout(Bv, pairs);
  if (!workspace || workspace_bytes < ws.total)
    return fail(TS_ERR_WORKSPACE, "%s: workspace %zu B < %zu B needed", who, workspace_bytes, ws.total);
  if (reinterpret_cast<uintptr_t>(workspace) % kWorkspaceAlign != 0)
    return fail(TS_ERR_WORKSPACE, "%s: workspace must be 256-byte aligned", who);
  auto enc = tensor_map_encoder();
  if (!enc) return fail(TS_ERR_CUDA, "%s: cuTensorMapEncodeTiled is unavailable", who);
  CUtensorMap kvmap;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(kDqk), static_cast<cuuint64_t>(num_pages) * kPS};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(kDqk) * 2};
  cuuint32_t box[2] = {64, kTok};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(&kvmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(kv_pool), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(TS_ERR_CUDA, "%s: cuTensorMapEncodeTiled failed (%d)", who, static_cast<int>(r));

  MlaParams prm;
  prm.q = static_cast<const __nv_bfloat16*>(q);
  prm.block_table = block_table;
  prm.seq_lens = seq_lens;
  prm.bt_stride = bt_stride;
  prm.B = Bv;
  prm.num_pages = num_pages;
  prm.scale_log2 = scale * kLog2eM;
  prm.out = static_cast<__nv_bfloat16*>(out);
  prm.lse = lse;
  unsigned char* wsb = static_cast<unsigned char*>(workspace);
  prm.err_word = reinterpret_cast<uint32_t*>(wsb);
  prm.split_info = reinterpret_cast<int2*>(wsb + ws.split_info);
  prm.part_o = reinterpret_cast<float*>(wsb + ws.part_o);
  prm.part_lse = reinterpret_cast<float*>(wsb + ws.part_lse);
  prm.q_len = q_len;
  prm.fold = fold;
  prm.steps = steps;
  int h_shift = 0;
  while ((1 << h_shift) < H) ++h_shift;
  prm.h_shift = h_shift;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  ts_status st = prepare_once(reinterpret_cast<const void*>(mla_decode_kernel), [](const void* k) {
    return cuda_check(cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMla),
                      "mla smem attribute");
  });
  if (st != TS_OK) return st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs);
  cfg.blockDim = dim3(kThreadsMla);
  cfg.dynamicSmemBytes = kSmemMla;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  {
    LaunchTrace trace("mla_decode_kernel", s);
    st = cuda_check(cudaLaunchKernelEx(&cfg, mla_decode_kernel, prm, kvmap), "mla decode launch");
  }
  if (st != TS_OK) return st;
  cudaLaunchAttribute pattr[1];
  pattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pattr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t mcfg = {};
  const long long warps = static_cast<long long>(Bv) * kH;
  mcfg.gridDim = dim3(static_cast<unsigned>((warps + 7) / 8));
  mcfg.blockDim = dim3(256);
  mcfg.stream = s;
  mcfg.attrs = pattr;
  mcfg.numAttrs = 1;
  LaunchTrace trace("mla_merge_kernel", s);
  return cuda_check(cudaLaunchKernelEx(&mcfg, mla_merge_kernel, prm), "mla merge launch");
}

}  // namespace
}  // namespace ts

extern "C" size_t ts_mla_workspace_size(int32_t B, int32_t H, int32_t D_v) {
  const int pairs = ts::mla_pairs();
  if (B < 0 || H != ts::kH || D_v != ts::kDv || pairs <= 0) return 0;
  return ts::mla_layout(B, pairs).total;
}

extern "C" size_t ts_mla_multi_workspace_size(int32_t B, int32_t q_len, int32_t H, int32_t D_v) {
  const int pairs = ts::mla_pairs();
  const int fold = ts::mla_fold(H, q_len);
  if (B < 0 || fold == 0 || D_v != ts::kDv || pairs <= 0 ||
      static_cast<long long>(B) * q_len > INT32_MAX / ts::kH)
    return 0;
  return ts::mla_layout(B * (q_len / fold), pairs).total;
}

extern "C" ts_status ts_mla_paged_decode(const void* q, const void* kv_pool, const int32_t* block_table,
                                         int32_t bt_stride, const int32_t* seq_lens, int32_t B,
                                         int32_t H, int32_t D_qk, int32_t D_v, int32_t page_size,
                                         int32_t num_pages, float scale, void* out, float* lse,
                                         void* workspace, size_t workspace_bytes, void* stream) {
  const char* who = "ts_mla_paged_decode";
  if (H != ts::kH)
    return ts::fail(TS_ERR_UNSUPPORTED, "%s: needs H=128 (got %d); ts_mla_paged_decode_multi folds "
                    "fewer heads", who, H);
  return ts::mla_launch(q, kv_pool, block_table, bt_stride, seq_lens, B, 1, H, D_qk, D_v, page_size,
                        num_pages, scale, out, lse, workspace, workspace_bytes, stream, who);
}

extern "C" ts_status ts_mla_paged_decode_multi(const void* q, const void* kv_pool, const int32_t* block_table,
                                               int32_t bt_stride, const int32_t* seq_lens, int32_t B,
                                               int32_t q_len, int32_t H, int32_t D_qk, int32_t D_v,
                                               int32_t page_size, int32_t num_pages, float scale, void* out,
                                               float* lse, void* workspace, size_t workspace_bytes,
                                               void* stream) {
  return ts::mla_launch(q, kv_pool, block_table, bt_stride, seq_lens, B, q_len, H, D_qk, D_v, page_size,
                        num_pages, scale, out, lse, workspace, workspace_bytes, stream,
                        "ts_mla_paged_decode_multi");
}
