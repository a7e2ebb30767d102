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
// fp8 input path (TokenSpeed deep dive, section 1: bf16 / fp16 / fp8 inputs):
// the query rows and the latent rows arrive as e4m3fn codes with one float32
// token-group scale per row (tokenspeed 딥다이브, section 6-4). The same
// cluster design runs kind::f8f6f4 products with K = 32 per instruction, so a
// page costs each CTA 9 score products instead of 18. The latent arrives in
// 128-byte (128-code) atoms, three per CTA: CTA 0 dims 0-383, CTA 1 dims
// 256-639 (the last 64 past the row zero-filled); each CTA scores 9 K-steps
// of 32 dims. Scores take the query row's and the key token's scales. For
// P V the key token's scale is folded into P, times a power-of-two gain G
// that keeps P <= 2^8 under the largest scale seen (O is rescaled when G
// changes, as when the running maximum grows); P is split into two e4m3
// terms, hi = e4m3(P) and lo = e4m3(P - hi): 4 significant bits each, so P
// keeps a relative error of at most 2^-8, as a bf16 P would. O = acc / (G * l).
//
// Several query tokens per sequence (section 7.2, fold_sq_factor): with H
// heads and q_len tokens, F = the largest factor of q_len with H * F <= 128
// tokens are folded into the 128 rows of a tile (row r = token r / H of the
// step, head r % H), and the q_len / F steps of a sequence are separate
// "virtual sequences" of the cut. With q laid out [B, q_len, H, 576], the
// rows of virtual sequence v are the contiguous rows v * 128 .. v * 128 + 127,
// and likewise for O and LSE. Row r of step st attends keys up to
// L - q_len + st * F + r / H (causal among the new tokens).
#include <cuda_fp8.h>

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
// fp8 path: stage = three 128-code atoms + the page's 64 scales + the gain
// G the tile takes (1024-aligned)
constexpr int kStageBytesF8 = 25 * 1024;
constexpr int kOffScalesF8 = 3 * kAtomBytes;
constexpr int kOffGainF8 = kOffScalesF8 + kPS * 4;
// TMEM: Q [0,72) S [96,160) P hi|lo of tiles j even / odd [160,192) [192,224) O [256,512)
constexpr uint32_t kTSF8 = 96, kTPF8 = 160;
// P <= 2^8 * 2^slack must stay below e4m3's largest finite value, 448
constexpr float kSlackF8 = 0.5f;


// Shared memory map (from a 1024-aligned base).
constexpr int kOffStages = 0;
// Score exchange buffers hold one 32 x 32 fp32 block per softmax warp (its
// rows, its half of the tokens), 128-byte rows with the 16-byte chunks
// swizzled by row, so that one bulk copy moves a warp's block.
constexpr int kWarpX = 32 * kTokHalf * 4;                       // 4 KB
constexpr int kXBufBytes = 8 * kWarpX;                          // a tile's 128 x 64 scores
template <bool kF8>
struct MlaSmem {
  static constexpr int kStage = kF8 ? kStageBytesF8 : kStageBytes;
  static constexpr int kOffX = kOffStages + kStages * kStage;   // score exchange, 2 tiles
  static constexpr int kOffRed = kOffX + 2 * kXBufBytes;        // pair exchange: [2][2][128] floats
  static constexpr int kOffBars = kOffRed + 2 * 2 * kH * 4;     // 40 mbarriers
  static constexpr int kOffMisc = kOffBars + 40 * 8;
  static constexpr int kSmem = kOffMisc + 192;
  static_assert(kSmem <= 232448, "shared memory of one CTA");
};

struct MlaParams {
  const void* q;            // [B, 128, 576] bf16, or e4m3 codes on the fp8 path
  const float* q_scale;     // fp8 path: [B, 128] one scale per query row
  const float* kv_scale;    // fp8 path: [num_pages, 64] one scale per latent row
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

template <bool kF8>
__global__ void __launch_bounds__(kThreadsMla, 1) mla_decode_kernel(const MlaParams p,
                                                                    const __grid_constant__ CUtensorMap kvmap) {
  using Sm = MlaSmem<kF8>;
  constexpr int kOffX = Sm::kOffX, kOffRed = Sm::kOffRed, kOffBars = Sm::kOffBars, kOffMisc = Sm::kOffMisc;
  constexpr int kStageB = Sm::kStage;
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
  const int n_atoms = kF8 ? 3 : 5;           // latent atoms this CTA loads
  const int atom0 = rank == 0 ? 0 : (kF8 ? 2 : 4);  // first latent atom
  const int q_words = kF8 ? 72 : 160;        // TMEM columns of this CTA's Q part
  // the shared atom 4 (stage atom 4 of CTA 0, 0 of CTA 1): CTA 0 takes its
  // 16-column steps 0-1, CTA 1 steps 2-3
  const int shared_atom = rank == 0 ? 4 : 0, shared_ks0 = rank == 0 ? 0 : 2;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBars);
  // [0,4) kv_full  [4,8) kv_empty  8 s_full  9 s_free  10 p_full  11 pv_done
  // 12 q_ready  [16,32) xfull[buf][w]: the peer's half rows for softmax warp w
  // landed in inbound buffer buf  [32,36) pair[q]: both softmax warps of TMEM
  // lane quarter q posted their value  [36,40) fp8: the stage's scales are
  // prepared (scale x G, G stored)  13, 14: fp8 p_full and pv_done of the
  // second P buffer (fp8 keeps two, tiles j even / odd)
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  auto b_pfull = [&](int j) { return bar(kF8 && (j & 1) ? 13 : 10); };
  auto b_pvdone = [&](int j) { return bar(kF8 && (j & 1) ? 14 : 11); };
  auto ph = [](int j) { return kF8 ? (j >> 1) & 1 : j & 1; };  // parity of tile j's use of its buffer
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
    mbar_init(bar(13), 8);
    mbar_init(bar(14), 1);
    mbar_init(bar(12), 8);
    for (int i = 16; i < 32; ++i) mbar_init(bar(i), 1);
    for (int q = 0; q < 4; ++q) mbar_init(bar(32 + q), 2);
    for (int i = 0; i < kStages; ++i) mbar_init(bar(36 + i), 1);
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
      const uint32_t st = smem_u32(smem + kOffStages + s * kStageB);
      if constexpr (kF8) {
        // three 128-code atoms and the page's 64 token scales (a bad page
        // reads page 0's scales against zero-filled codes; it is flagged)
        mbar_arrive_expect_tx(bar(s), n_atoms * kAtomBytes + kPS * 4);
        for (int a = 0; a < n_atoms; ++a) tma_load_2d(st + a * kAtomBytes, &kvmap, (atom0 + a) * 128, row, bar(s));
        const int sp = (page >= 0 && page < p.num_pages) ? page : 0;
        bulk_g2s(st + kOffScalesF8, p.kv_scale + static_cast<int64_t>(sp) * kPS, kPS * 4, bar(s));
      } else {
        mbar_arrive_expect_tx(bar(s), n_atoms * kAtomBytes);
        for (int a = 0; a < n_atoms; ++a) tma_load_2d(st + a * kAtomBytes, &kvmap, (atom0 + a) * 64, row, bar(s));
      }
    }
    if (!ok) set_device_error(p.err_word, TS_DEVERR_TIMEOUT);
  } else if (have_work && warp == 1 && lane == 0) {
    // ---------------- MMA issuer ----------------
    constexpr uint32_t iS = kF8 ? idesc_e4m3(kH, kTok, 0) : idesc_bf16(kH, kTok, 0);
    constexpr uint32_t iO = kF8 ? idesc_e4m3(kH, 256, 1) : idesc_bf16(kH, 256, 1);
    Walker w;
    w.init(p, pair, start, end, s_start[0], s_start[1], q_pages, r_pages, total);
    auto issue_s = [&](int j) {
      const int s = j % kStages;
      if (!mbar_wait(bar(s), (j / kStages) & 1)) return false;
      tc_fence_after();
      const uint32_t st = smem_u32(smem + kOffStages + s * kStageB);
      if constexpr (kF8) {
        // 9 K-steps of 32 dims from dim 288 * rank: atom d / 128, byte d % 128
#pragma unroll
        for (int i = 0; i < 9; ++i) {
          const int d = static_cast<int>(rank) * 288 + 32 * i;
          mma_e4m3_tmem_a(tmem + kTSF8, tmem + kTQ + i * 8,
                          desc_sw128(st + (d / 128 - atom0) * kAtomBytes + d % 128), iS, i > 0 ? 1u : 0u);
        }
      } else {
        // the first product issued (atom 0, step 0 on CTA 0; step 2 on CTA 1)
        // overwrites S, the others accumulate
#pragma unroll
        for (int a = 0; a < 5; ++a)
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            if (a != shared_atom || (ks >> 1) == (shared_ks0 >> 1))
              mma_bf16_tmem_a(tmem + kTS, tmem + kTQ + a * 32 + ks * 8, desc_sw128(st + a * kAtomBytes + ks * 32),
                              iS, (a == 0 && ks == shared_ks0) ? 0u : 1u);
      }
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
      ok = mbar_wait(b_pfull(j), ph(j));
      if (!ok) break;
      tc_fence_after();
      const int s = j % kStages;
      const uint32_t st = smem_u32(smem + kOffStages + s * kStageB);
      if constexpr (kF8) {
        // O[:, 0:256] += (P_hi + P_lo) V: V is MN-major over this CTA's first two
        // 128-code atoms (LBO = atom stride); K-steps of 32 tokens (4 KB)
#pragma unroll
        for (int t = 0; t < 2; ++t)
#pragma unroll
          for (int ks = 0; ks < 2; ++ks)
            mma_e4m3_tmem_a(tmem + kTO, tmem + kTPF8 + (j & 1) * 32 + t * 16 + ks * 8,
                            desc_sw128(st + ks * 4096, kAtomBytes, 1024), iO, !(cur.first && t == 0 && ks == 0));
      } else {
        // O[:, 0:256] += P V: V is MN-major over four 64-column atoms (LBO = atom stride)
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          mma_bf16_tmem_a(tmem + kTO, tmem + kTP + ks * 8, desc_sw128(st + ks * 2048, kAtomBytes, 1024), iO,
                          !(cur.first && ks == 0));
      }
      mma_commit(b_pvdone(j));
      mma_commit(bar(4 + s));
      cur = nxt;
      has_cur = has_nxt;
      nxt = nn;
      has_nxt = has_nn;
    }
    if (!ok) set_device_error(p.err_word, TS_DEVERR_TIMEOUT);
  } else if (kF8 && have_work && warp == 3) {
    // ---------------- fp8 scale warp ----------------------------------------
    // Per tile: the largest token scale of the valid rows (two per lane, then
    // across the warp), the gain G = 2^(8 - e) with 2^e the smallest power of
    // two >= it (G of the segment: the smallest so far, reset at a segment's
    // start), and each token's scale x G written back in place (0 for rows
    // past the sequence's end, whose scales may be NaN). The softmax reads
    // these products and G once they are marked ready.
    Walker w;
    w.init(p, pair, start, end, s_start[0], s_start[1], q_pages, r_pages, total);
    Tile t;
    float G = 1.f;
    for (int j = 0; ok && w.next(t); ++j) {
      const int s = j % kStages;
      ok = __all_sync(0xffffffffu, mbar_wait(bar(s), (j / kStages) & 1));
      if (!ok) break;
      float* scl = reinterpret_cast<float*>(smem + kOffStages + s * kStageB + kOffScalesF8);
      const int valid = t.valid();
      const float c0 = lane < valid ? scl[lane] : 0.f, c1 = lane + 32 < valid ? scl[lane + 32] : 0.f;
      float cmax = fmax3(1e-30f, c0, c1);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, o));
      const uint32_t bits = __float_as_uint(cmax);
      const int e = static_cast<int>((bits >> 23) & 0xffu) - 127 + ((bits & 0x7fffffu) != 0u ? 1 : 0);
      const float Gt = __uint_as_float(static_cast<uint32_t>(127 + 8 - e) << 23);
      G = t.first ? Gt : fminf(G, Gt);
      scl[lane] = c0 * G;
      scl[lane + 32] = c1 * G;
      if (lane == 0) *reinterpret_cast<float*>(smem + kOffStages + s * kStageB + kOffGainF8) = G;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(36 + s));
    }
    if (!ok && lane == 0) set_device_error(p.err_word, TS_DEVERR_TIMEOUT);
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
      if constexpr (kF8) {
        // this CTA's 288 codes of the row (from dim 288 * rank), four per TMEM
        // column: warp hf 0 bytes 0-159 -> columns 0-39, hf 1 bytes 160-287 ->
        // columns 40-71
        const uint4* src = reinterpret_cast<const uint4*>(
            static_cast<const unsigned char*>(p.q) + (static_cast<int64_t>(b) * kH + h) * kDqk + rank * 288 +
            hf * 160);
#pragma unroll
        for (int c0 = 0; c0 < 32; c0 += 16) {
          uint32_t u[16];
#pragma unroll
          for (int x = 0; x < 4; ++x) {
            const uint4 v = src[c0 / 4 + x];
            u[4 * x] = v.x;
            u[4 * x + 1] = v.y;
            u[4 * x + 2] = v.z;
            u[4 * x + 3] = v.w;
          }
          tmem_st16(trow + kTQ + hf * 40 + c0, u);
        }
        if (hf == 0) {
          uint32_t u[8];
#pragma unroll
          for (int x = 0; x < 2; ++x) {
            const uint4 v = src[8 + x];
            u[4 * x] = v.x;
            u[4 * x + 1] = v.y;
            u[4 * x + 2] = v.z;
            u[4 * x + 3] = v.w;
          }
          tmem_st8(trow + kTQ + 32, u);
        }
      } else {
        const uint4* src = reinterpret_cast<const uint4*>(
            static_cast<const __nv_bfloat16*>(p.q) + (static_cast<int64_t>(b) * kH + h) * kDqk + atom0 * 64 +
            hf * q_half * 2);
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
      }
      tmem_wait_st();
    };
    // fp8: the query row's scale times scale * log2(e) (read where it is used:
    // a register kept a tile ahead made the softmax spill more)
    auto row_scale = [&](int b) {
      return kF8 ? p.q_scale[static_cast<int64_t>(b) * kH + h] * p.scale_log2 : p.scale_log2;
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
    auto epilogue = [&](const Tile& t, float m, float l_half, float ginv) {
      float l_other = 0.f;
      if (!pair_exchange(l_half, l_other)) return false;
      const float l = l_half + l_other;
      const float inv = l > 0.f ? ginv / l : 0.f;
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
        constexpr uint32_t kTSc = kF8 ? kTSF8 : kTS;  // S columns of this path
        tmem_ld16(trow + kTSc + hf * kTokHalf, u[0]);
        tmem_ld16(trow + kTSc + hf * kTokHalf + 16, u[1]);
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
    // fp8: gain G (a power of two) applied to P so that P <= 2^8 under the
    // largest token scale of the segment so far
    float G = 1.f;
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
      float Gj = 1.f;  // fp8: the gain G of this tile (from the scale warp)
      // fp8: the stage's 64 token scales x G (prepared by the scale warp; rows
      // past the end hold 0), read from shared memory where needed
      const float4* sc4 = reinterpret_cast<const float4*>(smem + kOffStages + (j % kStages) * kStageB +
                                                          kOffScalesF8) + hf * 8;
      float qg = 0.f;  // fp8: the query row's scale / G (its scores' factor in log2 units)
      if constexpr (kF8) {
        ok = mbar_wait(bar(36 + j % kStages), (j / kStages) & 1);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        Gj = *reinterpret_cast<const float*>(smem + kOffStages + (j % kStages) * kStageB + kOffGainF8);
        qg = row_scale(cur.b) * __frcp_rn(Gj);  // G is a power of two: exact
        // s = S x key-token scale x G here; the row's factor qg (> 0) applies
        // in the exponent and to the row maximum
#pragma unroll
        for (int c4 = 0; c4 < kTokHalf / 4; ++c4) {
          const float4 v = sc4[c4];
          const float2 a = make_float2(s[4 * c4] * v.x, s[4 * c4 + 1] * v.y);  // scalar: packed pairs spill
          const float2 b = make_float2(s[4 * c4 + 2] * v.z, s[4 * c4 + 3] * v.w);
          const int c = hf * kTokHalf + 4 * c4;
          s[4 * c4] = c < lim ? a.x : -INFINITY;
          s[4 * c4 + 1] = c + 1 < lim ? a.y : -INFINITY;
          s[4 * c4 + 2] = c + 2 < lim ? b.x : -INFINITY;
          s[4 * c4 + 3] = c + 3 < lim ? b.y : -INFINITY;
          mx = fmax3(mx, s[4 * c4], s[4 * c4 + 1]);
          mx = fmax3(mx, s[4 * c4 + 2], s[4 * c4 + 3]);
        }
        mx *= qg;
      } else {
#pragma unroll
        for (int c = 0; c < kTokHalf; ++c) {
          s[c] = hf * kTokHalf + c < lim ? s[c] * p.scale_log2 : -INFINITY;
          mx = fmaxf(mx, s[c]);
        }
      }
      {
        float mo;
        if (!pair_exchange(mx, mo)) { ok = false; break; }
        mx = fmaxf(mx, mo);
      }
      // Rescale O and l to a new maximum (both warps of the quarter see the
      // same row maxima: same decision) and, fp8, to a lower gain G (a tile
      // with a larger scale lowers G for every row alike).
      auto rescale_to = [&](float mnew, float gnew) {
        const float alpha = m == -INFINITY ? 0.f : fast_exp2(m - mnew);
        const float beta = alpha * (gnew / G);  // O carries G, l does not
        m = mnew;
        l *= alpha;
        G = gnew;
        for (int c0 = 0; c0 < 128; c0 += 16) {
          uint32_t u[16];
          tmem_ld16(trow + kTO + hf * 128 + c0, u);
          tmem_wait_ld();
#pragma unroll
          for (int x = 0; x < 16; ++x) u[x] = __float_as_uint(__uint_as_float(u[x]) * beta);
          tmem_st16(trow + kTO + hf * 128 + c0, u);
        }
        tmem_wait_st();
      };
      if constexpr (kF8) {
        const bool grow = !cur.first && __any_sync(0xffffffffu, mx > m + kSlackF8);
        const bool rescale = !cur.first && (grow || Gj < G);
        // O complete (PV(j-1) done) to finish the previous sequence or to
        // rescale; otherwise only P's buffer must be free: PV(j-2)
        if (j > 0 && (prev_last || rescale)) {
          ok = mbar_wait(b_pvdone(j - 1), ph(j - 1));
          if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
          tc_fence_after();
          if (prev_last && !epilogue(prev, m, l, 1.0f / G)) { ok = false; break; }
        } else if (j > 1) {
          ok = mbar_wait(b_pvdone(j - 2), ph(j - 2));
          if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
          tc_fence_after();
        }
        if (cur.first) {
          m = mx;
          l = 0.f;
          G = Gj;
        } else if (rescale) {
          rescale_to(grow ? fmaxf(m, mx) : m, fminf(G, Gj));
        }
      } else {
        // PV(j-1) done: P and O are free; finish the previous sequence if it ended
        if (j > 0) {
          ok = mbar_wait(b_pvdone(j - 1), ph(j - 1));
          if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
          tc_fence_after();
          if (prev_last && !epilogue(prev, m, l, 1.0f)) { ok = false; break; }
        }
        if (cur.first) {
          m = mx;
          l = 0.f;
        } else if (__any_sync(0xffffffffu, mx > m + kSlackM)) {
          rescale_to(fmaxf(m, mx), 1.f);
        }
      }
      const float ms = m == -INFINITY ? 0.f : m;
      float ls = 0.f;
      if constexpr (kF8) {
        // P = exp2(s * row scale - m) * key scale * G in two e4m3 terms:
        // hi = e4m3(P), lo = e4m3(P - hi), the difference taken in f16 (exact:
        // hi has 4 significant bits, P in f16 11); token t at byte t % 4 of
        // column t / 4, hi in columns [0, 16), lo in [16, 32)
#pragma unroll
        for (int half = 0; half < 2; ++half) {  // 16 tokens (4 columns of hi and of lo) at a time
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int xx = 0; xx < 4; ++xx) {
          const int x = half * 4 + xx;
          const float4 v = sc4[x];
          uint32_t hw[2], lw[2];
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const float2 ee = make_float2(fast_exp2(fmaf(s[4 * x + 2 * k], qg, -ms)),
                                          fast_exp2(fmaf(s[4 * x + 2 * k + 1], qg, -ms)));
            ls += ee.x + ee.y;
            const float2 w = make_float2(ee.x * (k == 0 ? v.x : v.z), ee.y * (k == 0 ? v.y : v.w));
            const __half2 wh = __floats2half2_rn(w.x, w.y);
            const __nv_fp8x2_storage_t h2 =
                __nv_cvt_halfraw2_to_fp8x2(static_cast<__half2_raw>(wh), __NV_SATFINITE, __NV_E4M3);
            const __half2 r = __hsub2(wh, __half2(__nv_cvt_fp8x2_to_halfraw2(h2, __NV_E4M3)));
            const __nv_fp8x2_storage_t l2 =
                __nv_cvt_halfraw2_to_fp8x2(static_cast<__half2_raw>(r), __NV_SATFINITE, __NV_E4M3);
            hw[k] = h2;
            lw[k] = l2;
          }
          hi[xx] = hw[0] | (hw[1] << 16);
          lo[xx] = lw[0] | (lw[1] << 16);
        }
        tmem_st4(trow + kTPF8 + (j & 1) * 32 + hf * 8 + half * 4, hi);
        tmem_st4(trow + kTPF8 + (j & 1) * 32 + 16 + hf * 8 + half * 4, lo);
        }
      } else {
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
        unsigned char* st = smem + kOffStages + sj * kStageB;
        // V: the first 4 (bf16) or 2 (fp8) atoms of the stage, 128-byte rows
        constexpr int kVAtoms = kF8 ? 2 : 4;
        for (int i = sw * 32 + lane; i < (kTok - valid) * kVAtoms * 8; i += 8 * 32) {
          const int row = valid + i / (kVAtoms * 8), a = (i / 8) % kVAtoms, c = i & 7;
          *reinterpret_cast<uint4*>(st + a * kAtomBytes + row * 128 + c * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_async_smem();  // each warp's zeros reach the MMA before its p_full arrive
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_pfull(j));
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
      ok = mbar_wait(b_pvdone(n_tiles - 1), ph(n_tiles - 1));
      if (__all_sync(0xffffffffu, ok)) {
        tc_fence_after();
        ok = epilogue(prev, m, l, 1.0f / G);
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

template <bool kF8>
ts_status mla_launch(const void* q, const float* q_scale, const void* kv_pool, const float* kv_scale,
                     const int32_t* block_table, int32_t bt_stride, const int32_t* seq_lens, int32_t B,
                     int32_t q_len, int32_t H, int32_t D_qk, int32_t D_v, int32_t page_size, int32_t num_pages,
                     float scale, void* out, float* lse, void* workspace, size_t workspace_bytes, void* stream,
                     const char* who) {
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
  if (!q || !kv_pool || !block_table || !seq_lens || !out || (kF8 && (!q_scale || !kv_scale)))
    return fail(TS_ERR_INVALID_ARG, "%s: null pointer", who);
  for (const void* ptr : {q, kv_pool, static_cast<const void*>(out), static_cast<const void*>(kv_scale)})
    if (reinterpret_cast<uintptr_t>(ptr) % 16 != 0)
      return fail(TS_ERR_INVALID_ARG, "%s: q, kv_pool, out (and kv_scale) must be 16-byte aligned", who);
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
  // the latent pool as (column, pool row); a box is one page of 128 bytes of
  // columns: 64 bf16 or 128 e4m3 codes (columns past 576 read as zero)
  const size_t esz = kF8 ? 1 : 2;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(kDqk), static_cast<cuuint64_t>(num_pages) * kPS};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(kDqk) * esz};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / esz), kTok};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(&kvmap, kF8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                   const_cast<void*>(kv_pool), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(TS_ERR_CUDA, "%s: cuTensorMapEncodeTiled failed (%d)", who, static_cast<int>(r));

  MlaParams prm;
  prm.q = q;
  prm.q_scale = q_scale;
  prm.kv_scale = kv_scale;
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
  ts_status st = prepare_once(reinterpret_cast<const void*>(mla_decode_kernel<kF8>), [](const void* k) {
    return cuda_check(cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, MlaSmem<kF8>::kSmem),
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
  cfg.dynamicSmemBytes = MlaSmem<kF8>::kSmem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  {
    LaunchTrace trace("mla_decode_kernel", s);
    st = cuda_check(cudaLaunchKernelEx(&cfg, mla_decode_kernel<kF8>, prm, kvmap), "mla decode launch");
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
  return ts::mla_launch<false>(q, nullptr, kv_pool, nullptr, block_table, bt_stride, seq_lens, B, 1, H, D_qk,
                               D_v, page_size, num_pages, scale, out, lse, workspace, workspace_bytes, stream, who);
}

extern "C" ts_status ts_mla_paged_decode_multi(const void* q, const void* kv_pool, const int32_t* block_table,
                                               int32_t bt_stride, const int32_t* seq_lens, int32_t B,
                                               int32_t q_len, int32_t H, int32_t D_qk, int32_t D_v,
                                               int32_t page_size, int32_t num_pages, float scale, void* out,
                                               float* lse, void* workspace, size_t workspace_bytes,
                                               void* stream) {
  return ts::mla_launch<false>(q, nullptr, kv_pool, nullptr, block_table, bt_stride, seq_lens, B, q_len, H, D_qk,
                               D_v, page_size, num_pages, scale, out, lse, workspace, workspace_bytes, stream,
                               "ts_mla_paged_decode_multi");
}

extern "C" ts_status ts_mla_paged_decode_fp8(const void* q_codes, const float* q_scale, const void* kv_codes,
                                             const float* kv_scale, const int32_t* block_table, int32_t bt_stride,
                                             const int32_t* seq_lens, int32_t B, int32_t q_len, int32_t H,
                                             int32_t D_qk, int32_t D_v, int32_t page_size, int32_t num_pages,
                                             float scale, void* out, float* lse, void* workspace,
                                             size_t workspace_bytes, void* stream) {
  return ts::mla_launch<true>(q_codes, q_scale, kv_codes, kv_scale, block_table, bt_stride, seq_lens, B, q_len, H,
                              D_qk, D_v, page_size, num_pages, scale, out, lse, workspace, workspace_bytes, stream,
                              "ts_mla_paged_decode_fp8");
}
