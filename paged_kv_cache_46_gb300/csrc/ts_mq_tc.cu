// Tensor-core path of ts_paged_decode_multi_attn: decode with q_len new query
// tokens per sequence (speculative verify) when their rows fill a real tile.
//
// TokenSpeed deep dive, section 7.2 (fold_sq_factor): folding query tokens
// into the head dimension turns the rows of a decode step into a tile that
// the tensor cores can take. Here one CTA takes HG (1, 2 or 4) kv heads of
// one sequence. The R = q_len x g query rows of head slot hs sit in TMEM
// lanes [hs * 128/HG, ...) (token j, query head (h0+hs)*g + i at row
// j*g + i; rows past R are zero). They attend the sequence's pages as
// S = Q K^T and O += P V on tcgen05, with the online softmax between them and
// the causal limit of each token (row of token j: keys before
// L - q_len + 1 + j). A key tile is 128 pool rows: 8 / HG pages of all HG
// heads, one TMA box per page and 64-column atom. A row scores only its own
// head's keys, and P is zero in the other heads' columns, so the product is
// block-diagonal over the heads.
//
// Roles (192 threads): warps 0-3 own one query row per thread (Q load,
// softmax, epilogue; warps whose 32 rows are all padding skip the softmax),
// warp 4 issues the TMA loads of K and V page boxes (one per lane; its lanes
// hold the page ids of the next key tile), warp 5 lane 0 issues the MMAs,
// S(j+1) or P V(j) whichever is ready first. TMEM: S (128 fp32 columns), O (D
// columns), P (two buffers of 64 columns of bf16 pairs, the P V product's A
// operand). K and V tiles sit in a 3-stage ring. At D = 128 the K, V and Q
// tiles are two 64-column atoms each, and one N = 128 product reads both of
// V's atoms.
//
// Tree verification (TokenSpeed deep dive, section 0: tree speculation): with
// a parents array the q_len draft tokens form a tree, and the row of token j
// sees the context (keys before L - q_len) and the draft keys of its own
// path from the context down to itself. Each row walks its path once, in a
// shared-memory copy of its sequence's parents, into a 64-bit mask; only the
// key tiles that hold draft keys test it.
#include <cmath>
#include <cstdlib>

#include "ts_tcgen05.cuh"

namespace ts {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

namespace {

constexpr int kBM = 128;  // query rows per tile
constexpr int kBN = 128;  // keys per tile
constexpr int kPS = 16;   // page size of this path
constexpr int kPagesPerTile = kBN / kPS;
constexpr int kThreads = 192;
constexpr int kAtom = kBN * 128;  // one [128 rows x 64 bf16] SW128 atom: 16 KB
constexpr int kStages = 3;        // K and V tile buffers
constexpr float kLog2eC = 1.4426950408889634f;
constexpr float kLn2C = 0.6931471805599453f;
constexpr float kSlack = 8.0f;
// Up to this many sequences the CTAs take them longest first (each CTA ranks
// the key-tile counts itself, B^2 / 192 comparisons per thread).
constexpr int kLongestFirstMaxB = 128;
// Draft tokens of a verified tree: one bit per token in a row's mask.
constexpr int kMaxTree = 64;

template <int kHD>
struct Layout {
  static constexpr int kAtoms = kHD / 64;
  static constexpr int kOffQ = 0;                          // kAtoms atoms of Q
  static constexpr int kOffK = kOffQ + kAtoms * kAtom;     // kStages buffers x kAtoms atoms
  static constexpr int kOffV = kOffK + kStages * kAtoms * kAtom;
  static constexpr int kOffBar = kOffV + kStages * kAtoms * kAtom;
  static constexpr int kOffTmem = kOffBar + 256;
  static constexpr int kOffPar = kOffTmem + 16;             // tree: the sequence's parents
  static constexpr int kSmem = kOffPar + kMaxTree * 4;
  static constexpr uint32_t kTmemO = 128;
  // two P buffers of 64 columns (bf16 pairs: key k of row r at column k/2):
  // the softmax writes P(j+1) while P V(j) still reads P(j)
  static constexpr uint32_t kTmemP = 128 + kHD;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr int kMinBlocks = 1;  // a softmax thread keeps its 128 scores in registers
};

struct MqParams {
  const __nv_bfloat16* q;       // [B, q_len, H_q, D]
  __nv_bfloat16* out;           // [B, q_len, H_q, D]
  float* lse;                   // [B, q_len, H_q] or nullptr
  const int32_t* block_table;   // [B, bt_stride]
  const int32_t* seq_lens;      // [B], counting the q_len new tokens
  const int32_t* parents;       // [B, q_len] draft-tree parents, or nullptr (causal)
  int32_t B, bt_stride, q_len, H_q, H_kv, g, num_pages;
  float scale_log2;
  uint32_t* err_word;
};

template <int kHD, int kHG>
__global__ void __launch_bounds__(kThreads, Layout<kHD>::kMinBlocks) mq_tc_kernel(
    const MqParams p, const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap) {
  using Lay = Layout<kHD>;
  constexpr int kAtoms = Lay::kAtoms;
  extern __shared__ __align__(1024) unsigned char smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Programmatic dependent launch: outputs are written only after the wait.
  pdl_launch_dependents();
  if ((smem_u32(smem) & 1023u) != 0) {
    if (tid == 0) set_device_error(p.err_word, TS_DEVERR_SMEM_ALIGN);
    return;
  }
  // A CTA takes HG kv heads of one sequence: head slot hs owns the lanes
  // [hs * Rw, (hs + 1) * Rw) of every tile, and a key tile holds TP pages of
  // all HG heads, so that one TMA box brings a page's rows of HG heads.
  constexpr int HG = kHG, TP = kPagesPerTile / HG, Rw = kBM / HG, kKeys = TP * kPS;
  const int hgroups = p.H_kv / HG;
  const int h0 = static_cast<int>(blockIdx.x % hgroups) * HG;  // first kv head
  int b = static_cast<int>(blockIdx.x / hgroups);
  {
    // CTAs start roughly in index order: handing out the sequences by
    // decreasing page count is the longest-first rule, which keeps the last
    // wave short when the lengths differ. Up to kLongestFirstMaxB sequences
    // each CTA ranks them exactly (ties by index), B^2 / 192 comparisons per
    // thread; beyond, by 32 buckets of page count (within a bucket by index),
    // three passes over the lengths. The scratch lies in the Q tile, which is
    // written only after the last read of it.
    auto pages = [&](int s) {
      const int len = p.seq_lens[s];
      return len > 0 ? min((len + kPS - 1) / kPS, p.bt_stride) : 0;
    };
    int* pick = reinterpret_cast<int*>(smem + Lay::kOffTmem + 8);
    if (p.B <= kLongestFirstMaxB) {
      for (int s = tid; s < p.B; s += kThreads) {
        const int ws = pages(s);
        int rank = 0;
        for (int t = 0; t < p.B; ++t) {
          const int wt = pages(t);
          rank += (wt > ws || (wt == ws && t < s)) ? 1 : 0;
        }
        if (rank == b) *pick = s;
      }
    } else {
      int* scratch = reinterpret_cast<int*>(smem + Lay::kOffQ);
      int* mx_s = scratch;       // the largest page count
      int* sel = scratch + 2;    // this CTA's bucket and its offset in it
      int* hist = scratch + 32;  // [32] sequences per bucket
      int* cnt = scratch + 64;   // [kThreads] bucket members in each thread's chunk
      int mx = 0;
      for (int s = tid; s < p.B; s += kThreads) mx = max(mx, pages(s));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      if (tid < 32) hist[tid] = 0;
      if (tid == 0) *mx_s = 0;
      __syncthreads();
      if (lane == 0) atomicMax(mx_s, mx);
      __syncthreads();
      const int maxp = *mx_s;
      auto bucket = [&](int s) { return 31 - min(31, pages(s) * 32 / (maxp + 1)); };  // 0: the longest
      for (int s = tid; s < p.B; s += kThreads) atomicAdd(&hist[bucket(s)], 1);
      __syncthreads();
      if (tid == 0) {
        int start = 0, k = 0;
        for (; k < 31 && start + hist[k] <= b; ++k) start += hist[k];
        sel[0] = k;
        sel[1] = b - start;
      }
      const int chunk = (p.B + kThreads - 1) / kThreads;
      const int s0 = min(p.B, tid * chunk), s1 = min(p.B, s0 + chunk);
      __syncthreads();
      const int kb = sel[0], off = sel[1];
      int c = 0;
      for (int s = s0; s < s1; ++s) c += bucket(s) == kb ? 1 : 0;
      cnt[tid] = c;
      __syncthreads();
      if (tid == 0) {
        int acc = 0;
        for (int t = 0; t < kThreads; ++t) {
          const int v = cnt[t];
          cnt[t] = acc;
          acc += v;
        }
      }
      __syncthreads();
      int before = cnt[tid];
      if (off >= before && off < before + c) {
        for (int s = s0; s < s1; ++s) {
          if (bucket(s) != kb) continue;
          if (before == off) *pick = s;
          ++before;
        }
      }
    }
    __syncthreads();
    b = *pick;
  }
  const int R = p.q_len * p.g;   // real rows
  const int L = p.seq_lens[b];   // tokens in the cache, the q_len new ones included
  const int n_pages = L > 0 ? min((L + kPS - 1) / kPS, p.bt_stride) : 0;
  const int n_kt = (n_pages + TP - 1) / TP;
  // Before this wait only the lengths are read (the queries, the pools with
  // freshly appended rows and the outputs may belong to the previous kernel).
  pdl_wait_primary();

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::kOffBar);
  // key tile j lives in buffer j % kStages as that buffer's (j / kStages)-th use
  auto b_kfull = [&](int buf) { return smem_u32(&bars[0 * kStages + buf]); };
  auto b_vfull = [&](int buf) { return smem_u32(&bars[1 * kStages + buf]); };
  auto b_kempty = [&](int buf) { return smem_u32(&bars[2 * kStages + buf]); };
  auto b_vempty = [&](int buf) { return smem_u32(&bars[3 * kStages + buf]); };
  const uint32_t b_sfull = smem_u32(&bars[4 * kStages]), b_sfree = smem_u32(&bars[4 * kStages + 1]);
  // per P buffer: written by the softmax (4 warps) / read by its P V product
  auto b_pfull = [&](int pb) { return smem_u32(&bars[4 * kStages + 2 + pb]); };
  auto b_pvdone = [&](int pb) { return smem_u32(&bars[4 * kStages + 4 + pb]); };
  static_assert((4 * kStages + 6) * 8 <= 256, "mbarriers fit their slot");
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Lay::kOffTmem);
  const uint32_t sQ = smem_u32(smem + Lay::kOffQ), sK = smem_u32(smem + Lay::kOffK);
  const uint32_t sV = smem_u32(smem + Lay::kOffV);
  constexpr int kTileKV = kAtoms * kAtom;  // one K (or V) tile: 128 keys x D

  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(b_kfull(i), 1);
      mbar_init(b_vfull(i), 1);
      mbar_init(b_kempty(i), 1);
      mbar_init(b_vempty(i), 1);
    }
    mbar_init(b_sfull, 1);
    mbar_init(b_sfree, 4);
    for (int i = 0; i < 2; ++i) {
      mbar_init(b_pfull(i), 4);
      mbar_init(b_pvdone(i), 1);
    }
    fence_mbar_init();
  }
  // Q tile: lane hs * Rw + r holds row r of head slot hs, (token r / g,
  // query head (h0 + hs) * g + r % g); rows past R are zero.
  if (warp < 4) {
    const int hs = tid / Rw, r = tid % Rw;
    const bool real = r < R;
    const uint4* src = reinterpret_cast<const uint4*>(
        p.q + ((static_cast<int64_t>(b) * p.q_len + (real ? r / p.g : 0)) * p.H_q + (h0 + hs) * p.g + r % p.g) *
                  kHD);
#pragma unroll
    for (int a = 0; a < kAtoms; ++a) {
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint4 v = real ? src[a * 8 + c] : make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(smem + Lay::kOffQ + a * kAtom + sw128_off(tid, c)) = v;
      }
    }
    fence_async_smem();
    if (p.parents != nullptr && tid < p.q_len)
      reinterpret_cast<int*>(smem + Lay::kOffPar)[tid] = p.parents[static_cast<int64_t>(b) * p.q_len + tid];
  }
  if (warp == 0) tmem_alloc(smem_u32(tmem_slot), Lay::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool ok = true;

  if (warp == 4) {
    // ---------------- TMA producer (lane 0 issues; lane i < 8 holds page i) ----
    const int oob = p.num_pages * kPS;  // a row coordinate past the pool: zero fill
    auto tile_rows = [&](int j) {       // this lane's page of key tile j, as a pool row
      const int pi = j * TP + lane;
      int row = oob;
      if (lane < TP && pi < n_pages) {
        const int page = p.block_table[static_cast<int64_t>(b) * p.bt_stride + pi];
        if (page >= 0 && page < p.num_pages)
          row = page * kPS;
        else
          set_device_error(p.err_word, TS_DEVERR_PAGE_RANGE);
      }
      return row;
    };
    // One box per lane: a page's 16 rows of the CTA's HG heads in one
    // 64-column atom, landing as [head][16 keys] blocks of 128-byte rows. A
    // single thread issuing the boxes one after another, or boxes of one
    // head, cap the tile rate well below HBM's.
    auto load_tile = [&](const CUtensorMap* map, uint32_t dst, uint32_t bar, int rows) {
      const int pg = lane / kAtoms, a = lane % kAtoms;
      const int row = __shfl_sync(0xffffffffu, rows, pg & (kPagesPerTile - 1));
      if (lane == 0) mbar_arrive_expect_tx(bar, kTileKV);
      __syncwarp();
      if (pg < TP) tma_load_3d(dst + a * kAtom + pg * (HG * kPS * 128), map, a * 64, row, h0, bar);
    };
    int rows = n_kt > 0 ? tile_rows(0) : oob;
    for (int j = 0; j < n_kt && ok; ++j) {
      const int rows_next = j + 1 < n_kt ? tile_rows(j + 1) : oob;  // page ids one tile ahead
      const int buf = j % kStages, ph = (j / kStages - 1) & 1;  // buffer; phase of its previous use
      ok = __shfl_sync(0xffffffffu, lane == 0 && j >= kStages ? mbar_wait(b_kempty(buf), ph) : true, 0);
      if (!ok) break;
      load_tile(&kmap, sK + buf * kTileKV, b_kfull(buf), rows);
      ok = __shfl_sync(0xffffffffu, lane == 0 && j >= kStages ? mbar_wait(b_vempty(buf), ph) : true, 0);
      if (!ok) break;
      load_tile(&vmap, sV + buf * kTileKV, b_vfull(buf), rows);
      rows = rows_next;
    }
    if (!ok && lane == 0) set_device_error(p.err_word, TS_DEVERR_TIMEOUT);
  } else if (warp == 5) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t iS = idesc_bf16(kBM, kBN, 0);
      constexpr uint32_t iO = idesc_bf16(kBM, kHD, 1);
      auto issue_s = [&](int js) {
        tc_fence_after();
        const uint32_t sKj = sK + (js % kStages) * kTileKV;
#pragma unroll
        for (int ks = 0; ks < kHD / 16; ++ks) {
          const uint32_t off = (ks >> 2) * kAtom + (ks & 3) * 32;  // atom, then 16 dims within it
          mma_bf16(tmem, desc_sw128(sQ + off), desc_sw128(sKj + off), iS, ks > 0);
        }
        mma_commit(b_sfull);
        mma_commit(b_kempty(js % kStages));
      };
      int js = 0;
      if (n_kt > 0) {
        ok = mbar_wait(b_kfull(0), 0);
        if (ok) issue_s(js++);
      }
      for (int j = 0; j < n_kt && ok; ++j) {
        const int buf = j % kStages;
        const unsigned long long t0 = globaltimer_ns();
        while (true) {
          if (js < n_kt && mbar_test(b_sfree, (js - 1) & 1) &&
              mbar_test(b_kfull(js % kStages), (js / kStages) & 1))
            issue_s(js++);
          if (mbar_test(b_pfull(j & 1), (j >> 1) & 1) && mbar_test(b_vfull(buf), (j / kStages) & 1)) break;
          if (globaltimer_ns() - t0 > kWaitLimitNs) {
            ok = false;
            break;
          }
        }
        if (!ok) break;
        tc_fence_after();
        const uint32_t sVj = sV + buf * kTileKV;
        // O[:, 0:D] += P V: V is MN-major over its 64-column atoms (LBO = atom stride)
#pragma unroll
        for (int ks = 0; ks < kBN / 16; ++ks)
          mma_bf16_tmem_a(tmem + Lay::kTmemO, tmem + Lay::kTmemP + (j & 1) * 64 + ks * 8,
                          desc_sw128(sVj + ks * 2048, kAtom, 1024),
                          iO, (j > 0 || ks > 0) ? 1u : 0u);
        mma_commit(b_pvdone(j & 1));
        mma_commit(b_vempty(buf));
      }
      if (!ok) set_device_error(p.err_word, TS_DEVERR_TIMEOUT);
    }
  } else {
    // ---------------- softmax warps: thread = query row ----------------
    // A warp whose 32 rows are all padding only keeps the barrier protocol:
    // its rows' S, P and O lanes are never read into an output. Row r of
    // head slot hs scores the tile's keys of its own head only: columns
    // [pb * HG * 16 + hs * 16, +16) for page block pb < TP; P is zero in the
    // other heads' columns, so the block-diagonal P V adds its head's V alone.
    const int hs = tid / Rw, r = tid % Rw;
    const bool warp_real = (warp * 32) % Rw < R;
    const uint32_t trow = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const uint32_t hcol = static_cast<uint32_t>(hs * kPS);
    const int jt = r / p.g;                            // this row's token
    const int ctx = L - p.q_len;                       // keys before the new tokens
    const bool tree = p.parents != nullptr;
    // keys below lim are visible (padding rows: none); with a tree, draft key
    // ctx + i is visible when bit i of anc is set (i on this row's path)
    const int lim = r >= R ? 0 : (tree ? ctx : ctx + 1 + jt);
    unsigned long long anc = 0ull;
    if (tree && r < R) {
      const int* par = reinterpret_cast<const int*>(smem + Lay::kOffPar);
      int a = jt;
      for (int step = 0; step < p.q_len && a >= 0; ++step) {
        anc |= 1ull << a;
        const int up = par[a];
        if (up >= a || up < -1) {  // not an earlier node: the path stops here
          set_device_error(p.err_word, TS_DEVERR_TREE);
          break;
        }
        a = up;
      }
    }
    // l: the row sum of exp2(s - m) for the LSE; lr: the same over P as
    // rounded to bf16 for the product, which normalises O, so that the
    // weights the product applied sum to one
    float m = -INFINITY, l = 0.f, lr = 0.f;
    if constexpr (HG > 1) {
      if (warp_real) {
      uint32_t z[16];
#pragma unroll
      for (int x = 0; x < 16; ++x) z[x] = 0u;
#pragma unroll
        for (int c = 0; c < 128; c += 16) tmem_st16(trow + Lay::kTmemP + c, z);  // both P buffers
        tmem_wait_st();
      }
    }
    for (int j = 0; j < n_kt && ok; ++j) {
      ok = mbar_wait(b_sfull, j & 1);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float s[kKeys];  // key c of the tile (page block c / 16) in s[c]
      if (warp_real) {
#pragma unroll
        for (int pb = 0; pb < TP; ++pb) {
          uint32_t u[16];
          tmem_ld16(trow + pb * HG * kPS + hcol, u);
          tmem_wait_ld();
#pragma unroll
          for (int x = 0; x < 16; ++x) s[pb * 16 + x] = __uint_as_float(u[x]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_sfree);
      float ms = 0.f;
      if (warp_real) {
        const int key0 = j * kKeys;
        // keys at or past this row's limit are masked (the sequence's end, the
        // causal limit of its token); the scale is folded into the exponent
        const float sl = p.scale_log2;
        float mx = -INFINITY;
        if (tree && key0 + kKeys > ctx) {  // a tile holding draft keys (same for every row)
#pragma unroll
          for (int c = 0; c < kKeys; ++c) {
            const int k = key0 + c, d = k - ctx;
            const bool vis = k < lim || (d >= 0 && k < L && ((anc >> (d & 63)) & 1ull) != 0ull);
            s[c] = vis ? s[c] * sl : -INFINITY;
            mx = fmaxf(mx, s[c]);
          }
        } else {
#pragma unroll
          for (int c = 0; c < kKeys; ++c) {
            s[c] = key0 + c < lim ? s[c] * sl : -INFINITY;
            mx = fmaxf(mx, s[c]);
          }
        }
        const bool need = mx > m + kSlack;
        if (j == 0) {
          m = mx;
        } else if (__any_sync(0xffffffffu, need)) {
          // O is rescaled: every P V issued so far (the last is P V(j-1)) must be done
          ok = mbar_wait(b_pvdone((j - 1) & 1), ((j - 1) >> 1) & 1);
          if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const float mnew = fmaxf(m, mx);
          const float alpha = m == -INFINITY ? 0.f : fast_exp2(m - mnew);
          m = mnew;
          l *= alpha;
          lr *= alpha;
#pragma unroll
          for (int c0 = 0; c0 < kHD; c0 += 16) {
            uint32_t u[16];
            tmem_ld16(trow + Lay::kTmemO + c0, u);
            tmem_wait_ld();
#pragma unroll
            for (int x = 0; x < 16; ++x) u[x] = __float_as_uint(__uint_as_float(u[x]) * alpha);
            tmem_st16(trow + Lay::kTmemO + c0, u);
          }
          tmem_wait_st();
        }
        ms = m == -INFINITY ? 0.f : m;
      }
      // P(j)'s buffer was last read by P V(j-2). Padding warps wait too, so
      // that an arrival for tile j only ever counts toward tile j's phase.
      if (j >= 2) {
        ok = mbar_wait(b_pvdone(j & 1), ((j >> 1) - 1) & 1);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      if (warp_real) {
        float2 ls2 = make_float2(0.f, 0.f), lr2 = make_float2(0.f, 0.f);
        // P straight into TMEM (the P V MMA reads its A operand there)
#pragma unroll
        for (int pb = 0; pb < TP; ++pb) {
          uint32_t pk[8];
#pragma unroll
          for (int x = 0; x < 16; x += 2) {
            const float e0 = fast_exp2(s[pb * 16 + x] - ms);
            const float e1 = fast_exp2(s[pb * 16 + x + 1] - ms);
            pk[x / 2] = float2_to_bf16x2(e0, e1);
            ls2 = __fadd2_rn(ls2, make_float2(e0, e1));
            lr2 = __fadd2_rn(lr2, bf16x2_to_float2(pk[x / 2]));
          }
          tmem_st8(trow + Lay::kTmemP + (j & 1) * 64 + (pb * HG * kPS + hcol) / 2, pk);
        }
        tmem_wait_st();
        l += ls2.x + ls2.y;
        lr += lr2.x + lr2.y;
      }
      // The last tile's V rows past the sequence may hold anything (NaN
      // included) and 0 * NaN is NaN in the product: zero them once landed.
      if (j == n_kt - 1 && (j + 1) * kKeys > L) {
        const int buf = j % kStages;
        ok = mbar_wait(b_vfull(buf), (j / kStages) & 1);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        // tile row t holds key (t / (HG * 16)) * 16 + t % 16 of its head
        if (j * kKeys + (tid / (HG * kPS)) * kPS + tid % kPS >= L) {
#pragma unroll
          for (int a = 0; a < kAtoms; ++a)
#pragma unroll
            for (int c = 0; c < 8; ++c)
              *reinterpret_cast<uint4*>(smem + Lay::kOffV + buf * kTileKV + a * kAtom + tid * 128 + c * 16) =
                  make_uint4(0, 0, 0, 0);
        }
        fence_async_smem();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_pfull(j & 1));
    }
    // epilogue: O row / l in bf16 and the LSE (no key: O = 0, LSE = -inf)
    if (ok && n_kt > 0) {
      ok = mbar_wait(b_pvdone((n_kt - 1) & 1), ((n_kt - 1) >> 1) & 1);
      if (!__all_sync(0xffffffffu, ok)) ok = false;
      else tc_fence_after();
    }
    if (ok && warp_real) {
      const bool real = r < R;
      const int64_t row = (static_cast<int64_t>(b) * p.q_len + jt) * p.H_q + (h0 + hs) * p.g + r % p.g;
      const float inv = lr > 0.f ? 1.0f / lr : 0.f;
#pragma unroll
      for (int c0 = 0; c0 < kHD; c0 += 16) {
        uint32_t u[16];
        if (n_kt > 0) {
          tmem_ld16(trow + Lay::kTmemO + c0, u);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int x = 0; x < 16; ++x) u[x] = 0u;
        }
        if (real) {
          uint4* dst = reinterpret_cast<uint4*>(p.out + row * kHD + c0);
#pragma unroll
          for (int x = 0; x < 16; x += 8)
            dst[x / 8] = make_uint4(float2_to_bf16x2(__uint_as_float(u[x]) * inv, __uint_as_float(u[x + 1]) * inv),
                                    float2_to_bf16x2(__uint_as_float(u[x + 2]) * inv, __uint_as_float(u[x + 3]) * inv),
                                    float2_to_bf16x2(__uint_as_float(u[x + 4]) * inv, __uint_as_float(u[x + 5]) * inv),
                                    float2_to_bf16x2(__uint_as_float(u[x + 6]) * inv, __uint_as_float(u[x + 7]) * inv));
        }
      }
      if (real && p.lse) p.lse[row] = l > 0.f ? (m + log2f(l)) * kLn2C : -INFINITY;
    }
    if (!ok) set_device_error(p.err_word, TS_DEVERR_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, Lay::kTmemCols);
  }
}

// 3-D map over a pool [P * 16 rows][H_kv][D] bf16 taken as (column, pool
// row, kv head): a box is one page (16 rows) of hg heads in one 64-column
// atom and lands head by head, [hg][16][64]; 128-byte swizzle, zero fill.
ts_status make_map(CUtensorMap* map, const void* pool, int num_pages, int H_kv, int D, int hg) {
  auto fn = tensor_map_encoder();
  if (!fn) return fail(TS_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(num_pages) * kPS,
                        static_cast<cuuint64_t>(H_kv)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(H_kv) * D * 2, static_cast<cuuint64_t>(D) * 2};
  cuuint32_t box[3] = {64, kPS, static_cast<cuuint32_t>(hg)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult res = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(pool), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (res != CUDA_SUCCESS) return fail(TS_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(res));
  return TS_OK;
}

template <int kHD, int kHG>
ts_status launch(const MqParams& prm, const CUtensorMap& kmap, const CUtensorMap& vmap, int B, cudaStream_t s) {
  using Lay = Layout<kHD>;
  ts_status st = prepare_once(reinterpret_cast<const void*>(mq_tc_kernel<kHD, kHG>), [](const void* k) {
    ts_status s2 = cuda_check(cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, Layout<kHD>::kSmem),
                              "multi-query tensor-core smem attribute");
    if (s2 != TS_OK) return s2;
    return cuda_check(cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout,
                                           static_cast<int>(cudaSharedmemCarveoutMaxShared)),
                      "multi-query tensor-core carveout attribute");
  });
  if (st != TS_OK) return st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(B) * static_cast<unsigned>(prm.H_kv / kHG));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Lay::kSmem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  LaunchTrace trace("mq_tc_kernel", s);
  return cuda_check(cudaLaunchKernelEx(&cfg, mq_tc_kernel<kHD, kHG>, prm, kmap, vmap),
                    "multi-query tensor-core launch");
}

}  // namespace

// Runs the tensor-core path when it applies (bf16, page 16, D 64 or 128,
// q_len * g <= 128, 16-byte aligned rows); TS_ERR_UNSUPPORTED otherwise, with
// nothing enqueued, so that the caller takes the CUDA-core path.
ts_status launch_multi_query_tc(const void* q, const void* k_pool, const void* v_pool, const int32_t* block_table,
                                int32_t bt_stride, const int32_t* seq_lens, int32_t B, int32_t q_len, int32_t H_q,
                                int32_t H_kv, int32_t D, int32_t page_size, int32_t num_pages, float scale,
                                ts_dtype dtype, void* out, float* lse, uint32_t* err_word, cudaStream_t stream,
                                const int32_t* parents) {
  const int g = H_q / H_kv;
  if (dtype != TS_BF16 || page_size != kPS || (D != 64 && D != 128) || q_len < 1 || q_len * g > kBM ||
      static_cast<int64_t>(B) * H_kv > 0x7fffffff || (parents != nullptr && q_len > kMaxTree))
    return TS_ERR_UNSUPPORTED;
  MqParams prm;
  prm.q = static_cast<const __nv_bfloat16*>(q);
  prm.out = static_cast<__nv_bfloat16*>(out);
  prm.lse = lse;
  prm.block_table = block_table;
  prm.seq_lens = seq_lens;
  prm.parents = parents;
  prm.B = B;
  prm.bt_stride = bt_stride;
  prm.q_len = q_len;
  prm.H_q = H_q;
  prm.H_kv = H_kv;
  prm.g = g;
  prm.num_pages = num_pages;
  prm.scale_log2 = scale * kLog2eC;
  prm.err_word = err_word;
  // Heads per CTA: more heads make fewer, larger TMA boxes, fewer heads more
  // CTAs. Take the most that the rows allow (hg * R <= 128 with R padded to a
  // warp's 32 lanes) while the grid still covers 1.5 waves of SMs, else one.
  // TS_MULTI_QUERY_HEAD_GROUP=1/2/4 forces a value the shape allows (tests).
  const int R = q_len * g;
  const int hg_max = R <= 32 ? 4 : (R <= 64 ? 2 : 1);
  int hg = 1;
  for (int c = hg_max; c > 1; c >>= 1)
    if (H_kv % c == 0 && static_cast<int64_t>(B) * (H_kv / c) * 2 >= 3 * static_cast<int64_t>(device_sm_count())) {
      hg = c;
      break;
    }
  if (const char* e = getenv("TS_MULTI_QUERY_HEAD_GROUP")) {
    const int f = atoi(e);
    if ((f == 1 || f == 2 || f == 4) && f <= hg_max && H_kv % f == 0) hg = f;
  }
  CUtensorMap kmap, vmap;
  ts_status st = make_map(&kmap, k_pool, num_pages, H_kv, D, hg);
  if (st != TS_OK) return st;
  st = make_map(&vmap, v_pool, num_pages, H_kv, D, hg);
  if (st != TS_OK) return st;
  if (D == 64)
    return hg == 4 ? launch<64, 4>(prm, kmap, vmap, B, stream)
                   : hg == 2 ? launch<64, 2>(prm, kmap, vmap, B, stream) : launch<64, 1>(prm, kmap, vmap, B, stream);
  return hg == 4 ? launch<128, 4>(prm, kmap, vmap, B, stream)
                 : hg == 2 ? launch<128, 2>(prm, kmap, vmap, B, stream) : launch<128, 1>(prm, kmap, vmap, B, stream);
}

}  // namespace ts
