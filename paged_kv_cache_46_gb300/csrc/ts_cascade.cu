// ts_cascade_decode_attn: decode attention with shared prefixes computed once.
//
// Tokasaurus blog, "Dynamic prefix identification and exploration": shared
// prefixes (Hydragen / cascade attention) let the attention over a prefix run
// once for all sequences that share it. For a group, the queries of all
// members against the group's prefix keys form a real dense product: here a
// tcgen05 kernel computes it with 128 query rows (members x the g query heads
// of one kv head) per CTA against 128-key tiles of the prefix.
//
//   cascade_plan_kernel    tile offsets per group (device-side, from the CSR)
//   cascade_prefix_kernel  per (group tile, kv head): S = Q K^T and O += P V on
//                          the tensor cores, online softmax in between; writes
//                          the fp32 prefix state (O, LSE) of every member row
//   paged kernel (prefix mode) + split merge (ts_paged_decode.cu): each
//                          sequence's own pages after the prefix, merged with
//                          the prefix state by LSE into the final output.
//
// Prefix kernel roles (192 threads): warps 0-3 own one query row per thread
// (Q load, softmax, epilogue), warp 4 issues the TMA loads of K and V page
// boxes (128-byte swizzle; its lanes hold the page ids of the next key tile),
// warp 5 lane 0 issues the MMAs, S(j+1) or P V(j), whichever is ready first.
// TMEM holds S (128 fp32 columns), O (64 columns) and P (64 columns of bf16
// pairs, the P V product's A operand). K and V tiles are double-buffered, so
// a tile's load latency hides behind the previous tile's softmax and
// products. Two CTAs share an SM.
#include <cmath>
#include <mutex>

#include "ts_tcgen05.cuh"

namespace ts {
namespace {

constexpr int kHD = 64;            // head dim of the tensor-core prefix path
constexpr int kBM = 128;           // query rows per tile
constexpr int kBN = 128;           // keys per tile
constexpr int kPS = 16;            // page size of the prefix path
constexpr int kPagesPerTile = kBN / kPS;
constexpr int kThreadsPfx = 192;
constexpr uint32_t kTmemCols = 256;  // S: [0, 128), O: [128, 192), P: [192, 256)
constexpr uint32_t kTmemO = 128;
constexpr uint32_t kTmemP = 192;     // P as bf16 pairs: key k of row r at column k / 2 of lane r
constexpr float kLog2eC = 1.4426950408889634f;
constexpr float kLn2C = 0.6931471805599453f;
constexpr float kSlack = 8.0f;

// Shared memory (offsets from a 1024-aligned base).
constexpr int kOffQ = 0;          // [128 x 64] bf16, SW128 K-major              16 KB
constexpr int kTileKV = 16384;    // one K or V tile: [128 keys x 64] bf16, SW128
constexpr int kOffK = 16384;      // K tiles, 2 buffers                           32 KB
constexpr int kOffV = 49152;      // V tiles, 2 buffers                           32 KB
constexpr int kOffBar = 81920;    // mbarriers
constexpr int kOffTmem = kOffBar + 128;
constexpr int kSmemPfx = kOffTmem + 16;
// Two CTAs share an SM: their shared memory plus the 1 KB each reserves fits.
static_assert(2 * (kSmemPfx + 1024) <= 233472, "two prefix CTAs per SM");

struct PrefixParams {
  const __nv_bfloat16* q;  // [B, H_q, 64]
  const int32_t* prefix_indptr;
  const int32_t* prefix_pages;
  const int32_t* prefix_len;
  const int32_t* member_indptr;
  const int32_t* member_ids;
  const int32_t* tile_offset;  // [G + 1]
  int32_t num_groups, H_q, H_kv, g, mpt, num_pages;
  float scale_log2;
  float* prefix_o;    // [B, H_q, 64]
  float* prefix_lse;  // [B, H_q]
  uint32_t* err_word;
  // nested prefixes: merge this launch's state into the member's state from
  // the launches of the levels above instead of overwriting it
  int32_t accumulate;
};

// --- kernels -----------------------------------------------------------------

// tile_offset[g + 1] = sum over groups <= g of ceil(members / mpt). One CTA.
__global__ void __launch_bounds__(1024) cascade_plan_kernel(const int32_t* member_indptr, int G,
                                                            int mpt, int32_t* tile_offset) {
  __shared__ int warp_sum[32];
  __shared__ int carry;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    carry = 0;
    tile_offset[0] = 0;
  }
  __syncthreads();
  for (int base = 0; base < G; base += blockDim.x) {
    const int i = base + tid;
    const int c = i < G ? (member_indptr[i + 1] - member_indptr[i] + mpt - 1) / mpt : 0;
    int x = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_sum[warp] = x;
    __syncthreads();
    int before = 0, total = 0;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) {
      if (w < warp) before += warp_sum[w];
      total += warp_sum[w];
    }
    if (i < G) tile_offset[i + 1] = carry + before + x;
    __syncthreads();
    if (tid == 0) carry += total;
    __syncthreads();
  }
}

__global__ void __launch_bounds__(kThreadsPfx, 2) cascade_prefix_kernel(
    const PrefixParams p, const __grid_constant__ CUtensorMap kmap,
    const __grid_constant__ CUtensorMap vmap) {
  // no room to realign two CTAs' worth: the swizzled tiles need a 1024-byte
  // aligned base, which the declaration asks for and the check confirms
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = smem_raw;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t = blockIdx.x, h = blockIdx.y;
  if ((smem_u32(smem) & 1023u) != 0) {
    if (tid == 0) set_device_error(p.err_word, TS_DEVERR_SMEM_ALIGN);
    return;
  }
  const int n_tiles_total = p.tile_offset[p.num_groups];
  if (t >= n_tiles_total) return;
  // group of this tile: largest gi with tile_offset[gi] <= t
  int lo = 0, hi = p.num_groups - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.tile_offset[mid] <= t) lo = mid; else hi = mid - 1;
  }
  const int gi = lo;
  const int mbeg = p.member_indptr[gi] + (t - p.tile_offset[gi]) * p.mpt;
  const int mcount = min(p.mpt, p.member_indptr[gi + 1] - mbeg);
  const int pp0 = p.prefix_indptr[gi];
  const int n_pages = p.prefix_indptr[gi + 1] - pp0;
  const int plen = n_pages * kPS;  // this node's own pages (the path above it is other launches')
  const int n_kt = (n_pages + kPagesPerTile - 1) / kPagesPerTile;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  // K and V tiles are double-buffered: tile j lives in buffer j % 2 and is
  // the (j / 2)-th phase of that buffer's full / empty barrier
  auto b_kfull = [&](int buf) { return smem_u32(&bars[0 + buf]); };
  auto b_vfull = [&](int buf) { return smem_u32(&bars[2 + buf]); };
  auto b_kempty = [&](int buf) { return smem_u32(&bars[4 + buf]); };
  auto b_vempty = [&](int buf) { return smem_u32(&bars[6 + buf]); };
  const uint32_t b_sfull = smem_u32(&bars[8]), b_sfree = smem_u32(&bars[9]);
  const uint32_t b_pfull = smem_u32(&bars[10]), b_pvdone = smem_u32(&bars[11]);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffTmem);
  const uint32_t sQ = smem_u32(smem + kOffQ), sK = smem_u32(smem + kOffK);
  const uint32_t sV = smem_u32(smem + kOffV);

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(b_kfull(i), 1);
      mbar_init(b_vfull(i), 1);
      mbar_init(b_kempty(i), 1);
      mbar_init(b_vempty(i), 1);
    }
    mbar_init(b_sfull, 1);
    mbar_init(b_sfree, 4);
    mbar_init(b_pfull, 4);
    mbar_init(b_pvdone, 1);
    fence_mbar_init();
  }
  // Q tile: row r = (member r / g, query head h*g + r % g); rows past the
  // tile's members are zero.
  if (warp < 4) {
    const int r = tid;
    const int mi = r / p.g;
    uint4 chunk[8];
    if (mi < mcount) {
      const int b = p.member_ids[mbeg + mi];
      const uint4* src = reinterpret_cast<const uint4*>(
          p.q + (static_cast<int64_t>(b) * p.H_q + h * p.g + r % p.g) * kHD);
#pragma unroll
      for (int c = 0; c < 8; ++c) chunk[c] = src[c];
    } else {
#pragma unroll
      for (int c = 0; c < 8; ++c) chunk[c] = make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int c = 0; c < 8; ++c)
      *reinterpret_cast<uint4*>(smem + kOffQ + sw128_off(r, c)) = chunk[c];
    fence_async_smem();
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool ok = true;

  if (warp == 4) {
    // ---------------- TMA producer (lane i < 8 holds and loads page i) ----
    const int oob = p.num_pages * kPS;  // a row coordinate past the pool: zero fill
    auto tile_rows = [&](int j) {       // this lane's page of key tile j, as a pool row
      const int pi = j * kPagesPerTile + lane;
      int row = oob;
      if (lane < kPagesPerTile && pi < n_pages) {
        const int page = p.prefix_pages[pp0 + pi];
        if (page >= 0 && page < p.num_pages)
          row = page * kPS;
        else
          set_device_error(p.err_word, TS_DEVERR_PAGE_RANGE);
      }
      return row;
    };
    // One box per lane: a single thread issuing a tile's boxes one after
    // another caps the tile rate (measured on the multi-query kernel).
    auto load_tile = [&](const CUtensorMap* map, uint32_t dst, uint32_t bar, int rows) {
      if (lane == 0) mbar_arrive_expect_tx(bar, kBN * kHD * 2);
      __syncwarp();
      if (lane < kPagesPerTile) tma_load_3d(dst + lane * (kPS * 128), map, 0, h, rows, bar);
    };
    int rows = n_kt > 0 ? tile_rows(0) : oob;
    for (int j = 0; j < n_kt && ok; ++j) {
      const int rows_next = j + 1 < n_kt ? tile_rows(j + 1) : oob;  // page ids one tile ahead
      const int buf = j & 1, ph = ((j >> 1) - 1) & 1;  // buffer; phase of its previous use
      ok = __shfl_sync(0xffffffffu, lane == 0 && j >= 2 ? mbar_wait(b_kempty(buf), ph) : true, 0);
      if (!ok) break;
      load_tile(&kmap, sK + buf * kTileKV, b_kfull(buf), rows);
      ok = __shfl_sync(0xffffffffu, lane == 0 && j >= 2 ? mbar_wait(b_vempty(buf), ph) : true, 0);
      if (!ok) break;
      load_tile(&vmap, sV + buf * kTileKV, b_vfull(buf), rows);
      rows = rows_next;
    }
    if (!ok && lane == 0) set_device_error(p.err_word, TS_DEVERR_TIMEOUT);
  } else if (warp == 5) {
    // ---------------- MMA issuer ----------------
    // Whichever is ready first: S(js) (the softmax has read S(js-1), K(js)
    // landed) or P V(j) (P(j) written, V(j) landed). A late K tile then no
    // longer holds back P V, nor a late P the next S.
    if (lane == 0) {
      constexpr uint32_t iS = idesc_bf16(kBM, kBN, 0);
      constexpr uint32_t iO = idesc_bf16(kBM, kHD, 1);
      auto issue_s = [&](int js) {
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < kHD / 16; ++ks)
          mma_bf16(tmem, desc_sw128(sQ + ks * 32), desc_sw128(sK + (js & 1) * kTileKV + ks * 32), iS, ks > 0);
        mma_commit(b_sfull);
        mma_commit(b_kempty(js & 1));
      };
      int js = 0;
      if (n_kt > 0) {
        ok = mbar_wait(b_kfull(0), 0);
        if (ok) issue_s(js++);
      }
      for (int j = 0; j < n_kt && ok; ++j) {
        const int buf = j & 1;
        const unsigned long long t0 = globaltimer_ns();
        while (true) {
          if (js < n_kt && mbar_test(b_sfree, (js - 1) & 1) && mbar_test(b_kfull(js & 1), (js >> 1) & 1))
            issue_s(js++);
          if (mbar_test(b_pfull, j & 1) && mbar_test(b_vfull(buf), (j >> 1) & 1)) break;
          if (globaltimer_ns() - t0 > kWaitLimitNs) {
            ok = false;
            break;
          }
        }
        if (!ok) break;
        tc_fence_after();
        const uint32_t sVj = sV + buf * kTileKV;
#pragma unroll
        for (int ks = 0; ks < kBN / 16; ++ks)
          mma_bf16_tmem_a(tmem + kTmemO, tmem + kTmemP + ks * 8,
                   desc_sw128(sVj + ks * 2048), iO, (j > 0 || ks > 0) ? 1u : 0u);
        mma_commit(b_pvdone);
        mma_commit(b_vempty(buf));
      }
      if (!ok) set_device_error(p.err_word, TS_DEVERR_TIMEOUT);
    }
  } else {
    // ---------------- softmax warps: thread = query row ----------------
    const int r = tid;
    const uint32_t trow = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    float m = -INFINITY, l = 0.f;
    for (int j = 0; j < n_kt && ok; ++j) {
      ok = mbar_wait(b_sfull, j & 1);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      float s[kBN];
#pragma unroll
      for (int c0 = 0; c0 < kBN; c0 += 16) {
        uint32_t u[16];
        tmem_ld16(trow + c0, u);
        tmem_wait_ld();
#pragma unroll
        for (int x = 0; x < 16; ++x) s[c0 + x] = __uint_as_float(u[x]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_sfree);
      const int key0 = j * kBN;
      // With a positive scale (the usual case) the scores stay unscaled: the
      // row max is taken on raw scores (three-input max) and the scale is
      // folded into the exponent's FFMA. Keys past the prefix are masked only
      // in its last, partial tile.
      const float sl = p.scale_log2;
      float mx;
      if (sl > 0.f) {
        if (key0 + kBN > plen) {
#pragma unroll
          for (int c = 0; c < kBN; ++c) s[c] = key0 + c < plen ? s[c] : -INFINITY;
        }
        float mr = fmax3(s[0], s[1], s[2]);
#pragma unroll
        for (int c = 3; c + 1 < kBN; c += 2) mr = fmax3(mr, s[c], s[c + 1]);
        mr = fmaxf(mr, s[kBN - 1]);
        mx = mr * sl;
      } else {
        mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < kBN; ++c) {
          s[c] = key0 + c < plen ? s[c] * sl : -INFINITY;
          mx = fmaxf(mx, s[c]);
        }
      }
      const float sx = sl > 0.f ? sl : 1.f;  // factor still to apply to s[] in the exponent
      // the previous P V must be done before P and O are touched
      if (j > 0) {
        ok = mbar_wait(b_pvdone, (j - 1) & 1);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
      }
      const bool need = mx > m + kSlack;
      if (j == 0) {
        m = mx;
      } else if (__any_sync(0xffffffffu, need)) {
        const float mnew = fmaxf(m, mx);
        const float alpha = m == -INFINITY ? 0.f : fast_exp2(m - mnew);
        m = mnew;
        l *= alpha;
#pragma unroll
        for (int c0 = 0; c0 < kHD; c0 += 16) {
          uint32_t u[16];
          tmem_ld16(trow + kTmemO + c0, u);
          tmem_wait_ld();
#pragma unroll
          for (int x = 0; x < 16; ++x) u[x] = __float_as_uint(__uint_as_float(u[x]) * alpha);
          tmem_st16(trow + kTmemO + c0, u);
        }
        tmem_wait_st();
      }
      const float ms = m == -INFINITY ? 0.f : m;
      float2 ls2 = make_float2(0.f, 0.f);
      // P straight into TMEM (the P V MMA reads its A operand there)
#pragma unroll
      for (int c = 0; c < kBN; c += 32) {
        uint32_t pk[16];
#pragma unroll
        for (int x = 0; x < 32; x += 2) {
          const float e0 = fast_exp2(fmaf(s[c + x], sx, -ms));
          const float e1 = fast_exp2(fmaf(s[c + x + 1], sx, -ms));
          ls2 = __fadd2_rn(ls2, make_float2(e0, e1));
          pk[x / 2] = float2_to_bf16x2(e0, e1);
        }
        tmem_st16(trow + kTmemP + c / 2, pk);
      }
      tmem_wait_st();
      l += ls2.x + ls2.y;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_pfull);
    }
    // epilogue: O row / l, LSE (an empty prefix gives O = 0, LSE = -inf)
    if (ok && n_kt == 0 && !p.accumulate) {
      const int mi = r / p.g;
      if (mi < mcount) {
        const int64_t row = static_cast<int64_t>(p.member_ids[mbeg + mi]) * p.H_q + h * p.g + r % p.g;
        for (int c = 0; c < kHD; ++c) p.prefix_o[row * kHD + c] = 0.f;
        p.prefix_lse[row] = -INFINITY;
      }
    }
    if (ok && n_kt > 0) {
      ok = mbar_wait(b_pvdone, (n_kt - 1) & 1);
      if (__all_sync(0xffffffffu, ok)) {
        tc_fence_after();
        const int mi = r / p.g;
        const bool valid = mi < mcount;
        const int b = valid ? p.member_ids[mbeg + mi] : 0;
        const int64_t row = static_cast<int64_t>(b) * p.H_q + h * p.g + r % p.g;
        float lse_new = l > 0.f ? (m + log2f(l)) * kLn2C : -INFINITY;
        // weights of the state already there (accumulate) and of this one,
        // by LSE (TokenSpeed deep dive, section 7.1)
        float w_old = 0.f, w_new = l > 0.f ? 1.0f / l : 0.f;
        if (p.accumulate && valid) {
          const float lse_old = p.prefix_lse[row];
          const float mx = fmaxf(lse_old, lse_new);
          const float ea = lse_old == -INFINITY ? 0.f : __expf(lse_old - mx);
          const float eb = lse_new == -INFINITY ? 0.f : __expf(lse_new - mx);
          const float den = ea + eb;
          const float iden = den > 0.f ? 1.0f / den : 0.f;
          w_old = ea * iden;
          w_new *= eb * iden;
          lse_new = den > 0.f ? mx + logf(den) : -INFINITY;
        }
#pragma unroll
        for (int c0 = 0; c0 < kHD; c0 += 16) {
          uint32_t u[16];
          tmem_ld16(trow + kTmemO + c0, u);
          tmem_wait_ld();
          if (valid) {
            float4* dst = reinterpret_cast<float4*>(p.prefix_o + row * kHD + c0);
#pragma unroll
            for (int x = 0; x < 16; x += 4) {
              float4 o = make_float4(__uint_as_float(u[x]) * w_new, __uint_as_float(u[x + 1]) * w_new,
                                     __uint_as_float(u[x + 2]) * w_new, __uint_as_float(u[x + 3]) * w_new);
              if (p.accumulate) {
                const float4 prev = dst[x / 4];
                o = make_float4(o.x + w_old * prev.x, o.y + w_old * prev.y, o.z + w_old * prev.z,
                                o.w + w_old * prev.w);
              }
              dst[x / 4] = o;
            }
          }
        }
        if (valid) p.prefix_lse[row] = lse_new;
      } else {
        ok = false;
      }
    }
    if (!ok) set_device_error(p.err_word, TS_DEVERR_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
  }
}

// --- host ------------------------------------------------------------------

// 3-D map over a pool [P * page_size rows][H_kv][64] bf16 with a box of one
// page of one kv head (16 rows x 128 B), 128-byte swizzle, zero fill.
ts_status make_page_map(CUtensorMap* map, const void* pool, int num_pages, int H_kv) {
  auto fn = tensor_map_encoder();
  if (!fn) return fail(TS_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(kHD), static_cast<cuuint64_t>(H_kv),
                        static_cast<cuuint64_t>(num_pages) * kPS};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(kHD) * 2, static_cast<cuuint64_t>(H_kv) * kHD * 2};
  cuuint32_t box[3] = {kHD, 1, kPS};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(pool), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(TS_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
  return TS_OK;
}

struct CascadeWs {
  size_t paged, tile_offset, prefix_o, prefix_lse, total;
};

CascadeWs cascade_layout(int B, int H_q, int D) {
  CascadeWs w;
  w.paged = 0;
  size_t off = align_up(paged_decode_workspace_bytes(B, H_q, D), kWorkspaceAlign);
  w.tile_offset = off;
  off = align_up(off + (static_cast<size_t>(B) + 2) * sizeof(int32_t), kWorkspaceAlign);
  w.prefix_o = off;
  off = align_up(off + static_cast<size_t>(B) * H_q * D * sizeof(float), kWorkspaceAlign);
  w.prefix_lse = off;
  off = align_up(off + static_cast<size_t>(B) * H_q * sizeof(float), kWorkspaceAlign);
  w.total = off;
  return w;
}

// One launch pair (plan + prefix kernel) over groups 0..G-1 of the given CSR
// arrays: every member row's fp32 state over its group's own pages, written
// to prefix_o / prefix_lse, or merged into what is there (accumulate).
ts_status prefix_pass(const void* q, const void* k_pool, const void* v_pool, const int32_t* prefix_indptr,
                      const int32_t* prefix_pages, const int32_t* prefix_len, const int32_t* member_indptr,
                      const int32_t* member_ids, int G, int B, int H_q, int H_kv, int num_pages, float scale,
                      float* prefix_o, float* prefix_lse, int32_t* tile_offset, uint32_t* err_word,
                      bool accumulate, cudaStream_t s) {
  const int g = H_q / H_kv;
  const int mpt = kBM / g;
  ts_status st;
  {
    LaunchTrace trace("cascade_plan_kernel", s);
    cascade_plan_kernel<<<1, 1024, 0, s>>>(member_indptr, G, mpt, tile_offset);
    st = cuda_check(cudaGetLastError(), "cascade plan launch");
  }
  if (st != TS_OK) return st;
  CUtensorMap kmap, vmap;
  st = make_page_map(&kmap, k_pool, num_pages, H_kv);
  if (st != TS_OK) return st;
  st = make_page_map(&vmap, v_pool, num_pages, H_kv);
  if (st != TS_OK) return st;
  PrefixParams pp;
  pp.q = static_cast<const __nv_bfloat16*>(q);
  pp.prefix_indptr = prefix_indptr;
  pp.prefix_pages = prefix_pages;
  pp.prefix_len = prefix_len;
  pp.member_indptr = member_indptr;
  pp.member_ids = member_ids;
  pp.tile_offset = tile_offset;
  pp.num_groups = G;
  pp.H_q = H_q;
  pp.H_kv = H_kv;
  pp.g = g;
  pp.mpt = mpt;
  pp.num_pages = num_pages;
  pp.scale_log2 = scale * kLog2eC;
  pp.prefix_o = prefix_o;
  pp.prefix_lse = prefix_lse;
  pp.err_word = err_word;
  pp.accumulate = accumulate ? 1 : 0;
  st = prepare_once(reinterpret_cast<const void*>(cascade_prefix_kernel), [](const void* k) {
    ts_status s2 = cuda_check(cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemPfx),
                              "prefix smem attribute");
    if (s2 != TS_OK) return s2;
    // all of the SM's unified L1/shared memory as shared memory: two CTAs per SM
    return cuda_check(cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout,
                                           static_cast<int>(cudaSharedmemCarveoutMaxShared)),
                      "prefix carveout attribute");
  });
  if (st != TS_OK) return st;
  // upper bound on tiles: sum ceil(n_g / mpt) <= B / mpt + G; extra CTAs exit at once
  const unsigned tiles = static_cast<unsigned>(B / mpt + G + 1);
  LaunchTrace trace("cascade_prefix_kernel", s);
  cascade_prefix_kernel<<<dim3(tiles, H_kv), kThreadsPfx, kSmemPfx, s>>>(pp, kmap, vmap);
  return cuda_check(cudaGetLastError(), "cascade prefix launch");
}

}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

}  // namespace ts

extern "C" size_t ts_cascade_decode_workspace_size(int32_t B, int32_t H_q, int32_t D) {
  if (B < 0 || H_q <= 0 || D <= 0 || ts::paged_decode_workspace_bytes(B, H_q, D) == 0) return 0;
  return ts::cascade_layout(B, H_q, D).total;
}

extern "C" ts_status ts_cascade_decode_attn(const void* q, const void* k_pool, const void* v_pool,
                                            const ts_prefix_groups* groups,
                                            const int32_t* block_table, int32_t bt_stride,
                                            const int32_t* seq_lens, int32_t B, int32_t H_q,
                                            int32_t H_kv, int32_t D, int32_t page_size,
                                            int32_t num_pages, float scale, ts_dtype dtype,
                                            void* out, float* lse, void* workspace,
                                            size_t workspace_bytes, void* stream) {
  using namespace ts;
  const char* who = "ts_cascade_decode_attn";
  if (!groups) return fail(TS_ERR_INVALID_ARG, "%s: null groups", who);
  if (B == 0) return TS_OK;
  if (B < 0 || H_q <= 0 || H_kv <= 0 || H_q % H_kv != 0 || num_pages <= 0 ||
      static_cast<long long>(num_pages) * page_size > INT32_MAX)
    return fail(TS_ERR_INVALID_ARG, "%s: bad sizes (B=%d H_q=%d H_kv=%d P=%d)", who, B, H_q, H_kv, num_pages);
  const int g = H_q / H_kv;
  if (dtype != TS_BF16 || D != kHD || page_size != kPS || (g != 1 && g != 2 && g != 4 && g != 8))
    return fail(TS_ERR_UNSUPPORTED, "%s: needs bf16, D=64, page_size=16, H_q/H_kv in {1,2,4,8}", who);
  const int G = groups->num_groups;
  if (G < 0 || G > B) return fail(TS_ERR_INVALID_ARG, "%s: num_groups=%d", who, G);
  if (!groups->group_of || (G > 0 && (!groups->prefix_indptr || !groups->prefix_pages ||
                                      !groups->prefix_len || !groups->member_indptr ||
                                      !groups->member_ids)))
    return fail(TS_ERR_INVALID_ARG, "%s: null group array", who);
  if (!q || !k_pool || !v_pool || !out || !block_table || !seq_lens)
    return fail(TS_ERR_INVALID_ARG, "%s: null pointer", who);
  for (const void* ptr : {q, k_pool, v_pool})
    if (reinterpret_cast<uintptr_t>(ptr) % 16 != 0)
      return fail(TS_ERR_INVALID_ARG, "%s: q and pools must be 16-byte aligned", who);
  const size_t need = ts_cascade_decode_workspace_size(B, H_q, D);
  if (need == 0) return fail(TS_ERR_CUDA, "%s: cannot size the workspace", who);
  if (!workspace || workspace_bytes < need)
    return fail(TS_ERR_WORKSPACE, "%s: workspace %zu B < %zu B needed", who, workspace_bytes, need);
  if (reinterpret_cast<uintptr_t>(workspace) % kWorkspaceAlign != 0)
    return fail(TS_ERR_WORKSPACE, "%s: workspace must be 256-byte aligned", who);
  const CascadeWs ws = cascade_layout(B, H_q, D);
  unsigned char* wsb = static_cast<unsigned char*>(workspace);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* prefix_o = reinterpret_cast<float*>(wsb + ws.prefix_o);
  float* prefix_lse = reinterpret_cast<float*>(wsb + ws.prefix_lse);

  if (G > 0) {
    const ts_status st = prefix_pass(q, k_pool, v_pool, groups->prefix_indptr, groups->prefix_pages,
                                     groups->prefix_len, groups->member_indptr, groups->member_ids, G, B, H_q,
                                     H_kv, num_pages, scale, prefix_o, prefix_lse,
                                     reinterpret_cast<int32_t*>(wsb + ws.tile_offset),
                                     reinterpret_cast<uint32_t*>(wsb), false, s);
    if (st != TS_OK) return st;
  }
  PrefixInputs pre;
  pre.group_of = groups->group_of;
  pre.prefix_len = groups->prefix_len;
  pre.prefix_o = prefix_o;
  pre.prefix_lse = prefix_lse;
  pre.num_groups = G;
  return launch_paged_decode_impl(q, k_pool, v_pool, block_table, bt_stride, seq_lens, B, H_q,
                                  H_kv, D, page_size, num_pages, scale, dtype, out, lse, workspace,
                                  ws.tile_offset, s, who, G > 0 ? &pre : nullptr);
}

extern "C" ts_status ts_cascade_nested_decode_attn(const void* q, const void* k_pool, const void* v_pool,
                                                   const ts_prefix_forest* forest,
                                                   const int32_t* level_indptr_host,
                                                   const int32_t* block_table, int32_t bt_stride,
                                                   const int32_t* seq_lens, int32_t B, int32_t H_q,
                                                   int32_t H_kv, int32_t D, int32_t page_size,
                                                   int32_t num_pages, float scale, ts_dtype dtype,
                                                   void* out, float* lse, void* workspace,
                                                   size_t workspace_bytes, void* stream) {
  using namespace ts;
  const char* who = "ts_cascade_nested_decode_attn";
  if (!forest) return fail(TS_ERR_INVALID_ARG, "%s: null forest", who);
  if (B == 0) return TS_OK;
  if (B < 0 || H_q <= 0 || H_kv <= 0 || H_q % H_kv != 0 || num_pages <= 0 ||
      static_cast<long long>(num_pages) * page_size > INT32_MAX)
    return fail(TS_ERR_INVALID_ARG, "%s: bad sizes (B=%d H_q=%d H_kv=%d P=%d)", who, B, H_q, H_kv, num_pages);
  const int g = H_q / H_kv;
  if (dtype != TS_BF16 || D != kHD || page_size != kPS || (g != 1 && g != 2 && g != 4 && g != 8))
    return fail(TS_ERR_UNSUPPORTED, "%s: needs bf16, D=64, page_size=16, H_q/H_kv in {1,2,4,8}", who);
  const int N = forest->num_nodes, L = forest->num_levels;
  if (N < 0 || L < 0 || (N > 0) != (L > 0)) return fail(TS_ERR_INVALID_ARG, "%s: %d nodes, %d levels", who, N, L);
  if (N > 0) {
    if (!level_indptr_host) return fail(TS_ERR_INVALID_ARG, "%s: null host level_indptr", who);
    if (level_indptr_host[0] != 0 || level_indptr_host[L] != N)
      return fail(TS_ERR_INVALID_ARG, "%s: level_indptr must run from 0 to num_nodes", who);
    for (int l = 0; l < L; ++l)
      if (level_indptr_host[l + 1] <= level_indptr_host[l])
        return fail(TS_ERR_INVALID_ARG, "%s: level %d holds no node", who, l);
  }
  if (!forest->group_of || (N > 0 && (!forest->prefix_indptr || !forest->prefix_pages || !forest->prefix_len ||
                                      !forest->member_indptr || !forest->member_ids)))
    return fail(TS_ERR_INVALID_ARG, "%s: null forest array", who);
  if (!q || !k_pool || !v_pool || !out || !block_table || !seq_lens)
    return fail(TS_ERR_INVALID_ARG, "%s: null pointer", who);
  for (const void* ptr : {q, k_pool, v_pool})
    if (reinterpret_cast<uintptr_t>(ptr) % 16 != 0)
      return fail(TS_ERR_INVALID_ARG, "%s: q and pools must be 16-byte aligned", who);
  const size_t need = ts_cascade_decode_workspace_size(B, H_q, D);
  if (need == 0) return fail(TS_ERR_CUDA, "%s: cannot size the workspace", who);
  if (!workspace || workspace_bytes < need)
    return fail(TS_ERR_WORKSPACE, "%s: workspace %zu B < %zu B needed", who, workspace_bytes, need);
  if (reinterpret_cast<uintptr_t>(workspace) % kWorkspaceAlign != 0)
    return fail(TS_ERR_WORKSPACE, "%s: workspace must be 256-byte aligned", who);
  const CascadeWs ws = cascade_layout(B, H_q, D);
  unsigned char* wsb = static_cast<unsigned char*>(workspace);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* prefix_o = reinterpret_cast<float*>(wsb + ws.prefix_o);
  float* prefix_lse = reinterpret_cast<float*>(wsb + ws.prefix_lse);
  // level by level: the roots write each member's prefix state, deeper levels
  // merge their stretch into it (a member is in one node per level, so no two
  // tiles of a launch touch the same row)
  for (int l = 0; l < L; ++l) {
    const int n0 = level_indptr_host[l], nl = level_indptr_host[l + 1] - n0;
    const ts_status st =
        prefix_pass(q, k_pool, v_pool, forest->prefix_indptr + n0, forest->prefix_pages, forest->prefix_len + n0,
                    forest->member_indptr + n0, forest->member_ids, nl, B, H_q, H_kv, num_pages, scale, prefix_o,
                    prefix_lse, reinterpret_cast<int32_t*>(wsb + ws.tile_offset),
                    reinterpret_cast<uint32_t*>(wsb), l > 0, s);
    if (st != TS_OK) return st;
  }
  PrefixInputs pre;
  pre.group_of = forest->group_of;   // deepest node
  pre.prefix_len = forest->prefix_len;  // tokens shared through it
  pre.prefix_o = prefix_o;
  pre.prefix_lse = prefix_lse;
  pre.num_groups = N;
  return launch_paged_decode_impl(q, k_pool, v_pool, block_table, bt_stride, seq_lens, B, H_q, H_kv, D, page_size,
                                  num_pages, scale, dtype, out, lse, workspace, ws.tile_offset, s, who,
                                  N > 0 ? &pre : nullptr);
}
