// Tensor-core path of ts_paged_decode_fp8_attn: decode over an fp8 (e4m3fn)
// KV cache whose rows carry one float32 scale per (page, row, kv head).
//
// tokenspeed 딥다이브 (fiv.co.kr), section 6-4: a cached row is its codes
// times its token group's scale. On the CUDA cores the g query heads of a kv
// head cost the same FMAs per element whatever its width, so an fp8 cache is
// no faster there; here the products run on tcgen05:
//
// - A CTA takes HG (2 or 4) kv heads of one sequence. A key tile is 128 pool
//   rows: 8 / HG pages of the HG heads. TMA brings each page's codes of the
//   HG heads in one box (landing [head][16 rows][D bytes]) and a bulk copy
//   each page's K and V scale rows, into a three-stage staging ring.
// - Four converter warps widen the codes to f16 (exactly, as their values
//   times 2^-8; the scales take the 2^8) into the 128-byte swizzled layout
//   the tensor cores read, zero the V rows past the sequence, and lay out
//   the tile's scales.
// - S = Q K^T and O += P V run as in the multi-query kernel (block-diagonal
//   over the HG heads), kind::f16. Q sits in TMEM as f16, each row scaled
//   by a power of two into f16 range (the score scale takes it back). A score
//   takes its key's K scale; a probability its key's V scale before it is
//   rounded to f16 for the product; the row sum does not.
//
// Roles (320 threads): warps 0-3 softmax (a query row per thread), warp 4 TMA
// producer (lane i < 8 / HG loads page i of a tile), warp 5 lane 0 MMA
// issuer, warps 6-9 converters (a tile row per thread).
#include <cuda_fp16.h>

#include <cmath>
#include <cstdlib>
#include <cstring>

#include "ts_tcgen05.cuh"

namespace ts {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

namespace {

constexpr int kBM = 128;  // query rows per tile
constexpr int kBN = 128;  // pool rows per key tile
constexpr int kPS = 16;   // page size of this path
constexpr int kPagesPerTile = kBN / kPS;
constexpr int kThreads = 320;
constexpr int kAtom = kBN * 128;   // one [128 rows x 64 f16] SW128 atom: 16 KB
constexpr int kScaleMax = 2048;    // bytes of a stage's K (or V) scale rows
constexpr int kStages = 3;         // staging ring
constexpr float kLog2eC = 1.4426950408889634f;
constexpr float kLn2C = 0.6931471805599453f;
constexpr float kSlack = 8.0f;
constexpr int kLongestFirstMaxB = 128;

template <int kHD>
struct Layout {
  static constexpr int kAtoms = kHD / 64;
  static constexpr int kCodeTile = kBN * kHD;                    // one K (or V) code tile, bytes
  static constexpr int kStage = 2 * kCodeTile + 2 * kScaleMax;   // codes K, V; scale rows K, V
  static constexpr int kConv = kAtoms * kAtom;                   // one widened K (or V) tile
  static constexpr int kOffStage = 0;                            // kStages staging stages
  static constexpr int kOffConv = kOffStage + kStages * kStage;  // widened K x 2, then V x 1
  static constexpr int kOffScl = kOffConv + 3 * kConv;           // K scales [2][128], V scales [128]
  static constexpr int kOffBar = kOffScl + 3 * kBM * 4;
  static constexpr int kOffTmem = kOffBar + 256;
  static constexpr int kSmem = kOffTmem + 16;
  static constexpr uint32_t kTmemO = 128;
  static constexpr uint32_t kTmemP = 128 + kHD;  // two 64-column P buffers
  static constexpr uint32_t kTmemQ = 256 + kHD;  // Q: kHD / 2 columns of f16 pairs
  static constexpr uint32_t kTmemCols = 512;
  static_assert(kOffConv % 1024 == 0 && kConv % 1024 == 0, "swizzled tiles 1024-byte aligned");
  static_assert(kTmemQ + kHD / 2 <= kTmemCols, "TMEM budget");
  static_assert(kSmem <= 227 * 1024, "shared memory budget");
};

struct Fp8Params {
  const __nv_bfloat16* q;      // [B, H_q, D]
  __nv_bfloat16* out;          // [B, H_q, D]
  float* lse;                  // [B, H_q] or nullptr
  const int32_t* block_table;  // [B, bt_stride]
  const int32_t* seq_lens;     // [B]
  const float* k_scale;        // [num_pages, 16, H_kv]
  const float* v_scale;
  int32_t B, bt_stride, H_q, H_kv, g, num_pages;
  float scale_log2;
  uint32_t* err_word;
};

// Instruction descriptor of kind::f16 with f16 A and B, fp32 accumulate.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, int b_mn_major) {
  return (1u << 4) | (static_cast<uint32_t>(b_mn_major) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// Two e4m3fn codes (bytes 0 and 1 of `two_codes`, after the byte spread
// below) as an f16x2 word holding their values times 2^-8, exactly. e4m3fn
// is sign | 4-bit exponent (bias 7) | 3-bit mantissa; placed as
// sign | 0 | exponent | mantissa << 7 in an f16 (bias 15), a normal code's
// exponent field reads 8 less and a subnormal code (exponent 0, value
// m * 2^-9) becomes the f16 subnormal m * 2^-17: both the value times 2^-8.
// Plain integer operations, so the widening runs at full ALU rate.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2_scaled(uint32_t spread) {
  // spread: code 0 in bits 0-7, code 1 in bits 16-23
  return ((spread & 0x00800080u) << 8) | ((spread & 0x007F007Fu) << 7);
}

// The factor 2^8 the widened codes lack.
constexpr float kWidenScale = 256.0f;

__device__ __forceinline__ uint32_t f16x2_bits(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  uint32_t u;
  memcpy(&u, &h, 4);
  return u;
}

// Widens one tile row of kHD codes (at src) to f16 (values times 2^-8) into
// the 128-byte swizzled tile at dst (row t), or writes zeros. Each thread walks its 16-byte chunks
// in a rotated order so that a warp's shared loads hit distinct banks.
template <int kHD>
__device__ __forceinline__ void widen_row(const unsigned char* src, unsigned char* dst, int t, bool zero) {
  constexpr int kChunks = kHD / 16;  // 16 codes each
#pragma unroll
  for (int i = 0; i < kChunks; ++i) {
    const int cc = (i + t) % kChunks;
    const uint4 v = zero ? make_uint4(0u, 0u, 0u, 0u) : *reinterpret_cast<const uint4*>(src + cc * 16);
    const uint32_t in[4] = {v.x, v.y, v.z, v.w};
    uint32_t w[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      w[2 * k] = e4m3x2_to_f16x2_scaled(__byte_perm(in[k], 0u, 0x4140));      // codes 0, 1
      w[2 * k + 1] = e4m3x2_to_f16x2_scaled(__byte_perm(in[k], 0u, 0x4342));  // codes 2, 3
    }
    const int e0 = cc * 16;                       // first element of the chunk
    const int a = e0 / 64, ch = (e0 % 64) / 8;    // atom, 16-byte chunk of the row in it
    *reinterpret_cast<uint4*>(dst + a * kAtom + sw128_off(t, ch)) = make_uint4(w[0], w[1], w[2], w[3]);
    *reinterpret_cast<uint4*>(dst + a * kAtom + sw128_off(t, ch + 1)) = make_uint4(w[4], w[5], w[6], w[7]);
  }
}

template <int kHD, int kHG>
__global__ void __launch_bounds__(kThreads, 1) fp8_tc_kernel(
    const Fp8Params p, const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap) {
  using Lay = Layout<kHD>;
  constexpr int HG = kHG, TP = kPagesPerTile / HG, Rw = kBM / HG, kKeys = TP * kPS;
  extern __shared__ __align__(1024) unsigned char smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Programmatic dependent launch: outputs are written only after the wait.
  pdl_launch_dependents();
  if ((smem_u32(smem) & 1023u) != 0) {
    if (tid == 0) set_device_error(p.err_word, TS_DEVERR_SMEM_ALIGN);
    return;
  }
  const int hgroups = p.H_kv / HG;
  const int h0 = static_cast<int>(blockIdx.x % hgroups) * HG;  // first kv head
  int b = static_cast<int>(blockIdx.x / hgroups);
  if (p.B <= kLongestFirstMaxB) {
    // sequences by decreasing page count (ties by index): longest first
    auto pages = [&](int s) {
      const int len = p.seq_lens[s];
      return len > 0 ? min((len + kPS - 1) / kPS, p.bt_stride) : 0;
    };
    int* pick = reinterpret_cast<int*>(smem + Lay::kOffTmem + 8);
    for (int s = tid; s < p.B; s += kThreads) {
      const int ws = pages(s);
      int rank = 0;
      for (int t = 0; t < p.B; ++t) {
        const int wt = pages(t);
        rank += (wt > ws || (wt == ws && t < s)) ? 1 : 0;
      }
      if (rank == b) *pick = s;
    }
    __syncthreads();
    b = *pick;
  }
  const int R = p.g;  // query rows of a kv head (one query token per sequence)
  const int L = p.seq_lens[b];
  const int n_pages = L > 0 ? min((L + kPS - 1) / kPS, p.bt_stride) : 0;
  const int n_kt = (n_pages + TP - 1) / TP;
  // Before this wait only the lengths are read.
  pdl_wait_primary();

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::kOffBar);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  // staging stage s: full (TMA bytes) / empty (converters done with it);
  // widened K buffer c: full (converters) / empty (S read it); the single
  // widened V buffer: full / empty (P V read it)
  auto stg_full = [&](int s) { return bar(0 + s); };
  auto stg_empty = [&](int s) { return bar(3 + s); };
  auto conv_kfull = [&](int c) { return bar(6 + c); };
  auto conv_kempty = [&](int c) { return bar(8 + c); };
  const uint32_t conv_vfull = bar(10), conv_vempty = bar(11);
  const uint32_t b_sfull = bar(12), b_sfree = bar(13);
  auto b_pfull = [&](int pb) { return bar(14 + pb); };
  auto b_pvdone = [&](int pb) { return bar(16 + pb); };
  const uint32_t b_qready = bar(18);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Lay::kOffTmem);
  const uint32_t sStage = smem_u32(smem + Lay::kOffStage), sConv = smem_u32(smem + Lay::kOffConv);

  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(stg_full(i), 1);
      mbar_init(stg_empty(i), 4);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(conv_kfull(i), 4);
      mbar_init(conv_kempty(i), 1);
      mbar_init(b_pfull(i), 4);
      mbar_init(b_pvdone(i), 1);
    }
    mbar_init(conv_vfull, 4);
    mbar_init(conv_vempty, 1);
    mbar_init(b_sfull, 1);
    mbar_init(b_sfree, 4);
    mbar_init(b_qready, 4);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(smem_u32(tmem_slot), Lay::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool ok = true;

  if (warp == 4) {
    // ---------------- TMA producer ----------------
    const int oob = p.num_pages * kPS;  // a row coordinate past the pool: zero fill
    const uint32_t sclb = static_cast<uint32_t>(kPS * p.H_kv * 4);  // one page's scale rows
    auto tile_page = [&](int j) {       // this lane's page of key tile j (-1: none or bad)
      const int pi = j * TP + lane;
      int page = -1;
      if (lane < TP && pi < n_pages) {
        page = p.block_table[static_cast<int64_t>(b) * p.bt_stride + pi];
        if (page < 0 || page >= p.num_pages) {
          set_device_error(p.err_word, TS_DEVERR_PAGE_RANGE);
          page = -1;
        }
      }
      return page;
    };
    const uint32_t stage_tx = 2u * Lay::kCodeTile + 2u * TP * sclb;
    int page = n_kt > 0 ? tile_page(0) : -1;
    for (int j = 0; j < n_kt && ok; ++j) {
      const int page_next = j + 1 < n_kt ? tile_page(j + 1) : -1;
      const int s = j % kStages;
      ok = __shfl_sync(0xffffffffu,
                       lane == 0 && j >= kStages ? mbar_wait(stg_empty(s), ((j / kStages) - 1) & 1) : true, 0);
      if (!ok) break;
      const uint32_t st = sStage + s * Lay::kStage;
      if (lane == 0) mbar_arrive_expect_tx(stg_full(s), stage_tx);
      __syncwarp();
      if (lane < TP) {
        const int row = page >= 0 ? page * kPS : oob;
        tma_load_3d(st + lane * (HG * kPS * kHD), &kmap, 0, row, h0, stg_full(s));
        tma_load_3d(st + Lay::kCodeTile + lane * (HG * kPS * kHD), &vmap, 0, row, h0, stg_full(s));
        // a page that is absent or bad: page 0's scale rows (its keys are masked)
        const size_t so = static_cast<size_t>(page >= 0 ? page : 0) * kPS * p.H_kv;
        bulk_g2s(st + 2 * Lay::kCodeTile + lane * sclb, p.k_scale + so, sclb, stg_full(s));
        bulk_g2s(st + 2 * Lay::kCodeTile + kScaleMax + lane * sclb, p.v_scale + so, sclb, stg_full(s));
      }
      page = page_next;
    }
    if (!ok && lane == 0) set_device_error(p.err_word, TS_DEVERR_TIMEOUT);
  } else if (warp >= 6) {
    // ---------------- converters: thread = tile row ----------------
    const int ct = tid - 6 * 32;
    const int pb = ct / (HG * kPS), hs = (ct / kPS) % HG, key = ct % kPS;
    float* scl_base = reinterpret_cast<float*>(smem + Lay::kOffScl);
    auto sync_ok = [&]() {
      if (!__all_sync(0xffffffffu, ok)) ok = false;
      return ok;
    };
    for (int j = 0; j < n_kt && ok; ++j) {
      const int s = j % kStages, cb = j & 1;
      ok = mbar_wait(stg_full(s), (j / kStages) & 1);
      // K: the buffer was last read by S(j-2), its scales by the softmax of
      // tile j-2 (done once that tile's P is written)
      if (ok && j >= 2) ok = mbar_wait(conv_kempty(cb), ((j >> 1) - 1) & 1);
      if (ok && j >= 2) ok = mbar_wait(b_pfull(cb), ((j >> 1) - 1) & 1);
      if (!sync_ok()) break;
      const unsigned char* stg = smem + Lay::kOffStage + s * Lay::kStage;
      unsigned char* conv = smem + Lay::kOffConv + cb * Lay::kConv;
      const int kpos = j * kKeys + pb * kPS + key;  // this row's token
      const int si = (pb * kPS + key) * p.H_kv + h0 + hs;
      float* scl = scl_base + cb * kBM;
      widen_row<kHD>(stg + ct * kHD, conv, ct, false);
      scl[ct] = reinterpret_cast<const float*>(stg + 2 * Lay::kCodeTile)[si] * kWidenScale;
      fence_async_smem();  // the widened tile is read by the tensor cores
      __syncwarp();
      if (lane == 0) mbar_arrive(conv_kfull(cb));
      // V: the buffer and its scales were last read by P V(j-1) and the
      // softmax of tile j-1
      if (j >= 1) ok = mbar_wait(conv_vempty, (j - 1) & 1);
      if (!sync_ok()) break;
      // V rows past the sequence may hold anything (NaN codes included) and
      // 0 * NaN is NaN in the product: they become zeros
      widen_row<kHD>(stg + Lay::kCodeTile + ct * kHD, smem + Lay::kOffConv + 2 * Lay::kConv, ct, kpos >= L);
      scl_base[2 * kBM + ct] =
          kpos < L ? reinterpret_cast<const float*>(stg + 2 * Lay::kCodeTile + kScaleMax)[si] * kWidenScale : 0.f;
      fence_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(conv_vfull);
        mbar_arrive(stg_empty(s));
      }
    }
    if (!ok) set_device_error(p.err_word, TS_DEVERR_TIMEOUT);
  } else if (warp == 5) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t iS = idesc_f16(kBM, kBN, 0);
      constexpr uint32_t iO = idesc_f16(kBM, kHD, 1);
      auto issue_s = [&](int js) {
        tc_fence_after();
        const uint32_t sKj = sConv + (js & 1) * Lay::kConv;
#pragma unroll
        for (int ks = 0; ks < kHD / 16; ++ks) {
          const uint32_t off = (ks >> 2) * kAtom + (ks & 3) * 32;  // atom, then 16 dims within it
          mma_bf16_tmem_a(tmem, tmem + Lay::kTmemQ + ks * 8, desc_sw128(sKj + off), iS, ks > 0);
        }
        mma_commit(b_sfull);
        mma_commit(conv_kempty(js & 1));
      };
      ok = mbar_wait(b_qready, 0);
      int js = 0;
      if (ok && n_kt > 0) {
        ok = mbar_wait(conv_kfull(0), 0);
        if (ok) issue_s(js++);
      }
      for (int j = 0; j < n_kt && ok; ++j) {
        const unsigned long long t0 = globaltimer_ns();
        while (true) {
          if (js < n_kt && mbar_test(b_sfree, (js - 1) & 1) && mbar_test(conv_kfull(js & 1), (js >> 1) & 1))
            issue_s(js++);
          if (mbar_test(b_pfull(j & 1), (j >> 1) & 1) && mbar_test(conv_vfull, j & 1)) break;
          if (globaltimer_ns() - t0 > kWaitLimitNs) {
            ok = false;
            break;
          }
        }
        if (!ok) break;
        tc_fence_after();
        const uint32_t sVj = sConv + 2 * Lay::kConv;
        // O[:, 0:D] += P V: V is MN-major over its 64-column atoms (LBO = atom stride)
#pragma unroll
        for (int ks = 0; ks < kBN / 16; ++ks)
          mma_bf16_tmem_a(tmem + Lay::kTmemO, tmem + Lay::kTmemP + (j & 1) * 64 + ks * 8,
                          desc_sw128(sVj + ks * 2048, kAtom, 1024), iO, (j > 0 || ks > 0) ? 1u : 0u);
        mma_commit(b_pvdone(j & 1));
        mma_commit(conv_vempty);
      }
      if (!ok) set_device_error(p.err_word, TS_DEVERR_TIMEOUT);
    }
  } else {
    // ---------------- softmax warps: thread = query row ----------------
    // Row r of head slot hs (lane hs * Rw + r): query head (h0 + hs) * g + r.
    // A warp whose rows are all padding only keeps the barrier protocol.
    const int hs = tid / Rw, r = tid % Rw;
    const bool warp_real = (warp * 32) % Rw < R;
    const uint32_t trow = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const uint32_t hcol = static_cast<uint32_t>(hs * kPS);
    const bool real = r < R;
    const int lim = real ? L : 0;  // keys the row attends (padding: none)
    // Q row -> f16 in TMEM, scaled by 2^-e so that its largest magnitude
    // lands in [2^14, 2^15); the score scale takes 2^e back.
    float sl = p.scale_log2;
    {
      const uint4* src = reinterpret_cast<const uint4*>(
          p.q + (static_cast<int64_t>(b) * p.H_q + (h0 + hs) * p.g + (real ? r : 0)) * kHD);
      float amax = 0.f;
      if (real) {
#pragma unroll
        for (int c = 0; c < kHD / 8; ++c) {
          const uint4 v = src[c];
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float2 f = bf16x2_to_float2(w[k]);
            amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
          }
        }
      }
      int e = 0;
      if (amax > 0.f) e = max(static_cast<int>((__float_as_uint(amax) >> 23) & 0xFF) - 127 - 14, -100);
      const float down = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);  // 2^-e
      sl *= __uint_as_float(static_cast<uint32_t>(127 + e) << 23);               // 2^e
#pragma unroll
      for (int c0 = 0; c0 < kHD; c0 += 32) {  // 32 elements = 16 TMEM columns
        uint32_t pk[16];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint4 v = real ? src[(c0 >> 3) + c] : make_uint4(0u, 0u, 0u, 0u);
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float2 f = bf16x2_to_float2(w[k]);
            pk[c * 4 + k] = f16x2_bits(f.x * down, f.y * down);
          }
        }
        tmem_st16(trow + Lay::kTmemQ + c0 / 2, pk);
      }
      // a copy writes only its own head's columns of P: the others stay zero
      uint32_t z[16];
#pragma unroll
      for (int x = 0; x < 16; ++x) z[x] = 0u;
#pragma unroll
      for (int c = 0; c < 128; c += 16) tmem_st16(trow + Lay::kTmemP + c, z);  // both P buffers
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_qready);
    }
    const float* scl_base = reinterpret_cast<const float*>(smem + Lay::kOffScl);
    float m = -INFINITY, l = 0.f;
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
      // the tile's scales: written by the converters before the tile's S
      const float* ksc = scl_base + (j & 1) * kBM;
      const float* vsc = scl_base + 2 * kBM;
      float ms = 0.f;
      if (warp_real) {
        const int key0 = j * kKeys;
        float mx = -INFINITY;
#pragma unroll
        for (int pb = 0; pb < TP; ++pb) {
#pragma unroll
          for (int x = 0; x < 16; x += 4) {
            const float4 k4 = *reinterpret_cast<const float4*>(ksc + pb * HG * kPS + hcol + x);
            const float kk[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
            for (int y = 0; y < 4; ++y) {
              const int c = pb * 16 + x + y;
              s[c] = key0 + c < lim ? s[c] * kk[y] * sl : -INFINITY;
              mx = fmaxf(mx, s[c]);
            }
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
      // the tile's V scales are laid out with its widened V rows
      ok = mbar_wait(conv_vfull, j & 1);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      if (warp_real) {
        float2 ls2 = make_float2(0.f, 0.f);
        // P straight into TMEM (the P V MMA reads its A operand there), each
        // probability times its key's V scale
#pragma unroll
        for (int pb = 0; pb < TP; ++pb) {
          uint32_t pk[8];
#pragma unroll
          for (int x = 0; x < 16; x += 4) {
            const float4 v4 = *reinterpret_cast<const float4*>(vsc + pb * HG * kPS + hcol + x);
            const float e0 = fast_exp2(s[pb * 16 + x] - ms), e1 = fast_exp2(s[pb * 16 + x + 1] - ms);
            const float e2 = fast_exp2(s[pb * 16 + x + 2] - ms), e3 = fast_exp2(s[pb * 16 + x + 3] - ms);
            ls2 = __fadd2_rn(ls2, make_float2(e0 + e2, e1 + e3));
            pk[x / 2] = f16x2_bits(e0 * v4.x, e1 * v4.y);
            pk[x / 2 + 1] = f16x2_bits(e2 * v4.z, e3 * v4.w);
          }
          tmem_st8(trow + Lay::kTmemP + (j & 1) * 64 + (pb * HG * kPS + hcol) / 2, pk);
        }
        tmem_wait_st();
        l += ls2.x + ls2.y;
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
      const int64_t row = static_cast<int64_t>(b) * p.H_q + (h0 + hs) * p.g + r;
      const float inv = l > 0.f ? 1.0f / l : 0.f;
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

// 3-D map over an fp8 pool [P * 16 rows][H_kv][D] bytes taken as (byte, pool
// row, kv head): a box is one page (16 rows) of hg heads, landing head by
// head, [hg][16][D]; no swizzle (the converters rearrange), zero fill.
ts_status make_map(CUtensorMap* map, const void* pool, int num_pages, int H_kv, int D, int hg) {
  auto fn = tensor_map_encoder();
  if (!fn) return fail(TS_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(num_pages) * kPS,
                        static_cast<cuuint64_t>(H_kv)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(H_kv) * D, static_cast<cuuint64_t>(D)};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(D), kPS, static_cast<cuuint32_t>(hg)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult res = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(pool), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (res != CUDA_SUCCESS) return fail(TS_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(res));
  return TS_OK;
}

template <int kHD, int kHG>
ts_status launch(const Fp8Params& prm, const CUtensorMap& kmap, const CUtensorMap& vmap, int B, cudaStream_t s) {
  using Lay = Layout<kHD>;
  ts_status st = prepare_once(reinterpret_cast<const void*>(fp8_tc_kernel<kHD, kHG>), [](const void* k) {
    ts_status s2 = cuda_check(cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, Layout<kHD>::kSmem),
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
  cfg.gridDim = dim3(static_cast<unsigned>(B) * static_cast<unsigned>(prm.H_kv / kHG));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Lay::kSmem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  LaunchTrace trace("fp8_tc_kernel", s);
  return cuda_check(cudaLaunchKernelEx(&cfg, fp8_tc_kernel<kHD, kHG>, prm, kmap, vmap), "fp8 tensor-core launch");
}

}  // namespace

// Runs the tensor-core path when TS_FP8_DECODE_PATH=tensor asks for it and
// the shape applies: page 16, D 64 or 128, 2 or 4 kv heads per CTA (g <= 32
// query rows per kv head; the most heads that keep the grid at 1.5 waves of
// SMs, else 2), a stage's scale rows within 2 KB. TS_FP8_HEAD_GROUP=2/4
// forces the head count. TS_ERR_UNSUPPORTED otherwise, with nothing
// enqueued, so that the caller takes the CUDA-core path. Not the default: on
// the Llama-3-8B layer shape it measured 142 us against the CUDA-core
// kernel's 107 us, the widening of every code on its way to the tensor
// cores costing about 50 us of it.
ts_status launch_fp8_decode_tc(const void* q, const void* k_pool, const void* v_pool, const float* k_scale,
                               const float* v_scale, const int32_t* block_table, int32_t bt_stride,
                               const int32_t* seq_lens, int32_t B, int32_t H_q, int32_t H_kv, int32_t D,
                               int32_t page_size, int32_t num_pages, float scale, void* out, float* lse,
                               uint32_t* err_word, cudaStream_t stream) {
  const char* path = getenv("TS_FP8_DECODE_PATH");
  const bool force_tc = path && std::strcmp(path, "tensor") == 0;
  if (!force_tc || B <= 0 || H_kv <= 0 || H_q % H_kv != 0 || page_size != kPS || (D != 64 && D != 128) ||
      num_pages <= 0 || bt_stride <= 0 || static_cast<long long>(num_pages) * kPS > INT32_MAX)
    return TS_ERR_UNSUPPORTED;
  const int g = H_q / H_kv;
  const int hg_max = g <= 32 ? 4 : (g <= 64 ? 2 : 1);
  int hg = 0;
  for (int c = hg_max; c > 1; c >>= 1)
    if (H_kv % c == 0 && static_cast<int64_t>(B) * (H_kv / c) * 2 >= 3 * static_cast<int64_t>(device_sm_count())) {
      hg = c;
      break;
    }
  if (hg == 0 && hg_max >= 2 && H_kv % 2 == 0) hg = 2;
  if (const char* e = getenv("TS_FP8_HEAD_GROUP")) {
    const int f = atoi(e);
    if ((f == 2 || f == 4) && f <= hg_max && H_kv % f == 0) hg = f;
  }
  if (hg == 0 || (kPagesPerTile / hg) * kPS * H_kv * 4 > kScaleMax ||
      static_cast<int64_t>(B) * (H_kv / hg) > 0x7fffffff)
    return TS_ERR_UNSUPPORTED;
  Fp8Params prm;
  prm.q = static_cast<const __nv_bfloat16*>(q);
  prm.out = static_cast<__nv_bfloat16*>(out);
  prm.lse = lse;
  prm.block_table = block_table;
  prm.seq_lens = seq_lens;
  prm.k_scale = k_scale;
  prm.v_scale = v_scale;
  prm.B = B;
  prm.bt_stride = bt_stride;
  prm.H_q = H_q;
  prm.H_kv = H_kv;
  prm.g = g;
  prm.num_pages = num_pages;
  prm.scale_log2 = scale * kLog2eC;
  prm.err_word = err_word;
  CUtensorMap kmap, vmap;
  ts_status st = make_map(&kmap, k_pool, num_pages, H_kv, D, hg);
  if (st != TS_OK) return st;
  st = make_map(&vmap, v_pool, num_pages, H_kv, D, hg);
  if (st != TS_OK) return st;
  if (D == 64)
    return hg == 4 ? launch<64, 4>(prm, kmap, vmap, B, stream) : launch<64, 2>(prm, kmap, vmap, B, stream);
  return hg == 4 ? launch<128, 4>(prm, kmap, vmap, B, stream) : launch<128, 2>(prm, kmap, vmap, B, stream);
}

}  // namespace ts
