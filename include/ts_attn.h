/*
 * ts_attn.h - decode-step attention over a paged KV cache, for GB300 (sm_103a).
 *
 * A C ABI: plain pointers and sizes, no framework types. Every function that
 * takes a `stream` (a cudaStream_t passed as void*, NULL = legacy default
 * stream) is asynchronous on it: it validates its arguments on the host,
 * enqueues its kernels and returns. Inputs must stay alive and unmodified
 * until the stream reaches the call. The library never allocates device
 * memory and keeps no state besides a per-device cache of the SM count and
 * of kernel attributes; scratch memory ("workspace") is passed in by the
 * caller and sized by the matching *_workspace_size function.
 *
 * Shared conventions
 *   - Element types: TS_F32 (float) or TS_BF16 (bfloat16, round-to-nearest-
 *     even on output). Arithmetic is float32 everywhere (fp32 accumulate).
 *   - K/V page pool layout ("NHD"): [num_pages, page_size, H_kv, D], row-major.
 *     Token t of sequence b lives in physical page block_table[b*bt_stride +
 *     t/page_size] at row t%page_size. (SwiftLLM page, section 3.1: the cache
 *     is split into fixed-size blocks found through a per-request block
 *     table; section 5.1: attention takes the query, block tables and
 *     context lengths.)
 *     Pools may be any size the device holds (byte offsets are 64-bit), but
 *     their row count num_pages * page_size must stay below 2^31 (rows are
 *     32-bit TMA coordinates); a larger num_pages is an argument error.
 *   - GQA: query head h reads kv head h / (H_q / H_kv).
 *   - LSE outputs are natural-log log-sum-exp of the scaled scores, float32.
 *     A sequence of length 0 yields O = 0 and LSE = -inf.
 *   - Device-side safety: a page id outside [0, num_pages) is never
 *     dereferenced. Attention treats the tokens of such a page as absent and
 *     sets bit TS_DEVERR_PAGE_RANGE in the workspace's error word; the append
 *     skips the write. No kernel traps; every pipeline wait is time-bounded
 *     and on timeout sets TS_DEVERR_TIMEOUT and leaves the kernel.
 *   - Errors: argument errors are returned before anything is enqueued; a
 *     failed launch returns TS_ERR_CUDA. ts_last_error_detail() describes the
 *     last non-OK status of the calling thread.
 *   - Overlap with the previous kernel (programmatic dependent launch): the
 *     append and paged-attention kernels may start while the previous kernel
 *     of the stream is still running, if that kernel allows it (a kernel that
 *     does not use programmatic dependent launch never does). Before waiting
 *     for it, ts_paged_decode_attn reads only seq_lens, the block table and,
 *     in cascade mode, the group descriptors; so a kernel that triggers its
 *     dependents early must not write those. Every other input is read, and
 *     every output written, after the wait. The library's own kernels follow
 *     this rule, so back-to-back calls are safe.
 */
#ifndef TS_ATTN_H_
#define TS_ATTN_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define TS_API __attribute__((visibility("default")))
#else
#define TS_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TS_OK = 0,
  TS_ERR_INVALID_ARG = 1,   /* null pointer, bad size, inconsistent shapes */
  TS_ERR_UNSUPPORTED = 2,   /* valid but not compiled (head dim, group size...) */
  TS_ERR_WORKSPACE = 3,     /* workspace missing, too small or misaligned */
  TS_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed */
  TS_ERR_CAPACITY = 5       /* a caller-provided output array is too small */
} ts_status;

typedef enum { TS_F32 = 0, TS_BF16 = 1 } ts_dtype;

/* Bits of the sticky device error word kept in the first 4 bytes of an
 * attention workspace. The library sets bits and never clears them. */
#define TS_DEVERR_PAGE_RANGE 0x1u
#define TS_DEVERR_TIMEOUT 0x2u
/* A kernel found its dynamic shared memory not aligned as its tile layout
 * needs (1024 bytes) and returned without computing anything. */
#define TS_DEVERR_SMEM_ALIGN 0x4u
/* A draft tree's parent index was not an earlier node or -1: the row's path
 * stops there (ts_paged_decode_tree_attn). */
#define TS_DEVERR_TREE 0x8u

/* Human-readable name of a status code. Never NULL. */
TS_API const char* ts_status_string(int status);

/* Details of the last non-OK status returned on the calling thread ("" if none). */
TS_API const char* ts_last_error_detail(void);

/* Library version string. */
TS_API const char* ts_version(void);

/*
 * ts_kv_append - write one new token's K and V per sequence into the pools.
 *
 * SwiftLLM page, section 3.1: blocks are allocated to a request on demand;
 * the token at position pos lands in page block_table[b][pos / page_size],
 * row pos % page_size. The block table must already hold that page.
 *
 *   k_new, v_new  device [B, H_kv, D] of dtype
 *   k_pool,v_pool device [num_pages, page_size, H_kv, D] of dtype (written)
 *   block_table   device int32 [B, bt_stride]
 *   positions     device int32 [B]: token index to write (= cached length
 *                 before the append); afterwards attention covers pos + 1
 *                 tokens.
 * The copy is bit-exact. Rows whose page index or page id is out of range
 * are skipped. B == 0 returns TS_OK with nothing enqueued.
 */
TS_API ts_status ts_kv_append(const void* k_new, const void* v_new, void* k_pool, void* v_pool,
                       const int32_t* block_table, int32_t bt_stride, const int32_t* positions,
                       int32_t B, int32_t H_kv, int32_t D, int32_t page_size, int32_t num_pages,
                       ts_dtype dtype, void* stream);

/*
 * ts_paged_decode_workspace_size - bytes of workspace ts_paged_decode_attn
 * needs on the current device for a batch of B sequences. Depends on the
 * device's SM count (the kernel runs one persistent CTA per SM). Returns 0 on
 * invalid arguments.
 */
TS_API size_t ts_paged_decode_workspace_size(int32_t B, int32_t H_q, int32_t D);

/*
 * ts_paged_decode_attn - one decode step of GQA attention over a paged cache.
 *
 * For every sequence b and query head h (kv head h / g, g = H_q / H_kv):
 *   s_t = scale * <q[b,h,:], K_b[t,:]> for t < seq_lens[b],
 *   O[b,h,:] = sum_t softmax(s)_t V_b[t,:],  LSE[b,h] = log sum_t exp(s_t).
 *
 * Flash-decoding split-KV (TokenSpeed deep dive, section 7 fig. 3 and 7.1):
 * the pages of the whole batch are cut into equal contiguous ranges, one per
 * SM; a sequence cut across ranges produces float32 partial (O, LSE) states
 * in the workspace that a second kernel reduces by LSE. Planning runs on the
 * device from seq_lens, so no host copy of the lengths is needed and the
 * call can be captured in a CUDA graph.
 *
 *   q             device [B, H_q, D] of dtype
 *   k_pool,v_pool device [num_pages, page_size, H_kv, D] of dtype
 *   block_table   device int32 [B, bt_stride]
 *   seq_lens      device int32 [B] tokens attended per sequence (>= 0)
 *   out           device [B, H_q, D] of dtype (written)
 *   lse           device float32 [B, H_q] (written) or NULL
 *   workspace     device, >= ts_paged_decode_workspace_size(B, H_q, D) bytes,
 *                 256-byte aligned; its first 4 bytes are the sticky device
 *                 error word (see TS_DEVERR_*), zero it to check it later.
 * Supported: D in {64, 128}, H_q / H_kv in {1, 2, 4, 8}, H_kv in {1, 2, 4, 8},
 * page_size in {8, 16, 32}, and one page of K+V for all kv heads within the
 * shared-memory stage budget. Others return TS_ERR_UNSUPPORTED.
 */
TS_API ts_status ts_paged_decode_attn(const void* q, const void* k_pool, const void* v_pool,
                               const int32_t* block_table, int32_t bt_stride,
                               const int32_t* seq_lens, int32_t B, int32_t H_q, int32_t H_kv,
                               int32_t D, int32_t page_size, int32_t num_pages, float scale,
                               ts_dtype dtype, void* out, float* lse, void* workspace,
                               size_t workspace_bytes, void* stream);

/*
 * ts_paged_decode_attn_noalloc - ts_paged_decode_attn without a workspace.
 *
 * The pages have no counterpart of this call; it exists for callers that
 * cannot allocate device memory: a plugin that its host runtime hands only
 * input and output buffers, or an engine that has reserved all free HBM for
 * its KV-cache pool and must not pay cudaMalloc's latency and implicit
 * synchronisation in its decode loop. Same arguments and results as
 * ts_paged_decode_attn minus the workspace. It allocates nothing: the
 * split-KV scratch is a fixed array of TS_NOALLOC_SCRATCH_BYTES bytes inside
 * the library's device image, held by every GPU that loads the library until
 * the process exits.
 *   - Sizes whose scratch need (ts_paged_decode_workspace_size(B, H_q, D))
 *     exceeds TS_NOALLOC_SCRATCH_BYTES return TS_ERR_WORKSPACE, nothing
 *     enqueued. On a 152-SM GB300 that allows H_q * D up to about 13,000 for
 *     moderate batches (e.g. 32 x 128 with B up to ~1.4 million).
 *   - All calls on one device share the array: calls that may overlap on the
 *     GPU (unordered streams) race and give wrong results.
 *   - The error word in the array is cleared at the start of every call;
 *     ts_read_device_error(NULL, ...) reads it for the current device, so
 *     device-side errors (page id out of range, timed-out wait) of the last
 *     call are visible as with a workspace.
 *   - Arguments and shape are checked first (TS_ERR_INVALID_ARG,
 *     TS_ERR_UNSUPPORTED), then the scratch size (TS_ERR_WORKSPACE).
 *   - The first call on each device looks up the array's address with that
 *     device current; make it before any stream capture.
 *   - Under CUDA's default lazy module loading, the array's memory is
 *     committed on a device when the library's module is first loaded there:
 *     at the first call (or ts_read_device_error(NULL, ...)). A caller that
 *     hands all free HBM to its KV-cache pool must make that first call
 *     before, or it fails with TS_ERR_CUDA (out of memory). Later calls
 *     allocate nothing.
 */
#define TS_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)
TS_API ts_status ts_paged_decode_attn_noalloc(const void* q, const void* k_pool,
                                              const void* v_pool, const int32_t* block_table,
                                              int32_t bt_stride, const int32_t* seq_lens,
                                              int32_t B, int32_t H_q, int32_t H_kv, int32_t D,
                                              int32_t page_size, int32_t num_pages, float scale,
                                              ts_dtype dtype, void* out, float* lse, void* stream);

/*
 * ts_fold_sq_factor - query tokens folded into the rows of one tile.
 *
 * TokenSpeed deep dive, section 7.2 (fold_sq_factor): the largest F with
 * q_len % F == 0 and num_heads * F <= tile_rows, so that a tile holds
 * num_heads * F rows and a sequence's q_len tokens take q_len / F tiles
 * (64 heads, 4 tokens, 128-row tile: F = 2). Returns 0 if an argument is not
 * positive. Host only.
 */
TS_API int32_t ts_fold_sq_factor(int32_t num_heads, int32_t q_len, int32_t tile_rows);

/*
 * ts_paged_decode_window_attn - decode attention over a sliding-window KV
 * group: each sequence's query attends its last `window` tokens only.
 *
 * TokenSpeed deep dive, section 4.1: a sliding_window KV group declares
 * sliding_window_tokens; tokenspeed 딥다이브 (fiv.co.kr), section 6-3: its
 * block table keeps the real blocks at the back of the window and a
 * placeholder (block 0) in the slots in front of it. The query of a sequence
 * with L = seq_lens[b] tokens attends positions max(0, L - window) .. L - 1;
 * token t lives in slot t / page_size at row t % page_size as everywhere, so
 * the slots wholly in front of the window (placeholders or stale pages) and
 * the rows of the window's first page in front of it are never read. With
 * window >= L this is ts_paged_decode_attn's result.
 *
 *   window    tokens, >= 1 (else TS_ERR_INVALID_ARG)
 *   workspace >= ts_paged_decode_workspace_size(B, H_q, D)
 *   all other arguments, support (dtype f32 / bf16) and errors as in
 *   ts_paged_decode_attn.
 */
TS_API ts_status ts_paged_decode_window_attn(const void* q, const void* k_pool, const void* v_pool,
                                             const int32_t* block_table, int32_t bt_stride,
                                             const int32_t* seq_lens, int32_t B, int32_t H_q, int32_t H_kv,
                                             int32_t D, int32_t page_size, int32_t num_pages, int32_t window,
                                             float scale, ts_dtype dtype, void* out, float* lse,
                                             void* workspace, size_t workspace_bytes, void* stream);

/*
 * ts_paged_decode_multi_workspace_size - workspace bytes for
 * ts_paged_decode_multi_attn (B sequences of q_len query tokens). Returns 0 on
 * invalid arguments.
 */
TS_API size_t ts_paged_decode_multi_workspace_size(int32_t B, int32_t q_len, int32_t H_q, int32_t D);

/*
 * ts_paged_decode_multi_attn - decode with q_len new query tokens per sequence
 * (speculative or multi-token verification).
 *
 * The q_len tokens' K/V rows are already in the cache (ts_kv_append once per
 * token) and seq_lens counts them. Query token j of sequence b sits at
 * position seq_lens[b] - q_len + j and attends tokens 0 .. that position
 * (causal among the new tokens); each (token, head) row is otherwise the
 * single-query decode of ts_paged_decode_attn. Tokens are folded into the
 * rows of a kv head (TokenSpeed deep dive, section 7.2). With R = q_len * g
 * rows per kv head from 8 to 128 (bf16, page 16, D 64 or 128) a tensor-core
 * kernel takes all R rows in one pass: S = Q K^T and P V on tcgen05, one CTA
 * per sequence and group of 1, 2 or 4 kv heads, P rounded to bf16 for the
 * product (O normalised by the sum of the rounded P; the LSE from the
 * unrounded sum). Otherwise the CUDA-core kernel folds F tokens with the g
 * heads of a kv head when g * F is 1, 2, 4 or 8 (the largest such factor F of
 * q_len) and runs the others as separate passes over the pages. The
 * environment variable TS_MULTI_QUERY_PATH=cuda|tensor forces one path where
 * the shape allows it.
 *
 *   q             device [B, q_len, H_q, D] of dtype
 *   out           device [B, q_len, H_q, D] of dtype (written)
 *   lse           device float32 [B, q_len, H_q] (written) or NULL
 *   seq_lens      device int32 [B], each >= q_len (rows of a token whose
 *                 position would be negative get O = 0, LSE = -inf)
 *   workspace     >= ts_paged_decode_multi_workspace_size(B, q_len, H_q, D)
 *   other arguments, support and errors as in ts_paged_decode_attn;
 *   q_len >= 1 (q_len == 1 gives exactly ts_paged_decode_attn's result).
 */
TS_API ts_status ts_paged_decode_multi_attn(const void* q, const void* k_pool, const void* v_pool,
                                            const int32_t* block_table, int32_t bt_stride,
                                            const int32_t* seq_lens, int32_t B, int32_t q_len,
                                            int32_t H_q, int32_t H_kv, int32_t D, int32_t page_size,
                                            int32_t num_pages, float scale, ts_dtype dtype, void* out,
                                            float* lse, void* workspace, size_t workspace_bytes,
                                            void* stream);

/*
 * ts_paged_decode_tree_attn - verify a tree of draft tokens in one decode
 * step (tree speculation).
 *
 * TokenSpeed deep dive, section 0 (the tree-speculation design document) and
 * its closing section (tree speculation as a serving workload). Each
 * sequence brings n draft tokens that form a tree: parents[b, j] is token j's
 * parent, an earlier token (< j) or -1 for a child of the last committed
 * token. Their K/V rows are already in the cache at positions L - n + j, in
 * token order (seq_lens counts them). Token j's query, for every query head,
 * attends the committed context (positions 0 .. L - n - 1) and the draft
 * tokens on its own path (its ancestors and itself), not its siblings'
 * branches. A chain (parents[j] = j - 1) gives ts_paged_decode_multi_attn's
 * causal result.
 *
 *   q        device bf16 [B, n, H_q, D];  out device bf16 [B, n, H_q, D]
 *   lse      device float32 [B, n, H_q] or NULL
 *   parents  device int32 [B, n]; a parent that is not -1 or an earlier token
 *            sets TS_DEVERR_TREE and ends that row's path there
 *   workspace >= 256 bytes, 256-byte aligned (its first 4 bytes are the
 *            error word; zero it to check it later)
 *   other arguments as ts_paged_decode_attn.
 * Supported (tensor-core path): bf16, page_size 16, D 64 or 128, 1 <= n <= 64,
 * n * H_q / H_kv <= 128; otherwise TS_ERR_UNSUPPORTED with nothing enqueued.
 * A sequence with L < n attends only the rows that exist (L >= n expected).
 */
TS_API ts_status ts_paged_decode_tree_attn(const void* q, const void* k_pool, const void* v_pool,
                                           const int32_t* block_table, int32_t bt_stride,
                                           const int32_t* seq_lens, const int32_t* parents, int32_t B,
                                           int32_t n, int32_t H_q, int32_t H_kv, int32_t D,
                                           int32_t page_size, int32_t num_pages, float scale,
                                           ts_dtype dtype, void* out, float* lse, void* workspace,
                                           size_t workspace_bytes, void* stream);

/*
 * ts_kv_append_fp8 - quantize one new token's K and V per sequence into an
 * fp8 (e4m3fn) cache.
 *
 * Placement as ts_kv_append. Quantization per token group (tokenspeed
 * 딥다이브, fiv.co.kr, section 6-4): a group is one (token, kv head) row of D
 * values; scale = max(max |x|, 1e-10) / 448 and code = e4m3fn(clamp(x / scale,
 * -448, 448)), the scale and the division in float32 rounded to nearest even,
 * the cast rounded to nearest even. Bit-exact with that definition.
 *
 *   k_new, v_new    device [B, H_kv, D] of dtype (bf16 or f32)
 *   k_pool, v_pool  device uint8 [num_pages, page_size, H_kv, D] e4m3fn codes (written)
 *   k_scale,v_scale device float32 [num_pages, page_size, H_kv] (written)
 *   block_table, positions, sizes as ts_kv_append. D in {64, 128}.
 */
TS_API ts_status ts_kv_append_fp8(const void* k_new, const void* v_new, void* k_pool, void* v_pool,
                                  float* k_scale, float* v_scale, const int32_t* block_table,
                                  int32_t bt_stride, const int32_t* positions, int32_t B, int32_t H_kv,
                                  int32_t D, int32_t page_size, int32_t num_pages, ts_dtype dtype,
                                  void* stream);

/*
 * ts_paged_decode_fp8_attn - ts_paged_decode_attn over an fp8 (e4m3fn) cache.
 *
 * Computes ts_paged_decode_attn's result over the cache's reconstruction
 * K[t] = code * k_scale[t] (and the same for V), with bf16 queries and
 * output: the kernel widens the codes exactly and applies each row's scale
 * to its score (K) and to its softmax weight (V), in float32.
 *
 *   q               device bf16 [B, H_q, D];  out device bf16 [B, H_q, D]
 *   k_pool, v_pool  device uint8 [num_pages, page_size, H_kv, D] e4m3fn codes
 *   k_scale,v_scale device float32 [num_pages, page_size, H_kv], 16-byte aligned
 *   workspace       >= ts_paged_decode_workspace_size(B, H_q, D)
 *   other arguments as ts_paged_decode_attn. Supported: D in {64, 128},
 *   H_q / H_kv in {1, 2, 4}, H_kv in {1, 2, 4, 8}, page_size in {8, 16, 32}.
 *
 * The CUDA-core split-KV kernel runs it. With the environment variable
 * TS_FP8_DECODE_PATH=tensor a tensor-core kernel runs it instead where the
 * shape allows (page 16, 2 or 4 kv heads per CTA): the codes are widened to
 * f16 on chip and the probabilities rounded to f16 for the P V product (the
 * row sum and the LSE stay float32). With TS_FP8_DECODE_PATH=mma, at 32
 * query heads over 8 kv heads, head dim 128 and page 16, a kernel that
 * multiplies the codes themselves (kind::f8f6f4) runs it: the query and the
 * probabilities enter as three e4m3 terms each (relative error at most
 * 2^-12, below bf16's rounding), the scores take the key scales, the
 * probabilities the value scales and a power-of-two gain; cut sequences are
 * merged inside the kernel. Both are measured slower than the CUDA-core
 * kernel on the Llama-3-8B layer shape, hence not the default.
 */
TS_API ts_status ts_paged_decode_fp8_attn(const void* q, const void* k_pool, const void* v_pool,
                                          const float* k_scale, const float* v_scale,
                                          const int32_t* block_table, int32_t bt_stride,
                                          const int32_t* seq_lens, int32_t B, int32_t H_q, int32_t H_kv,
                                          int32_t D, int32_t page_size, int32_t num_pages, float scale,
                                          void* out, float* lse, void* workspace, size_t workspace_bytes,
                                          void* stream);

/*
 * ts_merge_states - merge two attention states over disjoint key sets.
 *
 * Per row r: m = max(lse_a, lse_b), w_a = exp(lse_a - m), w_b = exp(lse_b - m),
 *   O = (w_a O_a + w_b O_b) / (w_a + w_b),  LSE = m + log(w_a + w_b).
 * A state with LSE = -inf has weight 0; two empty states give O = 0,
 * LSE = -inf. (TokenSpeed deep dive, section 7 fig. 3: partials are reduced
 * by their LSE; Tokasaurus blog, shared-prefix attention is combined with the
 * per-sequence part.)
 *
 *   o_a, o_b   device [rows, D] of dtype;  lse_a, lse_b device float32 [rows]
 *   o_out      device [rows, D] of dtype;  lse_out device float32 [rows] or NULL
 * o_out may alias o_a or o_b (each element is read before it is written by
 * the same thread). D must be a multiple of 4 (bf16: of 8), at most 1024.
 */
TS_API ts_status ts_merge_states(const void* o_a, const float* lse_a, const void* o_b,
                          const float* lse_b, void* o_out, float* lse_out, int64_t rows,
                          int32_t D, ts_dtype dtype, void* stream);

/*
 * Shared-prefix groups (Tokasaurus blog, "Dynamic prefix identification and
 * exploration": a greedy depth-first search before each forward pass finds
 * the longest shared prefixes; Hydragen / cascade attention then computes
 * attention over each shared prefix once per group).
 *
 * CSR arrays, all int32. The caller allocates every array; the capacities say
 * how large they are.
 *   prefix_indptr[capacity_groups + 1], prefix_pages[capacity_prefix_pages]
 *   prefix_len[capacity_groups]        tokens shared (= pages * page_size)
 *   member_indptr[capacity_groups + 1], member_ids[capacity_members]
 *   group_of[B]                        group of each sequence, -1 if none
 */
typedef struct {
  int32_t num_groups;
  int32_t* prefix_indptr;
  int32_t* prefix_pages;
  int32_t* prefix_len;
  int32_t* member_indptr;
  int32_t* member_ids;
  int32_t* group_of;
  int32_t capacity_groups;
  int32_t capacity_prefix_pages;
  int32_t capacity_members;
} ts_prefix_groups;

/*
 * ts_group_prefixes - host-side greedy longest-shared-prefix grouping.
 *
 * Runs on the CPU over HOST copies of the block table and lengths. Prefixes
 * are whole pages shared by physical page id; each member keeps at least one
 * suffix token (a member of length L shares at most (L-1)/page_size pages).
 * Greedy longest-first: repeatedly the deepest prefix shared by at least
 * min_group ungrouped sequences becomes a group with all of them (ties: more
 * members first, then the smaller page-id path). Sequences in no group take
 * the flat paged path. min_group >= 2. Returns TS_ERR_CAPACITY if an output
 * array is too small (num_groups is then the count needed, if known).
 */
TS_API ts_status ts_group_prefixes(const int32_t* block_table, int32_t bt_stride, const int32_t* seq_lens,
                            int32_t B, int32_t page_size, int32_t min_group, ts_prefix_groups* out);

/*
 * A forest of shared prefixes (ts_group_prefixes_nested). Nodes are listed
 * level by level: level l holds nodes level_indptr[l] .. level_indptr[l+1]-1
 * (roots at level 0). Node i owns the pages of its own stretch only,
 * prefix_pages[prefix_indptr[i] .. prefix_indptr[i+1]-1] (the path above it
 * belongs to its ancestors); prefix_len[i] counts the tokens shared from the
 * root through node i; parent[i] is its parent node or -1; its members
 * (member_ids[member_indptr[i] ..]) are all sequences that share its path.
 * group_of[b] is the deepest node of sequence b, -1 if none. All arrays int32
 * and caller-allocated (capacities say their sizes: level_indptr holds
 * capacity_levels + 1, prefix_indptr and member_indptr capacity_nodes + 1).
 */
typedef struct {
  int32_t num_nodes;
  int32_t num_levels;
  int32_t* level_indptr;
  int32_t* parent;
  int32_t* prefix_indptr;
  int32_t* prefix_pages;
  int32_t* prefix_len;
  int32_t* member_indptr;
  int32_t* member_ids;
  int32_t* group_of;
  int32_t capacity_nodes;
  int32_t capacity_levels;
  int32_t capacity_prefix_pages;
  int32_t capacity_members;
} ts_prefix_forest;

/*
 * ts_group_prefixes_nested - the greedy longest-shared-prefix search kept as a
 * tree (Tokasaurus blog, "Dynamic prefix identification and exploration").
 *
 * Host only, over host copies of the block table and lengths; same page and
 * cap rules as ts_group_prefixes (whole pages by physical id, a member of
 * length L shares at most (L-1)/page_size pages). A node is a maximal stretch
 * of pages shared by at least min_group sequences; at its end, members that
 * can go deeper branch on the next page and branches of at least min_group
 * sequences become child nodes. Each sequence's shared depth is then the
 * largest d for which at least min_group sequences (itself included) share
 * its first d pages within their caps. Returns TS_ERR_CAPACITY (with
 * num_nodes / num_levels set to the counts needed) if an array is too small.
 */
TS_API ts_status ts_group_prefixes_nested(const int32_t* block_table, int32_t bt_stride,
                                          const int32_t* seq_lens, int32_t B, int32_t page_size,
                                          int32_t min_group, ts_prefix_forest* out);

/*
 * ts_cascade_decode_workspace_size - workspace bytes for ts_cascade_decode_attn.
 */
TS_API size_t ts_cascade_decode_workspace_size(int32_t B, int32_t H_q, int32_t D);

/*
 * ts_cascade_decode_attn - decode attention with shared prefixes computed once.
 *
 * Same result as ts_paged_decode_attn over the full block tables (up to
 * float32 rounding). For each group the queries of all members (members * g
 * rows per kv head) attend the group's prefix pages as one dense
 * tensor-core product (tcgen05, accumulators in TMEM); each sequence's own
 * pages (the suffix after its group's prefix, or everything if ungrouped)
 * go through the paged split-KV path; the two states are merged by LSE.
 *
 *   groups       device copies of the CSR arrays of ts_group_prefixes
 *                (num_groups, prefix_indptr, prefix_pages, prefix_len,
 *                member_indptr, member_ids, group_of; capacities ignored)
 *   other arguments as in ts_paged_decode_attn (seq_lens = full lengths).
 * Supported: D == 64 with H_q / H_kv == 4 and bf16 for the tensor-core
 * prefix; page_size 16.
 */
TS_API ts_status ts_cascade_decode_attn(const void* q, const void* k_pool, const void* v_pool,
                                 const ts_prefix_groups* groups, const int32_t* block_table,
                                 int32_t bt_stride, const int32_t* seq_lens, int32_t B,
                                 int32_t H_q, int32_t H_kv, int32_t D, int32_t page_size,
                                 int32_t num_pages, float scale, ts_dtype dtype, void* out,
                                 float* lse, void* workspace, size_t workspace_bytes,
                                 void* stream);

/*
 * ts_cascade_nested_decode_attn - ts_cascade_decode_attn over a forest of
 * nested shared prefixes (ts_group_prefixes_nested).
 *
 * Same result as ts_paged_decode_attn over the full block tables (up to
 * float32 rounding). Level by level, the queries of each node's members
 * attend the node's own stretch of pages as one dense tensor-core product,
 * and each member's state over its path is merged by LSE (TokenSpeed deep
 * dive, section 7.1); a prefix shared by a large set is thus computed once
 * even where subsets share longer ones. Each sequence's pages past its
 * deepest node take the paged split-KV path and are merged last.
 *
 *   forest            device copies of the arrays of ts_group_prefixes_nested
 *                     (num_nodes and num_levels as returned; capacities ignored)
 *   level_indptr_host HOST copy of forest level_indptr (num_levels + 1 entries)
 *   workspace         >= ts_cascade_decode_workspace_size(B, H_q, D)
 *   other arguments and support as ts_cascade_decode_attn.
 */
TS_API ts_status ts_cascade_nested_decode_attn(const void* q, const void* k_pool, const void* v_pool,
                                               const ts_prefix_forest* forest, const int32_t* level_indptr_host,
                                               const int32_t* block_table, int32_t bt_stride,
                                               const int32_t* seq_lens, int32_t B, int32_t H_q, int32_t H_kv,
                                               int32_t D, int32_t page_size, int32_t num_pages, float scale,
                                               ts_dtype dtype, void* out, float* lse, void* workspace,
                                               size_t workspace_bytes, void* stream);

/*
 * ts_mla_workspace_size - workspace bytes for ts_mla_paged_decode.
 */
TS_API size_t ts_mla_workspace_size(int32_t B, int32_t H, int32_t D_v);

/*
 * ts_mla_paged_decode - absorbed multi-head latent attention decode.
 *
 * Every query head attends the one shared latent head:
 *   s[h,t] = scale * <q[b,h,0:D_qk], C_b[t,0:D_qk]>,
 *   O[b,h,:] = sum_t softmax_t(s[h,:]) C_b[t,0:D_v],  LSE[b,h] = log sum_t exp(s[h,t]).
 * (TokenSpeed deep dive, section 7 fig. 3 and 7.1: split-KV partials plus a
 * reduction kernel, 512-wide output rows.)
 *
 *   q        device bf16 [B, H, D_qk]
 *   kv_pool  device bf16 [num_pages, page_size, D_qk]  (V = first D_v columns)
 *   out      device bf16 [B, H, D_v];  lse device float32 [B, H] or NULL
 * Supported: H == 128, D_qk == 576, D_v == 512, page_size 64, bf16.
 */
TS_API ts_status ts_mla_paged_decode(const void* q, const void* kv_pool, const int32_t* block_table,
                              int32_t bt_stride, const int32_t* seq_lens, int32_t B, int32_t H,
                              int32_t D_qk, int32_t D_v, int32_t page_size, int32_t num_pages,
                              float scale, void* out, float* lse, void* workspace,
                              size_t workspace_bytes, void* stream);

/*
 * ts_mla_multi_workspace_size - workspace bytes for ts_mla_paged_decode_multi
 * (B sequences of q_len query tokens, H heads). 0 on invalid or unsupported
 * arguments.
 */
TS_API size_t ts_mla_multi_workspace_size(int32_t B, int32_t q_len, int32_t H, int32_t D_v);

/*
 * ts_mla_paged_decode_multi - absorbed-MLA decode with q_len new query tokens
 * per sequence (speculative or multi-token verification).
 *
 * TokenSpeed deep dive, section 7 fig. 3 and 7.2: decode over q_seqlen query
 * tokens whose tokens are folded into the head rows of a 128-row tile,
 * F = fold_sq_factor = the largest factor of q_len with H * F <= 128, so a
 * tile holds F tokens x H heads and a sequence takes q_len / F tiles (64
 * heads, 4 tokens: F = 2, two tiles). The new tokens' latent rows are already
 * in the cache (seq_lens counts them): token j sits at position
 * L - q_len + j and attends latent rows 0 .. L - q_len + j.
 *
 *   q        device bf16 [B, q_len, H, D_qk]
 *   out      device bf16 [B, q_len, H, D_v];  lse device float32 [B, q_len, H] or NULL
 *   workspace >= ts_mla_multi_workspace_size(B, q_len, H, D_v)
 *   other arguments as ts_mla_paged_decode. A sequence with L < q_len gives
 *   O = 0 and LSE = -inf for the rows that see no key.
 * Supported: H * F == 128 (H = 128 with any q_len; 64 with even q_len; 32
 * with q_len a multiple of 4, ...), D_qk == 576, D_v == 512, page_size 64,
 * bf16; otherwise TS_ERR_UNSUPPORTED. q_len == 1 with H == 128 is
 * ts_mla_paged_decode.
 */
TS_API ts_status ts_mla_paged_decode_multi(const void* q, const void* kv_pool, const int32_t* block_table,
                                           int32_t bt_stride, const int32_t* seq_lens, int32_t B,
                                           int32_t q_len, int32_t H, int32_t D_qk, int32_t D_v,
                                           int32_t page_size, int32_t num_pages, float scale, void* out,
                                           float* lse, void* workspace, size_t workspace_bytes,
                                           void* stream);

/*
 * ts_mla_paged_decode_fp8 - absorbed-MLA decode on the fp8 input path.
 *
 * TokenSpeed deep dive, section 1: the MLA decode kernel takes bf16, fp16 or
 * fp8 inputs. Here the query rows and the cached latent rows are e4m3fn codes
 * with one float32 token-group scale per row (tokenspeed 딥다이브, section
 * 6-4: value = code * scale). The result is ts_mla_paged_decode_multi's over
 * the reconstructed rows: s[h,t] = scale * <q[h] * q_scale[h], C[t] *
 * kv_scale[t]> over all 576 columns, O = softmax(s) C[:, 0:512]. Scores run on
 * e4m3 tensor-core products (32 columns per instruction); for the product
 * with the values the softmax weights, times the token scales, are carried
 * as two e4m3 terms (hi and the remainder): relative error at most 2^-8, as
 * with bf16 weights.
 *
 *   q_codes   device uint8 [B, q_len, H, 576] (q_len = 1: [B, H, 576])
 *   q_scale   device float32 [B, q_len, H]: one scale per query row
 *   kv_codes  device uint8 [num_pages, page_size, 576]
 *   kv_scale  device float32 [num_pages, page_size], 16-byte aligned
 *   out       device bf16 [B, q_len, H, 512];  lse float32 [B, q_len, H] or NULL
 *   workspace >= ts_mla_multi_workspace_size(B, q_len, H, D_v)
 *   other arguments and support (H * fold == 128, D_qk 576, D_v 512, page 64)
 *   as ts_mla_paged_decode_multi. Rows past a sequence's end may hold any
 *   codes and scales (NaN included); they are never weighted.
 */
TS_API ts_status ts_mla_paged_decode_fp8(const void* q_codes, const float* q_scale, const void* kv_codes,
                                         const float* kv_scale, const int32_t* block_table, int32_t bt_stride,
                                         const int32_t* seq_lens, int32_t B, int32_t q_len, int32_t H,
                                         int32_t D_qk, int32_t D_v, int32_t page_size, int32_t num_pages,
                                         float scale, void* out, float* lse, void* workspace,
                                         size_t workspace_bytes, void* stream);

/*
 * ts_read_device_error - copy the sticky error word of an attention
 * workspace to *error_bits (synchronises the stream). workspace == NULL
 * reads the error word of ts_paged_decode_attn_noalloc's static scratch on
 * the current device.
 */
TS_API ts_status ts_read_device_error(const void* workspace, uint32_t* error_bits, void* stream);

/*
 * Launch trace (a measurement aid; the pages have no counterpart). While it
 * is enabled, every kernel the library launches is bracketed by two CUDA
 * events recorded on the launch's own stream, so that a caller can learn how
 * long each kernel of a call ran. Off by default; enabling it adds two event
 * records per launch and serialises launches that would otherwise overlap
 * (programmatic dependent launch), so time a step without it.
 *
 * ts_trace_enable(on): 1 = record from now on, 0 = stop recording. Process-
 *   wide; records made while on stay until collected.
 * ts_trace_collect(out, capacity): waits for every recorded launch to finish,
 *   writes up to `capacity` records in launch order (kernel name, NUL-
 *   terminated, and its device time in milliseconds) to the caller's array
 *   `out` (may be NULL to only count), forgets all records, and returns how
 *   many there were (possibly more than `capacity`), or -1 if reading an
 *   event failed (ts_last_error_detail() says which).
 */
typedef struct {
  char kernel[48];
  float ms;
} ts_launch_record;

TS_API ts_status ts_trace_enable(int32_t on);
TS_API int32_t ts_trace_collect(ts_launch_record* out, int32_t capacity);

/*
 * ts_clock_stamp - a measurement aid (the pages have no counterpart):
 * enqueues on `stream` a kernel of n CTAs whose first thread each writes
 * three uint64 values to stamps[3 i], stamps[3 i + 1], stamps[3 i + 2]: the
 * SM it ran on (%smid), that SM's cycle counter (%clock64) and the global
 * nanosecond timer (%globaltimer), read back to back. Two calls around a
 * stretch of work on the same stream give each SM's average clock over it:
 * the cycle difference over the timer difference, matched by SM. The CTAs
 * of one call usually land on distinct SMs; with n = 2 x the SM count
 * nearly every SM is covered.
 * stamps: device memory of 3 n uint64, 8-byte aligned, owned by the caller;
 * n in [1, 65535]. TS_ERR_INVALID_ARG for a null or unaligned pointer or n
 * out of range (nothing is enqueued); TS_ERR_CUDA if the launch fails.
 */
TS_API ts_status ts_clock_stamp(void* stamps, int32_t n, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* TS_ATTN_H_ */
