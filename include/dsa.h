/*
 * dsa.h - C ABI of the GB300 (sm_103a) DSA sparse MLA attention library (libdsa_gb300.so).
 *
 * What the library computes is defined by sglang PR #38547 "Enable zero-RoPE TileLang DSA on
 * gfx950":
 *   - Summary / Contract table: the 256+0 latent geometry (256-wide NoPE latent, zero-width
 *     RoPE tail; Q [tokens, 64, 256], KV [slots, 1, 256], output BF16 [tokens, 64, 256]) and
 *     the DeepSeek-style 512+64 layout kept as a control (d_v = 512, 64-wide RoPE tail);
 *   - Contract table, "scaled FP8 cache row": 264 bytes = 256 e4m3 + 2 fp32 scales + 0 RoPE,
 *     656 bytes = 512 e4m3 + 4 fp32 scales + 64 bf16 RoPE values;
 *   - Scope list: quant_k_cache (pack rows), dequant_k_cache (direct, paged, gather/dequant);
 *   - Direct GLM geometry coverage list: top-k widths 2048 / 2112, rows padded with -1, the
 *     reference computation (gather the rows, mask padding, score, softmax, weight the rows),
 *     and repeated runs that agree bit for bit.
 *
 * Conventions for every entry point:
 *   - All pointers are DEVICE pointers unless stated otherwise; the caller owns all memory.
 *     The library allocates nothing and keeps no per-call state, so calls on different
 *     streams may run concurrently when they use different output/workspace buffers.
 *   - Work is enqueued on `stream` (a cudaStream_t passed as void*; NULL = legacy default
 *     stream) and runs asynchronously. The return value reports host-side argument checks and
 *     launch errors only. Problems found on the device (an index that addresses no slot, a
 *     bounded wait that timed out) are OR-ed into the optional device word `error_word`
 *     (DSA_DEVERR_* bits), which the caller reads after synchronising.
 *   - bf16 tensors are IEEE bfloat16 bit patterns (uint16); all strides are in elements.
 *   - On error nothing is launched and no output is written.
 */
#ifndef DSA_GB300_H
#define DSA_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define DSA_API __attribute__((visibility("default")))
#else
#define DSA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DSA_OK = 0,
  DSA_ERR_INVALID_ARGUMENT = 1,   /* null pointer, negative size, bad stride or alignment */
  DSA_ERR_UNSUPPORTED = 2,        /* a geometry or head count this build has no kernel for */
  DSA_ERR_WORKSPACE_TOO_SMALL = 3,
  DSA_ERR_CUDA = 4,               /* a CUDA runtime/driver call failed (see dsa_last_cuda_error) */
  DSA_ERR_NO_DEVICE = 5           /* the current device is not an sm_103 GPU */
} dsa_status_t;

/* Bits OR-ed into the optional device error word. */
#define DSA_DEVERR_INDEX_OUT_OF_RANGE 0x1  /* an index / page addressed no slot: entry masked */
#define DSA_DEVERR_TIMEOUT 0x2             /* a bounded device-side wait gave up */
#define DSA_DEVERR_SLOT_OUT_OF_RANGE 0x4   /* quant_k_cache: out_loc outside [0, num_slots): row skipped */

typedef enum {
  DSA_CACHE_BF16 = 0,        /* bf16 latent rows [num_slots, d_nope + d_rope] */
  DSA_CACHE_FP8_SCALED = 1   /* packed rows [num_slots, dsa_packed_row_bytes(d_nope, d_rope)] uint8 */
} dsa_cache_kind_t;

/* Human-readable name of a status code (static string). */
DSA_API const char* dsa_status_string(dsa_status_t status);

/* The CUDA error code (cudaError_t as int) behind the last DSA_ERR_CUDA of this thread. */
DSA_API int dsa_last_cuda_error(void);

/* Bytes of one packed scaled-FP8 row: d_nope codes + 4 * (d_nope / 128) scale bytes +
 * 2 * d_rope RoPE bytes (Contract table: 264 for 256+0, 656 for 512+64). Returns -1 when
 * d_nope is not a positive multiple of 128 or d_rope < 0. */
DSA_API int64_t dsa_packed_row_bytes(int d_nope, int d_rope);

/* Bytes of one cache row of the given kind (bf16 rows: 2 * (d_nope + d_rope)). */
DSA_API int64_t dsa_cache_row_bytes(dsa_cache_kind_t kind, int d_nope, int d_rope);

/*
 * dsa_quant_k_cache - pack latent rows into the scaled-FP8 cache (quant_k_cache, Scope list;
 * memory_pool write sites). For row i and each 128-element tile j of its NoPE part:
 *   amax = max |x|, scale = amax / 448 (fp32), code = e4m3_rne_satfinite(x / scale) (one IEEE
 *   fp32 division per element; an all-zero tile stores scale 0 and codes 0),
 * written to slot out_loc[i] (or slot i when out_loc is NULL) as
 *   [d_nope codes][d_nope/128 fp32 scales, little endian][d_rope bf16 RoPE values, copied].
 *   k_nope        bf16 [n, d_nope], row i at k_nope + i * k_nope_row_stride (stride >= d_nope, even)
 *   k_rope        bf16 [n, d_rope], row i at k_rope + i * k_rope_row_stride; NULL iff d_rope == 0
 *   out_loc       int64 [n] destination slots, or NULL; a slot outside [0, num_slots) skips the row
 *                 and sets DSA_DEVERR_SLOT_OUT_OF_RANGE
 *   cache         uint8 [num_slots, row_bytes], 8-byte aligned base
 * Supported: d_nope in {256, 512}, d_rope in {0, 64}. n == 0 is a no-op.
 */
DSA_API dsa_status_t dsa_quant_k_cache(const void* k_nope, int64_t k_nope_row_stride, const void* k_rope,
                               int64_t k_rope_row_stride, int64_t n, int d_nope, int d_rope,
                               const int64_t* out_loc, void* cache, int64_t num_slots,
                               int32_t* error_word, void* stream);

/*
 * dsa_gather_dequant - gather latent rows by index and widen them to bf16 (dequant_k_cache:
 * direct, paged and gather/dequant paths; Contract table "paged dequant/gather").
 *   indices       int32 [n]; an entry < 0 yields a zero row
 *   block_table   int32 [R, bt_stride] physical page of each logical page, or NULL (direct mode:
 *                 the index is the slot). Paged: slot = block_table[r, i / page_size] * page_size
 *                 + i % page_size with r = req_of_index[k] (0 when req_of_index is NULL) and
 *                 i < max_pages * page_size.
 *   out           bf16 [n, d_nope + d_rope] (contiguous). FP8 rows: bf16_rne(fp32(e4m3(code)) * scale),
 *                 RoPE bits copied; BF16 rows: copied.
 * An index that addresses no slot yields a zero row and sets DSA_DEVERR_INDEX_OUT_OF_RANGE.
 */
DSA_API dsa_status_t dsa_gather_dequant(const void* cache, dsa_cache_kind_t kind, int64_t num_slots,
                                int d_nope, int d_rope, const int32_t* indices, int64_t n,
                                const int32_t* block_table, int64_t bt_stride, int page_size,
                                int max_pages, const int32_t* req_of_index, void* out,
                                int32_t* error_word, void* stream);

/*
 * dsa_gather_requant - gather packed scaled-FP8 rows by index and pack them again
 * (dequant_k_cache: the gather/dequant/requant path; PR #38547, its production-file list). Row i
 * of the result is exactly dsa_quant_k_cache applied to the bf16 row dsa_gather_dequant returns
 * for indices[i]: each gathered tile is widened to bf16_rne(fp32(e4m3(code)) * scale), then
 * re-packed (new amax, scale = amax / 448, codes = e4m3_rne_satfinite(x / scale)); RoPE bits are
 * copied. A masked index (< 0), or one that addresses no slot (which also sets
 * DSA_DEVERR_INDEX_OUT_OF_RANGE), packs the all-zero row.
 *   cache         uint8 [num_slots, row_bytes] packed rows (8-byte aligned base)
 *   indices, block_table, bt_stride, page_size, max_pages, req_of_index: as for dsa_gather_dequant
 *   out_loc       int64 [n] destination row of each result in `out`, or NULL (row i); a row
 *                 outside [0, out_slots) is skipped and sets DSA_DEVERR_SLOT_OUT_OF_RANGE
 *   out           uint8 [out_slots, row_bytes] (8-byte aligned base); may not overlap `cache`
 * Supported: d_nope in {256, 512}, d_rope in {0, 64}. n == 0 is a no-op.
 */
DSA_API dsa_status_t dsa_gather_requant(const void* cache, int64_t num_slots, int d_nope, int d_rope,
                                const int32_t* indices, int64_t n, const int32_t* block_table,
                                int64_t bt_stride, int page_size, int max_pages,
                                const int32_t* req_of_index, const int64_t* out_loc, void* out,
                                int64_t out_slots, int32_t* error_word, void* stream);

/*
 * dsa_topk_select - the top-k position list of each query token from its index-logits, the
 * input dsa_sparse_attn gathers by (FreeToken PR #270 "glm5_next: support GLM-5.3-Flash",
 * Summary, the DSA key-pooling bullet: pooled keys are scored and the best-scoring positions
 * read; PR #38547, Direct GLM geometry coverage list: top-k widths 2048 and 2112, lists padded
 * with -1). The pages give the scoring itself no formula: the scores are an input.
 *   scores        fp32 [T, S], row t at scores + t * score_stride_t (stride >= S); finite or
 *                 +-inf (NaN is outside the contract); may be NULL when S == 0
 *   lengths       int32 [T] positions each row considers (0 .. n_t - 1, n_t = lengths[t]
 *                 clamped to [0, S]: a causal limit), or NULL (n_t = S)
 *   K             result width, 1 .. 16384
 *   indices       int32 [T, K] at indices + t * idx_stride_t (stride >= K): the positions of the
 *                 min(K, n_t) largest scores of row t in descending score order, equal scores
 *                 in ascending position order (-0.0 equals +0.0), then -1 up to K
 * The result depends only on the inputs (integer decisions on order-preserving keys). T == 0 is
 * a no-op; errors: DSA_ERR_INVALID_ARGUMENT (sizes, strides, null or misaligned pointers),
 * DSA_ERR_UNSUPPORTED (S above 2^31 - 1).
 */
DSA_API dsa_status_t dsa_topk_select(const float* scores, int64_t T, int64_t S, int64_t score_stride_t,
                             const int32_t* lengths, int K, int32_t* indices, int64_t idx_stride_t,
                             void* stream);

/* Arguments of dsa_sparse_attn. Zero-initialise, then fill. */
typedef struct dsa_attn_args {
  const void* q;                 /* bf16 [T, H, d_nope + d_rope]; element (t,h,d) at
                                    q + t*q_stride_t + h*q_stride_h + d; 16-byte aligned base,
                                    strides multiples of 8 elements */
  int64_t q_stride_t, q_stride_h;
  int64_t T;                     /* query tokens (0 = no-op) */
  int H;                         /* heads: 64 */
  const void* cache;             /* BF16 rows or packed FP8 rows, see dsa_cache_kind_t */
  dsa_cache_kind_t kind;
  int64_t num_slots;
  int d_nope, d_rope, d_v;       /* (256, 0, 256) or (512, 64, 512) */
  const int32_t* indices;        /* int32 [T, topk] at indices + t*idx_stride_t; < 0 = masked */
  int64_t idx_stride_t;
  int topk;                      /* 1 .. 16384 */
  const int32_t* block_table;    /* int32 [R, bt_stride] or NULL (direct slots) */
  int64_t bt_stride;
  int page_size, max_pages;
  const int32_t* req_of_token;   /* int32 [T] request of each token, or NULL (request 0) */
  float sm_scale;                /* softmax scale applied to q.k: any finite value (0 gives the
                                    mean of the valid rows, a negative value is allowed) */
  void* out;                     /* bf16 [T, H, d_v]; (t,h,d) at out + t*out_stride_t + h*out_stride_h + d */
  int64_t out_stride_t, out_stride_h;
  float* lse;                    /* optional fp32 [T, H] natural-log sum of exp(scores); NULL ok */
  void* workspace;               /* device scratch of dsa_sparse_attn_workspace_size bytes,
                                    zero-filled before its first use. A call tags the merge flags
                                    it sets with a per-workspace counter and clears every flag it
                                    consumes before it ends, so the workspace needs no clearing
                                    between calls (zero-fill it again after a call that reported
                                    DSA_DEVERR_TIMEOUT). One call at a time per workspace. */
  size_t workspace_bytes;
  int32_t* error_word;           /* optional device int32; DSA_DEVERR_* bits are OR-ed in */
} dsa_attn_args_t;

/*
 * dsa_sparse_attn_workspace_size - bytes of workspace dsa_sparse_attn needs for these arguments
 * on the current device (depends on the device's SM count and d_v only).
 */
DSA_API dsa_status_t dsa_sparse_attn_workspace_size(const dsa_attn_args_t* args, size_t* bytes);

/*
 * dsa_sparse_attn - DSA sparse MLA attention forward (the TileLang BF16 "partial" kernel and
 * the FP8 kernel of the Scope list, re-designed for sm_103a). For every token t and head h:
 *   valid entries j: indices[t, j] >= 0 (translated through block_table in paged mode);
 *   k_j = the latent row (BF16 as stored; FP8: e4m3 code * tile scale, RoPE bf16 as stored);
 *   s_j = sm_scale * dot(q[t,h,:], k_j), p = softmax_j(s), out[t,h,:] = sum_j p_j * k_j[0:d_v];
 *   lse[t,h] = log(sum_j exp(s_j)). A token with no valid entry gets out = 0 and lse = -inf.
 * Duplicate indices are separate terms. The result is bit-identical across repeated calls with
 * the same inputs on the same device.
 * Arithmetic. BF16 rows: products of bf16 operands accumulated in fp32 (tensor cores);
 * probabilities enter the value product as bf16. 256+0 FP8 rows: 8-bit tensor-core products
 * accumulated in fp32; the e4m3 codes enter exactly, the bf16 query as two e4m3 terms per head
 * and 128-column tile (a power-of-two scale each; exact for every component within 2^9 of the
 * tile's largest), the fp32 tile scales multiply the score accumulators, and the probabilities
 * (times each key's tile scale) enter the value product as two e4m3 terms, 8 significant bits.
 * The keys are thus the exact products code * scale (never rounded to bf16). 512+64 FP8 rows:
 * keys are bf16_rne(code * scale), the rows dsa_gather_dequant returns.
 */
DSA_API dsa_status_t dsa_sparse_attn(const dsa_attn_args_t* args, void* stream);

/*
 * dsa_sparse_attn_static_ws - dsa_sparse_attn for callers that cannot allocate device memory.
 * (The pages have no counterpart: this is a deployment variant of the same computation.)
 *
 * Who needs it: callers that have no device allocator to offer, or may not use one when they
 * call: serving engines that reserve all device memory up front for their KV page pool and
 * hand libraries only input and output buffers, runtimes that work from a fixed memory plan,
 * and latency-critical paths where an allocation could stall or synchronise the device. This
 * entry point takes no workspace (args->workspace and workspace_bytes are ignored): its
 * split-token scratch lives in a fixed device array inside the library, about 10.6 MB, enough
 * for the partial results of up to 160 CTAs. Every GPU that loads the library holds that array
 * until the process exits. The call allocates nothing.
 *
 * Arguments, results and errors are those of dsa_sparse_attn; the result is identical to
 * dsa_sparse_attn's on GPUs with at most 160 SMs. On a GPU with more SMs the kernel runs on 160
 * CTAs; if the array could not hold the scratch of the launch the call returns
 * DSA_ERR_WORKSPACE_TOO_SMALL without launching.
 *
 * The first call on each device does one-time set-up: it looks up the array's device address
 * (cudaGetSymbolAddress) and sets the attention kernels' shared-memory limits on that device.
 * All calls share the one array,
 * which keeps what the last call left there: a call tags the flags it sets with a fresh value
 * and clears every flag it consumes, so nothing has to be cleared between calls. Two calls
 * whose kernels overlap on the GPU (different streams, no ordering between them) race on the
 * array: order such calls, or use dsa_sparse_attn with separate workspaces.
 */
DSA_API dsa_status_t dsa_sparse_attn_static_ws(const dsa_attn_args_t* args, void* stream);

/*
 * FP8 block-scaled projection GEMM, for the dense MLA projections around the attention
 * (sglang PR #31955 "Opt-in prefill-only FP8 dense projection GEMM for MLA q_b/o_proj",
 * Motivation and Modifications: weights repacked into e4m3 with one UE8M0 (power-of-two) scale
 * per 128x128 block, activations quantised per token and 128-column group, "a8w8 blockscale").
 *
 * dsa_blockscale_bytes - bytes of the scale tensor of a [rows, cols] matrix (cols a multiple of
 * 128): ceil(rows / 128) * (cols / 128) * 512; -1 for invalid sizes.
 *
 * dsa_quant_fp8_blockscale - quantise bf16 x [rows, cols] (row stride in elements, a multiple
 * of 8; cols a multiple of 128) into e4m3 codes [rows, cols] (uint8, contiguous) and scales.
 * block_rows = 128 (weights: 128 x 128 blocks) or 1 (activations: 1 x 128 blocks). Per block,
 * e = the smallest integer in [-127, 127] with 448 * 2^e >= max |x| (0 for an all-zero block) and
 * code = e4m3 round-to-nearest-even of x / 2^e (exact; nothing saturates). The UE8M0 bytes e + 127
 * are stored in the GEMM's 32-element block-scale layout: each 128-column block is four equal
 * 32-column scales; tiles of 128 rows x 4 scale columns (512 bytes; row r, scale column c at
 * (r % 32) * 16 + ((r % 128) / 32) * 4 + c % 4) in row-tile-major order. Scales of rows past
 * `rows` in the last tile read 127 (scale 1). Inputs must be finite. Pointers 16-byte aligned.
 *
 * dsa_proj_gemm - y[m, n] = sum_k x[m, k] w[n, k] over the dequantised operands (x from
 * block_rows = 1, w [N, K] from block_rows = 128), fp32 accumulation, bf16 output y [M, N] with
 * row stride y_stride (elements, a multiple of 8). N and K multiples of 128. The product runs in
 * cuBLASLt (e4m3 operands with 32-element UE8M0 block scales); `workspace` (256-byte aligned,
 * may be NULL with workspace_bytes 0) is its scratch. Calls on one device are serialised on the
 * host (the library keeps one cuBLASLt handle and a plan cache per device).
 */
DSA_API int64_t dsa_blockscale_bytes(int64_t rows, int64_t cols);
DSA_API dsa_status_t dsa_quant_fp8_blockscale(const void* x, int64_t rows, int64_t cols, int64_t row_stride,
                                              int block_rows, void* codes, void* scales, void* stream);
DSA_API dsa_status_t dsa_proj_gemm(const void* x_codes, const void* x_scales, const void* w_codes,
                                   const void* w_scales, int64_t M, int64_t N, int64_t K, void* y, int64_t y_stride,
                                   void* workspace, size_t workspace_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DSA_GB300_H */
