// dsa_attn_f8.cu - DSA sparse MLA attention forward over the packed scaled-FP8 cache of the
// 256+0 latent geometry on sm_103a, with 8-bit operands on the tensor core.
//
// What is computed (sglang PR #38547 "Enable zero-RoPE TileLang DSA on gfx950", Summary,
// Contract table row "scaled FP8 cache row" and Direct GLM geometry coverage list): for every
// query token t and head h, gather the 264-byte rows named by t's top-k list (entries < 0
// masked), dequantise k = code * scale (one fp32 scale per 128-column tile), score
// s_j = sm_scale * q[t,h].k_j, softmax over j and return sum_j p_j * k_j (all 256 columns) in
// bf16, with the natural-log sum of exp(s_j) as an optional second output.
//
// Kernel design (GB300-first; the pages' TileLang/HIP kernels are prior art):
//  * The gathered K tile stays 8-bit in shared memory: 128 keys x 256 e4m3 codes (32 KB), one
//    128-byte swizzled chunk per scale tile. Loader warps only issue cp.async copies of each
//    row's codes and scales into it (16-byte copies for rows that start 16-byte aligned, 8-byte
//    copies for the others); three stages keep about 66 KB of rows in flight per SM.
//  * Scores S^T = K Q^T (M = 128 keys, N = 64 heads) run as tcgen05 kind::f8f6f4. The bf16
//    query of each head is split exactly into two e4m3 terms per 128-column tile,
//    q = 2^e (hi + lo) with e a power of two per head and tile (hi keeps the top four
//    significant bits, lo the other four), and both terms accumulate into the same fp32
//    accumulator, one per scale tile (S_0, S_1). The softmax warps make the split of each
//    token's query at the end of the previous token, before its epilogue, so that the next
//    token's score products can start while they finish the previous token.
//  * Softmax per key (thread = TMEM lane). Each row's two scales and the query factors 2^e
//    are applied in fp32 to the accumulators: x = c * (sc0 2^e0_h S_0 + sc1 2^e1_h S_1),
//    c = sm_scale * log2(e). Three running maxima per head: m of x, for the row sums of
//    p = 2^(x - m), and m'_t of x + log2 sc_t, the reference of output half t (columns
//    128t .. 128t + 127, scale tile t). The weights of the output product,
//    P_t = p * sc_t * 2^(m - m'_t + 4) = 2^(x + log2 sc_t - m'_t + 4), are proportional to the
//    size of each key's contribution to that half, so they stay in e4m3 range (below 2^8.5)
//    whatever the scales are, with the largest near 2^4. P_t is written as two e4m3 terms
//    (hi: P_t truncated to four significant bits, lo: the rest rounded), 8 significant bits in
//    all, each key's two 64-head rows side by side (128 bytes per key and half). Two P buffers,
//    so that the pass of tile g + 1 runs while the output product of tile g reads its P.
//  * Output O^T += V^T P^T in two M = 128 halves of d_v (V^T read MN-major from the same 8-bit
//    tile, one half per scale tile), N = 64 heads, the hi and lo terms of P into the same
//    accumulator. Half t is normalised by 2^(m'_t - m - 4) / l at the token's end.
//  * Persistent cooperative launch, one CTA per SM; (token, 128-position tile) units split into
//    contiguous ranges per CTA; a token cut by a range boundary is merged in-kernel by the CTA
//    holding its first tiles: the other parts' partial results come into idle shared memory by
//    bulk copies (two in flight) and are added, in a fixed order, into its O columns of tensor
//    memory (no atomics on data).
//  * Warp roles: 0 producer (index read, -1 compaction into dense 128-key tiles, page
//    translation), 1 score-MMA issuer, 2 output-MMA issuer, 4-11 softmax, query split and
//    epilogue (two warps per TMEM lane quarter, 32 heads each), 3 and 12-15 row loaders (which
//    also pull the next token's query into L2 at each token end).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "dsa_attn_common.h"
#include "dsa_host.h"
#include "dsa_ptx.cuh"

namespace dsa {
namespace f8 {

constexpr int kH = kAttnHeads;  // heads: MMA N
constexpr int kD = 256;         // latent width (= d_v)
constexpr int kRB = 264;        // packed row bytes
constexpr int kBN = 128;        // gathered keys per tile: MMA M
constexpr int kKST = 3;         // K tile stages
constexpr int kMST = 8;         // meta ring depth
constexpr int kWarps = 16;
constexpr int kThreads = 32 * kWarps;
constexpr int kNSM = 8;         // softmax warps 4-11 (two per TMEM lane quarter, 32 heads each)
constexpr int kNLD = 5;         // loader warps 3, 12-15
constexpr int kPBUF = 2;        // P buffers
constexpr int kMaxParts = 16;   // most parts of one split token (the launch guarantees it)
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr int kSplitMaxCtas = 192;
constexpr float kTau = 4.5f;     // lazy maxima of the output halves: a tile may exceed them by 2^4.5
constexpr float kTauL = 20.0f;   // lazy maximum of the row sums (fp32 sums: a wide margin is safe)
constexpr int kPShift = 4;       // P weights carry an extra 2^4: the largest is about 2^4 ...
constexpr float kPMax = 400.0f;  // ... and at most 2^(4.5 + 4) = 362 (with margin; e4m3 tops at 448)

// shared memory carve-up (offsets from a 1024-aligned base)
constexpr int Q_OFF = 0;                // Q: [hi chunk 0 | hi chunk 1 | lo 0 | lo 1], 8 KB each
constexpr int Q_BYTES = 2 * kH * kD;    // 32 KB
constexpr int KT_OFF = Q_OFF + Q_BYTES;
constexpr int KT_BYTES = kBN * kD;      // 32 KB: chunk c (columns 128c..) at c * 16 KB
constexpr int P_OFF = KT_OFF + kKST * KT_BYTES;
constexpr int P_BYTES = 2 * kBN * 128;  // per buffer: P_t at t * 16 KB, per key 128 B = [64 hi | 64 lo]
constexpr int SC_OFF = P_OFF + kPBUF * P_BYTES;
constexpr int SC_BYTES = kBN * 8;       // per stage: (scale0, scale1) per row
constexpr int SQ_OFF = SC_OFF + kKST * SC_BYTES;  // per column tile: c * 2^e of each head
constexpr int META_OFF = SQ_OFF + 2 * kH * 4;
constexpr int META_HDR = 48;
constexpr int META_BYTES = META_HDR + 4 * kBN;
constexpr int CMP_OFF = META_OFF + kMST * META_BYTES;
constexpr int RED_OFF = CMP_OFF + 4 * 256;
// m[64], m'[2][64], r[64][2], alpha[3][64], part[3][4][64], wk[2][kMaxParts][64], votes[2][kNSM], -m[64]
constexpr int RED_FLOATS = 20 * kH + 2 * kMaxParts * kH + 2 * kNSM + kH;
constexpr int SPLIT_OFF = RED_OFF + ((RED_FLOATS * 4 + 15) & ~15);
constexpr int BAR_OFF = SPLIT_OFF + 8 * (kSplitMaxCtas + 1);
// barrier indices
enum : int {
  B_QFULL = 0, B_QEMPTY = 1, B_KFULL = 2, B_KEMPTY = B_KFULL + kKST, B_MFULL = B_KEMPTY + kKST,
  B_MEMPTY = B_MFULL + kMST, B_SFULL = B_MEMPTY + kMST, B_SEMPTY = B_SFULL + 2, B_PFULL = B_SEMPTY + 2,
  B_PVDONE = B_PFULL + kPBUF, B_XBAR = B_PVDONE + 2, B_DRAIN = B_XBAR + 1, B_RANGE = B_DRAIN + 2, B_MERGE = B_RANGE + 1,
  NBARS = B_MERGE + 3
};
constexpr int MISC_OFF = BAR_OFF + 8 * NBARS;
constexpr int SMEM_BYTES = MISC_OFF + 32 + 1024;  // + alignment slack
// tensor memory columns
constexpr int S_COLS = 128;             // per S buffer (two): S_0 at +0, S_1 at +64
constexpr int O_COL = 2 * S_COLS;       // O^T halves: dv 0-127 at O_COL, dv 128-255 at O_COL + 64
constexpr int L_COL = O_COL + 128;      // per-lane partial row sums, two buffers of 64 columns
constexpr int TMEM_COLS = 512;
static_assert(L_COL + 128 <= TMEM_COLS, "TMEM budget");
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(KT_OFF % 1024 == 0 && P_OFF % 1024 == 0 && KT_BYTES % 1024 == 0 && P_BYTES % 1024 == 0,
              "operand alignment");
static_assert(kNSM <= 8, "one publish flag per softmax warp, eight per CTA");

enum : int { kTile = 1, kSegEnd = 2, kDone = 3 };
enum : int { kComplete = 0, kHead = 1, kPart = 2 };

struct MetaHdr {
  int type;
  int token;
  int n_valid;     // kTile: valid rows in this tile
  int first;       // kTile: first non-empty tile of its segment
  int kind;        // kSegEnd: segment kind
  int had_tiles;   // kSegEnd: the segment had at least one non-empty tile
  int merge_last;  // kSegEnd: last CTA holding a part of this token
  int seg;         // index of the segment within this CTA's range
  int next_token;  // kSegEnd: token of the CTA's next segment, -1 at the end of its range
  int pad[3];
};
static_assert(sizeof(MetaHdr) == META_HDR, "meta header size");

struct Params {
  const uint8_t* cache;
  int64_t num_slots;
  const uint16_t* q;
  int64_t q_st, q_sh;
  const int32_t* idx;
  int64_t idx_stride;
  int topk;
  const int32_t* bt;
  int64_t bt_stride;
  int page_size;
  int max_pages;
  uint32_t pg_mul;  // x / page_size == (x * pg_mul) >> pg_shift for 0 <= x < 2^31
  int pg_shift;
  const int32_t* req;
  float c_log2;  // sm_scale * log2(e)
  uint16_t* out;
  int64_t out_st, out_sh;
  float* lse;
  float* ws_o;   // [G][256 dv][64 heads] partial O^T (half t relative to 2^(m'_t - kPShift))
  float* ws_ml;  // [G][4][64] partial max m, row sum, and the output halves' maxima m'_0, m'_1
  int* flags;    // [G][8] partial published (holds the call's tag), one per softmax warp
  int epoch;
  int32_t* err;
  int64_t T;
  int NT;
  int64_t U;
  int G;
  const int64_t* bounds;
  int split_gap;
};

__device__ __forceinline__ void set_err(int32_t* err, int bits) {
  if (err) atomicOr(err, bits);
}
__device__ __forceinline__ int64_t unit_begin(int64_t b, int64_t U, int G) { return (b * U) / G; }
__device__ __forceinline__ float u2f(uint32_t u) { return __uint_as_float(u); }
__device__ __forceinline__ uint32_t f2u(float f) { return __float_as_uint(f); }

// floor(log2(w)) of a finite w > 0 (normal or subnormal), from its bits
__device__ __forceinline__ int ilog2f(float w) {
  const uint32_t b = __float_as_uint(w);
  return b >= 0x800000u ? (int)(b >> 23) - 127 : (31 - __clz((int)b)) - 149;
}
// 2^k for an integer k in [-126, 127]
__device__ __forceinline__ float pow2i(int k) { return __uint_as_float((uint32_t)(k + 127) << 23); }

// v truncated to its four leading significant bits (sign and exponent kept): exactly an e4m3
// value for 2^-6 <= |v| <= 448
__device__ __forceinline__ float trunc4(float v) { return __uint_as_float(__float_as_uint(v) & 0xFFF00000u); }

// Four values as two e4m3 terms each: hi codes (v truncated) and lo codes (v - hi rounded),
// packed low byte first.
__device__ __forceinline__ void split4(float a, float b, float c, float d, uint32_t& hi, uint32_t& lo) {
  const float ha = trunc4(a), hb = trunc4(b), hc = trunc4(c), hd = trunc4(d);
  hi = (uint32_t)f32x2_to_e4m3x2(ha, hb) | ((uint32_t)f32x2_to_e4m3x2(hc, hd) << 16);
  lo = (uint32_t)f32x2_to_e4m3x2(a - ha, b - hb) | ((uint32_t)f32x2_to_e4m3x2(c - hc, d - hd) << 16);
}

// Exchange among the softmax warps (one arrival each on `xbar`, phase `n` of it; `sm` is the
// warp's softmax index): returns the OR of `v` over the warps, with every warp's earlier
// shared-memory writes visible, or -1 when a warp did not arrive within the time limit.
static __device__ __noinline__ int softmax_exchange(uint32_t xbar, int* votes, uint32_t n, int sm, int v) {
  const int lane = threadIdx.x & 31;
  const int slot = n & 1;
  const bool any = __any_sync(0xffffffffu, v != 0);
  if (lane == 0) votes[slot * kNSM + sm] = any ? 1 : 0;
  __syncwarp();
  if (lane == 0) mbar_arrive(xbar);
  const bool ok = mbar_wait(xbar, n & 1, kWaitNs);
  if (!__all_sync(0xffffffffu, ok)) return -1;
  int r = 0;
#pragma unroll
  for (int w = 0; w < kNSM; ++w) r |= votes[slot * kNSM + w];
  return r ? 1 : 0;
}

// Splits the query of token t for the score products (warp sm of the softmax warps takes heads
// 8 sm .. 8 sm + 7; lane l columns 8l .. 8l + 7, lanes 0-15 in tile 0 and 16-31 in tile 1): per
// head and 128-column tile, e = the binary exponent of the tile's largest |q| minus 7,
// x = q * 2^-e (exact), hi = x truncated to four significant bits and lo = x - hi (the other
// four: exact for every component within 2^9 of the tile's largest); the terms go to the K-major
// 128-byte-swizzled Q operand (rows = heads) and c * 2^e to sq[head][tile].
static __device__ __forceinline__ void split_query(const Params& p, int64_t t, uint8_t* qbuf, float* sq, int sm,
                                                   int lane) {
  const uint16_t* qrow = p.q + t * p.q_st + 8 * lane;
  const int c = lane >> 4, gq = (lane & 15) >> 1, half = lane & 1;
  uint4 v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __ldg(reinterpret_cast<const uint4*>(qrow + (8 * sm + i) * p.q_sh));
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int h = 8 * sm + i;
    const uint32_t wd[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
    float f[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      f[2 * j] = u2f(wd[j] << 16);
      f[2 * j + 1] = u2f(wd[j] & 0xFFFF0000u);
    }
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(f[j]));
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    int e = amax > 0.0f ? ilog2f(amax) - 7 : 0;
    e = e < -120 ? -120 : (e > 120 ? 120 : e);
    const float inv = pow2i(-e);
#pragma unroll
    for (int j = 0; j < 8; ++j) f[j] *= inv;
    uint32_t h0, l0, h1, l1;
    split4(f[0], f[1], f[2], f[3], h0, l0);
    split4(f[4], f[5], f[6], f[7], h1, l1);
    const int off = c * (kH * 128) + h * 128 + ((gq ^ (h & 7)) << 4) + 8 * half;
    *reinterpret_cast<uint2*>(qbuf + off) = make_uint2(h0, h1);
    *reinterpret_cast<uint2*>(qbuf + 2 * kH * 128 + off) = make_uint2(l0, l1);
    if ((lane & 15) == 0) sq[2 * h + c] = pow2i(e) * p.c_log2;
  }
}

__global__ void __launch_bounds__(kThreads, 1) attn_f8_kernel(const __grid_constant__ Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const uint32_t bar0 = sbase + BAR_OFF;
  auto bar = [&](int i) { return bar0 + 8 * i; };
  const uint32_t q_full = bar(B_QFULL), q_empty = bar(B_QEMPTY);
  auto k_full = [&](int s) { return bar(B_KFULL + s); };
  auto k_empty = [&](int s) { return bar(B_KEMPTY + s); };
  auto m_full = [&](int s) { return bar(B_MFULL + s); };
  auto m_empty = [&](int s) { return bar(B_MEMPTY + s); };
  auto s_full = [&](int i) { return bar(B_SFULL + i); };
  auto s_empty = [&](int i) { return bar(B_SEMPTY + i); };
  auto p_full = [&](int i) { return bar(B_PFULL + i); };
  auto pv_done = [&](int i) { return bar(B_PVDONE + i); };
  const uint32_t xbar = bar(B_XBAR);        // softmax-warp exchange
  const uint32_t mma_drain = bar(B_DRAIN);  // every MMA of an issuer complete (+0: scores, +8: output)
  const uint32_t range_ready = bar(B_RANGE);
  // a head's merge: the other parts' (m, l, m'_0, m'_1) rows (+0) and their O^T halves, two
  // parts in flight (+1, +2)
  auto merge_bar = [&](int i) { return bar(B_MERGE + i); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + MISC_OFF + 4);
  int64_t* range = reinterpret_cast<int64_t*>(smem + MISC_OFF + 8);  // this CTA's units [u0, u1)
  float* sq = reinterpret_cast<float*>(smem + SQ_OFF);                 // [64][2 tiles] c * 2^e

  if (threadIdx.x == 0) {
    // Q: one split per segment, in order; the score issuer releases it per segment
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int s = 0; s < kKST; ++s) {
      mbar_init(k_full(s), 32 * kNLD);  // one cp.async arrive per loader thread
      mbar_init(k_empty(s), 1);
    }
    for (int s = 0; s < kMST; ++s) {
      mbar_init(m_full(s), 1);
      mbar_init(m_empty(s), 2 + kNSM + kNLD);  // 2 MMA threads, softmax warps, loader warps
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(s_full(i), 1);
      mbar_init(s_empty(i), kNSM);
      mbar_init(p_full(i), kNSM);
      mbar_init(pv_done(i), 1);
    }
    mbar_init(xbar, kNSM);
    mbar_init(mma_drain, 1);
    mbar_init(mma_drain + 8, 1);
    mbar_init(range_ready, 1);
    for (int i = 0; i < 3; ++i) mbar_init(merge_bar(i), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int b = blockIdx.x;

  auto fail = [&](int bits) {
    set_err(p.err, bits);
    *abort_flag = 1;
  };
  auto wait = [&](uint32_t bar, uint32_t par) -> bool {
    if (mbar_wait(bar, par, kWaitNs)) return true;
    fail(DSA_DEVERR_TIMEOUT);
    return false;
  };
  // L2 prefetch of token t's query rows (64 heads x 512 bytes), one warp
  auto prefetch_q = [&](int64_t t) {
    const uint16_t* qt = p.q + t * p.q_st;
    for (int i = lane; i < kH * 4; i += 32)
      asm volatile("prefetch.global.L2 [%0];" ::"l"(qt + (i >> 2) * p.q_sh + 64 * (i & 3)));
  };

  if (warp == 0) {
    // =========================================================== producer (one warp) ====
    // Walks this CTA's unit range segment by segment (one segment per token). The index window
    // of a segment is read 256 entries per step (two steps ahead, block-table rows one step
    // ahead); entries < 0 are dropped and the valid ones packed, in index order, into dense
    // 128-key tiles, so runs of padding cost only their index reads.
    uint32_t mc = 0;
    int64_t* sb = reinterpret_cast<int64_t*>(smem + SPLIT_OFF);
    if (p.bounds) {
      // a work-balanced split: bounds spaced to at least split_gap units by a running maximum
      // of bounds[c] - c * gap, capped at U - (G - c) * gap
      const int64_t gap = p.split_gap;
      constexpr int kPer = (kSplitMaxCtas + 32) / 32;
      int64_t v[kPer];
      int64_t run = INT64_MIN;
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const int c = kPer * lane + i;
        v[i] = c <= p.G ? p.bounds[c] - c * gap : INT64_MIN;
        run = v[i] > run ? v[i] : run;
        v[i] = run;
      }
      int64_t pre = INT64_MIN;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int64_t x = __shfl_up_sync(0xffffffffu, run, o);
        if (lane >= o) run = x > run ? x : run;
      }
      pre = __shfl_up_sync(0xffffffffu, run, 1);
      if (lane == 0) pre = INT64_MIN;
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const int c = kPer * lane + i;
        if (c <= p.G) {
          const int64_t lo = (v[i] > pre ? v[i] : pre) + c * gap, hi = p.U - (int64_t)(p.G - c) * gap;
          sb[c] = c == 0 ? 0 : (c == p.G ? p.U : (lo < hi ? lo : hi));
        }
      }
      __syncwarp();
    }
    const int64_t u0 = p.bounds ? sb[b] : unit_begin(b, p.U, p.G);
    const int64_t u1 = p.bounds ? sb[b + 1] : unit_begin(b + 1, p.U, p.G);
    if (lane == 0) {
      range[0] = u0;
      range[1] = u1;
      mbar_arrive(range_ready);  // the softmax warps split the first segment's query at once
    }
    auto emit_begin = [&](int& st) -> MetaHdr* {
      st = mc % kMST;
      if (mc >= (uint32_t)kMST) wait(m_empty(st), ((mc / kMST) & 1) ^ 1);
      return reinterpret_cast<MetaHdr*>(smem + META_OFF + st * META_BYTES);
    };
    auto emit_end = [&](int st) {
      __syncwarp();
      if (lane == 0) mbar_arrive(m_full(st));
      ++mc;
    };
    const int64_t pos_limit = p.bt ? (int64_t)p.max_pages * p.page_size : p.num_slots;
    int64_t u = u0;
    int64_t t = u0 / p.NT;
    int j0 = (int)(u0 - t * p.NT);
    int seg = 0;
    while (u < u1 && !*abort_flag) {
      const int j1 = (int)((int64_t)(p.NT - j0) < u1 - u ? p.NT : j0 + (u1 - u));
      const int64_t uend = u + (j1 - j0);
      const int kind = j0 > 0 ? kPart : (j1 < p.NT ? kHead : kComplete);
      const int64_t req = p.req ? p.req[t] : 0;
      const int32_t* irow = p.idx + t * p.idx_stride;
      const int32_t* btrow = p.bt ? p.bt + req * p.bt_stride : nullptr;
      const int e0 = j0 * kBN, e1 = min(j1 * kBN, p.topk);
      {  // pull this segment's index window and the request's block-table row into L2
        const uintptr_t a0 = reinterpret_cast<uintptr_t>(irow + e0) & ~uintptr_t(127);
        const uintptr_t a1 = reinterpret_cast<uintptr_t>(irow + e1);
        for (uintptr_t a = a0 + 128 * lane; a < a1; a += 32 * 128) asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
        if (btrow) {
          const uintptr_t c0 = reinterpret_cast<uintptr_t>(btrow) & ~uintptr_t(127);
          const uintptr_t c1 = reinterpret_cast<uintptr_t>(btrow + p.max_pages);
          for (uintptr_t a = c0 + 128 * lane; a < c1; a += 32 * 128) asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
        }
      }
      constexpr int V = 4;
      auto load_step = [&](int pos, int (&v)[V]) {
#pragma unroll
        for (int k = 0; k < V; ++k) {
          const int e = pos + 32 * k + lane;
          v[k] = e < e1 ? __ldg(irow + e) : -1;
        }
      };
      auto page_of = [&](const int (&x)[V], int (&pg)[V]) {
#pragma unroll
        for (int k = 0; k < V; ++k) {
          if (x[k] < 0) pg[k] = -1;
          else if (x[k] >= pos_limit) pg[k] = -2;
          else pg[k] = btrow ? __ldg(btrow + (int)(((uint64_t)(uint32_t)x[k] * p.pg_mul) >> p.pg_shift)) : x[k];
        }
      };
      int ia[V], ib[V], pa[V];
      load_step(e0, ia);
      load_step(e0 + 32 * V, ib);
      page_of(ia, pa);
      bool had = false, open = false;
      int cnt = 0, st = 0;
      int* slots = nullptr;
      MetaHdr* mh = nullptr;
      auto open_tile = [&]() {
        mh = emit_begin(st);
        slots = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(mh) + META_HDR);
        if (lane == 0) {
          mh->type = kTile;
          mh->token = (int)t;
          mh->first = had ? 0 : 1;
          mh->seg = seg;
        }
        had = true;
        open = true;
        cnt = 0;
      };
      auto close_tile = [&](int n) {
        if (lane == 0) mh->n_valid = n;
        emit_end(st);
        open = false;
      };
      int* cbuf = reinterpret_cast<int*>(smem + CMP_OFF);
      for (int pos = e0; pos < e1 && !*abort_flag; pos += 32 * V) {
        int ic[V], pb[V];
        load_step(pos + 64 * V, ic);
        page_of(ib, pb);
        int bad = 0, nstep = 0;
#pragma unroll
        for (int k = 0; k < V; ++k) {
          int64_t slot = -1;
          if (pa[k] >= 0) {
            if (btrow) {
              const int pq = (int)(((uint64_t)(uint32_t)ia[k] * p.pg_mul) >> p.pg_shift);
              slot = (int64_t)pa[k] * p.page_size + (ia[k] - pq * p.page_size);
              if (slot >= p.num_slots) slot = -2;
            } else {
              slot = pa[k];
            }
          } else if (pa[k] == -2 || (btrow && ia[k] >= 0)) {
            slot = -2;  // outside the addressable range, or a negative block-table page
          }
          bad |= (slot == -2);
          const bool ok = slot >= 0;
          const uint32_t bal = __ballot_sync(0xffffffffu, ok);
          if (ok) cbuf[nstep + __popc(bal & ((1u << lane) - 1u))] = (int)slot;
          nstep += __popc(bal);
        }
        if (bad) set_err(p.err, DSA_DEVERR_INDEX_OUT_OF_RANGE);
        __syncwarp();
        for (int c = 0; c < nstep;) {
          if (!open) open_tile();
          const int take = min(kBN - cnt, nstep - c);
          for (int i = lane; i < take; i += 32) slots[cnt + i] = cbuf[c + i];
          cnt += take;
          c += take;
          if (cnt == kBN) close_tile(kBN);
        }
        __syncwarp();
#pragma unroll
        for (int k = 0; k < V; ++k) {
          ia[k] = ib[k];
          ib[k] = ic[k];
          pa[k] = pb[k];
        }
      }
      if (open) close_tile(cnt);
      {
        int st2;
        MetaHdr* me = emit_begin(st2);
        if (lane == 0) {
          me->type = kSegEnd;
          me->token = (int)t;
          me->kind = kind;
          me->had_tiles = had ? 1 : 0;
          me->seg = seg;
          me->next_token = uend < u1 ? (int)(t + 1) : -1;
          int last = b;
          if (kind == kHead) {
            // the last CTA c whose range starts at or before the token's last unit
            const int64_t L1 = (t + 1) * p.NT;
            if (p.bounds) {
              int lo = b, hi = p.G - 1;
              while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (sb[mid] <= L1 - 1) lo = mid;
                else hi = mid - 1;
              }
              last = lo;
            } else {
              const int64_t c = (L1 * p.G + p.U - 1) / p.U - 1;
              last = (int)(c < p.G - 1 ? c : p.G - 1);
            }
          }
          me->merge_last = last;
        }
        emit_end(st2);
      }
      u = uend;
      ++t;
      ++seg;
      j0 = 0;
    }
    {
      int st;
      MetaHdr* mh = emit_begin(st);
      if (lane == 0) mh->type = kDone;
      emit_end(st);
    }
  } else if (warp == 1 || warp == 2) {
    // ======================================================= MMA issuers (2 threads) ====
    // Warp 1 issues the score products, warp 2 the output products; each is a blocking loop
    // over the meta ring. Every MMA is straight-line code with one 32-bit add per descriptor.
    if (lane == 0) {
      constexpr uint32_t idS = idesc_e4m3(128, kH, 0, 0);   // A = K tile (K-major), B = Q term (K-major)
      constexpr uint32_t idPV = idesc_e4m3(128, kH, 1, 1);  // A = V^T (MN-major), B = P^T term (MN-major)
      const uint32_t k_hi = (uint32_t)(sw128_desc(0, 16, 1024) >> 32);
      const uint32_t mn_hi = (uint32_t)(sw128_desc(0, 16384, 1024) >> 32);
      const uint32_t q_lo = (uint32_t)sw128_desc(sbase + Q_OFF, 16, 1024);
      uint32_t mc = 0, g = 0;
      for (;;) {
        const int st = mc % kMST;
        if (!wait(m_full(st), (mc / kMST) & 1)) break;
        const MetaHdr* mh = reinterpret_cast<const MetaHdr*>(smem + META_OFF + st * META_BYTES);
        const int type = mh->type;
        const int first = mh->first, had = mh->had_tiles, seg = mh->seg;
        mbar_arrive(m_empty(st));
        ++mc;
        if (type == kDone) break;
        if (type == kSegEnd) {
          // the segment's score products are issued: Q is free for the next split once they
          // complete (a segment without tiles still takes its split's phase)
          if (warp == 1) {
            if (had) {
              mma_commit(q_empty);
            } else {
              if (!wait(q_full, seg & 1)) break;
              mbar_arrive(q_empty);
            }
          }
          continue;
        }
        const int ks = g % kKST;
        if (warp == 1) {
          // ---- scores S^T = K Q^T for tile g: per scale tile t, four K-steps of 32 columns,
          // each the product with Q's hi term then its lo term into the same accumulator
          if (first && !wait(q_full, seg & 1)) break;
          if (g >= 2 && !wait(s_empty(g & 1), ((g >> 1) & 1) ^ 1)) break;
          if (!wait(k_full(ks), (g / kKST) & 1)) break;
          // rows arrive by cp.async (generic proxy): order them before the tensor core reads
          fence_proxy_async_smem();
          tc_fence_after();
          const uint32_t k_lo = (uint32_t)sw128_desc(sbase + KT_OFF + ks * KT_BYTES, 16, 1024);
          const uint32_t d0 = tmem + (g & 1) * S_COLS;
#pragma unroll
          for (int t = 0; t < 2; ++t) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint32_t ka = k_lo + (uint32_t)((t * (kBN * 128) + 32 * kk) >> 4);
              const uint32_t qa = q_lo + (uint32_t)((t * (kH * 128) + 32 * kk) >> 4);
              if (kk == 0) mma_f8_lohi<0>(d0 + 64 * t, ka, k_hi, qa, k_hi, idS);
              else mma_f8_lohi<1>(d0 + 64 * t, ka, k_hi, qa, k_hi, idS);
              mma_f8_lohi<1>(d0 + 64 * t, ka, k_hi, qa + ((2 * kH * 128) >> 4), k_hi, idS);
            }
          }
          mma_commit(s_full(g & 1));
        } else {
          // ---- output O^T += V^T P^T for tile g once its probabilities are written: half h of
          // d_v (scale tile h) takes P_h, hi term then lo term (64 bytes further in each row)
          if (!wait(p_full(g & 1), (g >> 1) & 1)) break;
          tc_fence_after();
          const uint32_t v_lo = (uint32_t)sw128_desc(sbase + KT_OFF + ks * KT_BYTES, 16384, 1024);
          const uint32_t p_lo = (uint32_t)sw128_desc(sbase + P_OFF + (g & 1) * P_BYTES, 16384, 1024);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t d = tmem + O_COL + 64 * h;
            const uint32_t va = v_lo + (uint32_t)((h * (kBN * 128)) >> 4);
            const uint32_t pa = p_lo + (uint32_t)((h * (kBN * 128)) >> 4);
            mma_f8_lohi_rt(d, va, mn_hi, pa, mn_hi, idPV, first ? 0u : 1u);
            mma_f8_lohi<1>(d, va, mn_hi, pa + (64 >> 4), mn_hi, idPV);
#pragma unroll
            for (int kk = 1; kk < kBN / 32; ++kk) {
              mma_f8_lohi<1>(d, va + ((4096 * kk) >> 4), mn_hi, pa + ((4096 * kk) >> 4), mn_hi, idPV);
              mma_f8_lohi<1>(d, va + ((4096 * kk) >> 4), mn_hi, pa + ((4096 * kk + 64) >> 4), mn_hi, idPV);
            }
          }
          mma_commit(k_empty(ks));
          mma_commit(pv_done(g & 1));
        }
        ++g;
      }
      const uint32_t drain = warp == 1 ? mma_drain : mma_drain + 8;
      mma_commit(drain);
      mbar_wait(drain, 0, kWaitNs);
    }
    __syncwarp();
  } else if (warp >= 4 && warp < 4 + kNSM) {
    // =================================== softmax, query split and epilogue (8 warps) ====
    // Thread = key of the tile = TMEM lane (quarter qd = warp % 4); the two warps of a quarter
    // take heads 0-31 and 32-63, in two 16-head chunks. Three running maxima per head: m (of x,
    // for the row sums) and m'_t (of x + log2 sc_t, the reference of output half t). Per tile
    // one pass computes p = 2^(x - m), the per-lane partial row sums (TMEM, two buffers: the pass
    // reads one and writes the other) and P_t = p * sc_t * r_t with r_t = 2^(m - m'_t + kPShift),
    // i.e. P_t = 2^(x + log2 sc_t - m'_t + kPShift), as e4m3 hi/lo terms. A vote then checks
    // that no P_t exceeded kPMax and no x - m exceeded kTauL; if one did (rare after a segment's
    // first tile), the tile takes the exact path: per-head maxima of x and the tile's largest
    // log2 sc_t give m and the upper bound m + LG_t of x + log2 sc_t; the maxima that grew past
    // their threshold are raised, O (per half) and the partial sums rescaled, and the pass
    // redone. A segment's first tile starts there.
    const int sm = warp - 4;                                 // softmax warp index
    const int qd = warp & 3;                                 // TMEM lane quarter
    const int hb = 32 * (sm >> 2);                           // first head of this warp
    const int tr = 32 * qd + lane;                           // key row of the tile / dv row of O^T
    const int sid = 32 * sm + lane;                          // softmax thread index
    const uint32_t tl = tmem + ((uint32_t)(32 * qd) << 16);  // this warp's lanes
    float* red = reinterpret_cast<float*>(smem + RED_OFF);
    float* red_m = red;              // [64] running max m of x (exp2 domain)
    float* red_mt = red + 64;        // [2][64] running max m'_t of x + log2 sc_t
    float* red_r = red + 192;        // [64][2] r_t = 2^(m - m'_t + kPShift), both tiles of a head together
    float* red_al = red + 320;       // [3][64] rescale factors (sums, O half 0, O half 1); epilogue:
                                     // weights of the own partial per half
    float* red_nm = red + 1280 + 2 * kMaxParts * kH + 2 * kNSM;  // [64] -m (the pass adds it)
    float* red_part = red + 512;     // [3][4 lane quarters][64]
    float* red_wk = red + 1280;      // [2][kMaxParts][64]: merge weights of the other parts per half
    int* votes = reinterpret_cast<int*>(red + 1280 + 2 * kMaxParts * kH);  // [2][kNSM]
    uint8_t* qbuf = smem + Q_OFF;
    uint32_t mc = 0, g = 0, xc = 0, lb = 0, qs = 0;
    auto xsync = [&](bool v) -> int {
      const int r = softmax_exchange(xbar, votes, xc++, sm, v ? 1 : 0);
      if (r < 0) fail(DSA_DEVERR_TIMEOUT);
      return r;
    };
    auto wait_all = [&](bool ok) -> bool {
      if (__all_sync(0xffffffffu, ok)) return true;
      fail(DSA_DEVERR_TIMEOUT);
      return false;
    };
    auto pv_wait = [&](int64_t last) -> bool {  // every output product up to tile `last` complete
      if (last < 0) return true;
      return mbar_wait(pv_done((uint32_t)last & 1), ((uint32_t)last >> 1) & 1, kWaitNs);
    };
    // split token t's query into Q (its previous use released) and publish it to the score issuer
    auto make_q = [&](int64_t t) -> bool {
      if (qs > 0 && !wait_all(mbar_wait(q_empty, (qs - 1) & 1, kWaitNs))) return false;
      split_query(p, t, qbuf, sq, sm, lane);
      fence_proxy_async_smem();
      if (xsync(false) < 0) return false;
      if (sid == 0) mbar_arrive(q_full);
      ++qs;
      return true;
    };
    const uint32_t sw = tr & 7;
    bool run = wait_all(mbar_wait(range_ready, 0, kWaitNs));
    if (run && range[1] > range[0]) run = make_q(range[0] / p.NT);
    while (run) {
      const int st = mc % kMST;
      if (!wait_all(mbar_wait(m_full(st), (mc / kMST) & 1, kWaitNs))) break;
      const MetaHdr* mh = reinterpret_cast<const MetaHdr*>(smem + META_OFF + st * META_BYTES);
      const int type = mh->type;
      if (type == kDone) {
        __syncwarp();
        if (lane == 0) mbar_arrive(m_empty(st));
        break;
      }
      if (type == kTile) {
        const int n_valid = mh->n_valid;
        const int first = mh->first;
        __syncwarp();
        if (lane == 0) mbar_arrive(m_empty(st));
        ++mc;
        const int ks = g % kKST;
        bool ok = mbar_wait(s_full(g & 1), (g >> 1) & 1, kWaitNs);
        ok = ok && mbar_wait(k_full(ks), (g / kKST) & 1, kWaitNs);  // the row scales
        ok = ok && pv_wait((int64_t)g - kPBUF);                       // this P buffer is free
        if (!wait_all(ok)) break;
        tc_fence_after();
        const bool valid = tr < n_valid;
        const float2 sc = *reinterpret_cast<const float2*>(smem + SC_OFF + ks * SC_BYTES + tr * 8);
        const uint32_t sa = tl + (g & 1) * S_COLS + hb;
        const uint32_t lcur = tl + L_COL + 64 * lb + hb, lnxt = tl + L_COL + 64 * (lb ^ 1) + hb;
        uint8_t* prow0 = smem + P_OFF + (g & 1) * P_BYTES + tr * 128;
        uint8_t* prow1 = prow0 + kBN * 128;
        // x (exp2 domain) of head h = hb + 16 ch + i: each tile's accumulator times its row scale
        // and the head's c * 2^e of that tile
        auto xval = [&](const uint32_t (&a)[16], const uint32_t (&bb)[16], int h, int i) -> float {
          return fmaf(u2f(a[i]), sc.x * sq[2 * h], u2f(bb[i]) * (sc.y * sq[2 * h + 1]));
        };
        bool exact = first != 0, bad = false;
        for (;;) {
          bool resc = false;
          if (exact) {
            // exact per-head maxima of x over this tile's keys (warp max-reductions over the keys,
            // then across the four lane quarters) and the tile's largest log2 sc_t (LG_t): the
            // output halves take m'_t = m + LG_t, an upper bound of x + log2 sc_t, so that every
            // P_t of the tile is at most 2^kPShift
            const float lg0 = valid && sc.x > 0.0f ? __log2f(sc.x) : -INFINITY;
            const float lg1 = valid && sc.y > 0.0f ? __log2f(sc.y) : -INFINITY;
            {
              const int l0 = redux_max_s32(f2ord(lg0)), l1 = redux_max_s32(f2ord(lg1));
              if (lane == 0 && hb == 0) {
                red_part[256 + qd] = ord2f(l0);
                red_part[256 + 4 + qd] = ord2f(l1);
              }
            }
#pragma unroll 1
            for (int ch = 0; ch < 2; ++ch) {
              uint32_t a[16], bb[16];
              tmem_ld32_x16(sa + 16 * ch, a);
              tmem_ld32_x16(sa + 64 + 16 * ch, bb);
              tc_wait_ld();
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const int h = hb + 16 * ch + i;
                const int m0 = redux_max_s32(f2ord(valid ? xval(a, bb, h, i) : -INFINITY));
                if (lane == ((16 * ch + i) & 31)) red_part[qd * 64 + h] = ord2f(m0);
              }
            }
            if (xsync(false) < 0) { bad = true; break; }
            bool grow_any = false;
            if (sid < kH) {
              const float mt = fmaxf(fmaxf(red_part[sid], red_part[64 + sid]), fmaxf(red_part[128 + sid], red_part[192 + sid]));
              const float* lg = red_part + 256;
              const float LG0 = fmaxf(fmaxf(lg[0], lg[1]), fmaxf(lg[2], lg[3]));
              const float LG1 = fmaxf(fmaxf(lg[4], lg[5]), fmaxf(lg[6], lg[7]));
              // m: grows past kTauL; m'_t: past kTau (a half with no non-zero scale yet keeps m)
              const float mo = first ? -INFINITY : red_m[sid];
              const bool gl = first || mt > mo + kTauL;
              const float mn = gl ? mt : mo;
              red_al[sid] = gl ? ex2_approx(mo - mn) : 1.0f;
              red_m[sid] = mn;
              red_nm[sid] = -mn;
              grow_any = gl && !first;
#pragma unroll
              for (int t = 0; t < 2; ++t) {
                const float cand = mt + (t ? LG1 : LG0);
                const float to = first ? -INFINITY : red_mt[t * kH + sid];
                const bool gt = first || cand > to + kTau;
                float tn = gt ? cand : to;
                if (tn == -INFINITY) tn = mn;  // no key with a non-zero scale: P_t is 0 anyway
                red_al[(1 + t) * kH + sid] = (gt && to != -INFINITY) ? ex2_approx(to - tn) : 1.0f;
                red_mt[t * kH + sid] = tn;
                red_r[2 * sid + t] = exp2f(mn - tn + (float)kPShift);
                grow_any |= gt && !first;
              }
            }
            const int r = xsync(grow_any);
            if (r < 0) { bad = true; break; }
            resc = r != 0;
          }
          if (resc) {
            // rare: some maximum grew; scale the O^T columns of those heads per half (every
            // issued PV complete) and the partial sums the pass reads next
            if (!wait_all(pv_wait((int64_t)g - 1))) { bad = true; break; }
            tc_fence_after();
#pragma unroll 1
            for (int ch = 0; ch < 2; ++ch) {
              uint32_t o0[16], o1[16], lv[16];
              tmem_ld32_x16(tl + O_COL + hb + 16 * ch, o0);
              tmem_ld32_x16(tl + O_COL + 64 + hb + 16 * ch, o1);
              tmem_ld32_x16(lcur + 16 * ch, lv);
              tc_wait_ld();
              const float* al = red_al + hb + 16 * ch;
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                lv[i] = f2u(u2f(lv[i]) * al[i]);
                o0[i] = f2u(u2f(o0[i]) * al[kH + i]);
                o1[i] = f2u(u2f(o1[i]) * al[2 * kH + i]);
              }
              tmem_st32_x16(tl + O_COL + hb + 16 * ch, o0);
              tmem_st32_x16(tl + O_COL + 64 + hb + 16 * ch, o1);
              tmem_st32_x16(lcur + 16 * ch, lv);
            }
            tc_wait_st();
          }
          // the pass: p = 2^(x - m) (one MUFU ex2 per score), partial row sums into the other
          // TMEM buffer, and P_t = p * sc_t * r_t as e4m3 hi/lo terms into this key's rows
          float xm = -INFINITY, pm = 0.0f;
          const float2 sc2 = make_float2(sc.x, sc.y);
#pragma unroll 1
          for (int ch = 0; ch < 2; ++ch) {
            uint32_t a[16], bb[16], l[16];
            tmem_ld32_x16(sa + 16 * ch, a);
            tmem_ld32_x16(sa + 64 + 16 * ch, bb);
            if (!first) tmem_ld32_x16(lcur + 16 * ch, l);
            tc_wait_ld();
            if (first) {
#pragma unroll
              for (int i = 0; i < 16; ++i) l[i] = 0u;
            }
            uint32_t hw0[4], lw0[4], hw1[4], lw1[4];
            if (valid) {
#pragma unroll
              for (int hq = 0; hq < 4; ++hq) {  // four heads at a time, two by two
                float g0[4], g1[4];
#pragma unroll
                for (int j = 0; j < 4; j += 2) {
                  const int i = 4 * hq + j, h = hb + 16 * ch + i;
                  // constants of heads h, h + 1: c * 2^e per tile, r per tile, -m
                  const float4 A = *reinterpret_cast<const float4*>(sq + 2 * h);
                  const float4 R = *reinterpret_cast<const float4*>(red_r + 2 * h);
                  const float2 nm = *reinterpret_cast<const float2*>(red_nm + h);
                  const float2 a0 = __fmul2_rn(sc2, make_float2(A.x, A.y));
                  const float2 a1 = __fmul2_rn(sc2, make_float2(A.z, A.w));
                  const float x0 = fmaf(u2f(a[i]), a0.x, fmaf(u2f(bb[i]), a0.y, nm.x));
                  const float x1 = fmaf(u2f(a[i + 1]), a1.x, fmaf(u2f(bb[i + 1]), a1.y, nm.y));
                  xm = fmaxf(xm, fmaxf(x0, x1));
                  const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                  l[i] = f2u(u2f(l[i]) + p0);
                  l[i + 1] = f2u(u2f(l[i + 1]) + p1);
                  const float2 w0 = __fmul2_rn(__fmul2_rn(sc2, make_float2(R.x, R.y)), make_float2(p0, p0));
                  const float2 w1 = __fmul2_rn(__fmul2_rn(sc2, make_float2(R.z, R.w)), make_float2(p1, p1));
                  pm = fmaxf(pm, fmaxf(fmaxf(w0.x, w0.y), fmaxf(w1.x, w1.y)));
                  g0[j] = w0.x;
                  g0[j + 1] = w1.x;
                  g1[j] = w0.y;
                  g1[j + 1] = w1.y;
                }
                split4(g0[0], g0[1], g0[2], g0[3], hw0[hq], lw0[hq]);
                split4(g1[0], g1[1], g1[2], g1[3], hw1[hq], lw1[hq]);
              }
            } else {
              // a row past the tile's valid count: no weight, no sum
#pragma unroll
              for (int hq = 0; hq < 4; ++hq) hw0[hq] = lw0[hq] = hw1[hq] = lw1[hq] = 0u;
            }
            tmem_st32_x16(lnxt + 16 * ch, l);
            const uint32_t gh = (hb >> 4) + ch;  // 16-byte granule of these 16 heads (hi term)
            *reinterpret_cast<uint4*>(prow0 + ((gh ^ sw) << 4)) = make_uint4(hw0[0], hw0[1], hw0[2], hw0[3]);
            *reinterpret_cast<uint4*>(prow0 + (((4 + gh) ^ sw) << 4)) = make_uint4(lw0[0], lw0[1], lw0[2], lw0[3]);
            *reinterpret_cast<uint4*>(prow1 + ((gh ^ sw) << 4)) = make_uint4(hw1[0], hw1[1], hw1[2], hw1[3]);
            *reinterpret_cast<uint4*>(prow1 + (((4 + gh) ^ sw) << 4)) = make_uint4(lw1[0], lw1[1], lw1[2], lw1[3]);
          }
          if (exact) break;
          const int r = xsync(xm > kTauL || pm > kPMax);
          if (r < 0) { bad = true; break; }
          if (r == 0) break;
          exact = true;
        }
        if (bad) break;
        lb ^= 1;
        fence_proxy_async_smem();
        tc_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(p_full(g & 1));
          mbar_arrive(s_empty(g & 1));
        }
        ++g;
        continue;
      }
      // ====================================================== kSegEnd: token epilogue ====
      const int64_t t = mh->token;
      const int kind = mh->kind, had = mh->had_tiles, last = mh->merge_last, next = mh->next_token;
      __syncwarp();
      if (lane == 0) mbar_arrive(m_empty(st));
      ++mc;
      // every softmax warp is past this segment's tiles (and its reads of sq): split the next
      // segment's query first, so that its score products run during this epilogue
      if (next >= 0) {
        if (xsync(false) < 0) break;
        if (!make_q(next)) break;
      }
      const uint32_t lfin = tl + L_COL + 64 * lb + hb;  // the partial sums the last pass wrote
      // row sums: per warp, a reduce-scatter over the lanes (keys) of each 16-head chunk leaves
      // the warp's sum of head 16 ch + (lane >> 1) in lanes 2i and 2i + 1; lane 2i writes it to
      // red_part[quarter][head], and thread h < 64 adds up the quarters
#pragma unroll 1
      for (int ch = 0; ch < 2; ++ch) {
        uint32_t l[16];
        if (had) {
          tmem_ld32_x16(lfin + 16 * ch, l);
          tc_wait_ld();
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) l[i] = 0u;
        }
        float v8[8], v4[4], v2[2];
        const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4, b1 = lane & 2;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float lo = u2f(l[i]), hi = u2f(l[i + 8]);
          v8[i] = (b4 ? hi : lo) + __shfl_xor_sync(0xffffffffu, b4 ? lo : hi, 16);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) v4[i] = (b3 ? v8[i + 4] : v8[i]) + __shfl_xor_sync(0xffffffffu, b3 ? v8[i] : v8[i + 4], 8);
#pragma unroll
        for (int i = 0; i < 2; ++i) v2[i] = (b2 ? v4[i + 2] : v4[i]) + __shfl_xor_sync(0xffffffffu, b2 ? v4[i] : v4[i + 2], 4);
        float v1 = (b1 ? v2[1] : v2[0]) + __shfl_xor_sync(0xffffffffu, b1 ? v2[0] : v2[1], 2);
        v1 += __shfl_xor_sync(0xffffffffu, v1, 1);
        if ((lane & 1) == 0) red_part[qd * 64 + hb + 16 * ch + (lane >> 1)] = v1;
      }
      if (xsync(false) < 0) break;
      float lsum = 0.0f, mrow = -INFINITY, mh0 = -INFINITY, mh1 = -INFINITY;
      if (sid < kH && had) {
        lsum = (red_part[sid] + red_part[64 + sid]) + (red_part[128 + sid] + red_part[192 + sid]);
        mrow = red_m[sid];
        mh0 = red_mt[sid];
        mh1 = red_mt[kH + sid];
      }
      // the quarter sums and maxima are read before a next tile's exact path rewrites them
      if (xsync(false) < 0) break;
      if (had) {
        if (!wait_all(pv_wait((int64_t)g - 1))) break;
        tc_fence_after();
      }
      float* wsml = p.ws_ml;  // [G][4][64]: m, l, m'_0, m'_1
      if (kind == kPart) {
        // publish (O^T, m, l, m'_0, m'_1) of this part in workspace slot b
        if (sid < kH) {
          wsml[((int64_t)b * 4 + 0) * kH + sid] = mrow;
          wsml[((int64_t)b * 4 + 1) * kH + sid] = lsum;
          wsml[((int64_t)b * 4 + 2) * kH + sid] = mh0;
          wsml[((int64_t)b * 4 + 3) * kH + sid] = mh1;
        }
        if (had) {
          // rows dv = tr and 128 + tr of O^T; the 16-byte granule of heads 4q .. 4q + 3 sits at
          // position q ^ (tr & 15) of its 256-byte row, so that the merge reads the rows from
          // shared memory without bank conflicts
          float* w0 = p.ws_o + ((int64_t)b * kD + tr) * kH;
          float* w1 = p.ws_o + ((int64_t)b * kD + 128 + tr) * kH;
#pragma unroll 1
          for (int ch = 0; ch < 2; ++ch) {
            uint32_t o0[16], o1[16];
            tmem_ld32_x16(tl + O_COL + hb + 16 * ch, o0);
            tmem_ld32_x16(tl + O_COL + 64 + hb + 16 * ch, o1);
            tc_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; i += 4) {
              const int pos = 4 * ((((hb + 16 * ch + i) >> 2) ^ tr) & 15);
              *reinterpret_cast<float4*>(w0 + pos) = make_float4(u2f(o0[i]), u2f(o0[i + 1]), u2f(o0[i + 2]), u2f(o0[i + 3]));
              *reinterpret_cast<float4*>(w1 + pos) = make_float4(u2f(o1[i]), u2f(o1[i + 1]), u2f(o1[i + 2]), u2f(o1[i + 3]));
            }
          }
        }
        __threadfence();
        __syncwarp();
        if (lane == 0)
          asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p.flags + 8 * b + sm), "r"(p.epoch) : "memory");
        tc_fence_before();
        continue;
      }
      // complete token, or the head of a split token: merge parts b+1 .. last in order
      const int nparts = kind == kHead ? last - b : 0;
      bool okp = true;
      for (int f0 = 0; f0 < nparts * kNSM && okp; f0 += 32) {
        const int f = f0 + lane;
        const bool mine = f < nparts * kNSM;
        const int* fp = p.flags + 8 * (b + 1 + f / kNSM) + f % kNSM;
        const uint64_t t0 = globaltimer_ns();
        for (;;) {
          int v = p.epoch;
          if (mine) asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(fp) : "memory");
          if (__all_sync(0xffffffffu, v == p.epoch)) break;
          if (__any_sync(0xffffffffu, globaltimer_ns() - t0 > kWaitNs)) {
            okp = false;
            break;
          }
          __nanosleep(64);
        }
      }
      __syncwarp();
      if (!okp) fail(DSA_DEVERR_TIMEOUT);
      const int np = (okp && nparts <= kMaxParts) ? nparts : 0;
      // The parts' rows come into shared memory by bulk copies: their (m, l, m'_0, m'_1) rows
      // (consecutive workspace slots b+1 .. b+np) into the Q buffer, and their O^T halves into
      // two slot pairs (K stages 0-1, and K stage 2 with P buffer 1), two parts in flight. A
      // head segment is its CTA's last, so none of these buffers is in use any more: every
      // output product is complete, and no further query split or row load follows.
      auto slot = [&](int pair, int half) -> uint32_t {
        return sbase + (pair == 0 ? KT_OFF + half * KT_BYTES : (half == 0 ? KT_OFF + 2 * KT_BYTES : P_OFF + P_BYTES));
      };
      auto fetch_part = [&](int k) {  // one thread: part k (1-based) into slot pair (k - 1) & 1
        const uint32_t mb = merge_bar(1 + ((k - 1) & 1));
        const float* src = p.ws_o + (int64_t)(b + k) * kD * kH;
        mbar_arrive_expect_tx(mb, kD * kH * 4);
        bulk_g2s(slot((k - 1) & 1, 0), src, 128 * kH * 4, mb);
        bulk_g2s(slot((k - 1) & 1, 1), src + 128 * kH, 128 * kH * 4, mb);
      };
      if (np > 0 && sid == 0) {
        // the flags were acquired by this warp; order the parts' data (read by the async proxy)
        // after them, and the buffers' earlier uses before the copies
        asm volatile("fence.proxy.async.global;" ::: "memory");
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(merge_bar(0), np * 4 * kH * 4);
        bulk_g2s(sbase + Q_OFF, wsml + (int64_t)(b + 1) * 4 * kH, np * 4 * kH * 4, merge_bar(0));
        fetch_part(1);
        if (np >= 2) fetch_part(2);
      }
      if (sid < kH) {
        // sums relative to the largest m over the parts; each half's O of each part weighted
        // by 2^(m'_t - M - kPShift) / L
        const float* pml = reinterpret_cast<const float*>(smem + Q_OFF);  // [np][4][64]
        if (np > 0 && !mbar_wait(merge_bar(0), 0, kWaitNs)) fail(DSA_DEVERR_TIMEOUT);
        float M = mrow;
        for (int k = 1; k <= np; ++k) M = fmaxf(M, pml[(k - 1) * 4 * kH + sid]);
        float L = lsum > 0.0f ? exp2f(mrow - M) * lsum : 0.0f;
        for (int k = 1; k <= np; ++k) {
          const float mk = pml[((k - 1) * 4 + 0) * kH + sid];
          const float lk = pml[((k - 1) * 4 + 1) * kH + sid];
          if (lk > 0.0f) L += exp2f(mk - M) * lk;
        }
        const float inv = L > 0.0f ? 1.0f / L : 0.0f;
        const float base = M + (float)kPShift;
        red_al[sid] = lsum > 0.0f ? exp2f(mh0 - base) * inv : 0.0f;
        red_al[kH + sid] = lsum > 0.0f ? exp2f(mh1 - base) * inv : 0.0f;
        for (int k = 1; k <= np; ++k) {
          const bool live = pml[((k - 1) * 4 + 1) * kH + sid] > 0.0f;
          red_wk[(k - 1) * kH + sid] = live ? exp2f(pml[((k - 1) * 4 + 2) * kH + sid] - base) * inv : 0.0f;
          red_wk[(kMaxParts + k - 1) * kH + sid] = live ? exp2f(pml[((k - 1) * 4 + 3) * kH + sid] - base) * inv : 0.0f;
        }
        if (p.lse) p.lse[t * kH + sid] = L > 0.0f ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
      }
      if (xsync(false) < 0) break;
      // combine: this CTA's O (TMEM) and the parts in order, then stage the bf16 block
      // [64 heads][256 columns] in P buffer 0 (idle: every output product is complete)
      uint16_t* stage = reinterpret_cast<uint16_t*>(smem + P_OFF);
      // The sum accumulates in this CTA's O columns of tensor memory (lane = d_v row): first its
      // own O times its weights, then each part in order as it lands, one 16-head chunk at a
      // time; the last step writes bf16 to the stage instead.
      bool okm = true;
      for (int k = 0; k <= np && okm; ++k) {
        const int pr = (k - 1) & 1;
        if (k > 0 && !wait_all(mbar_wait(merge_bar(1 + pr), ((k - 1) >> 1) & 1, kWaitNs))) {
          okm = false;
          break;
        }
#pragma unroll 1
        for (int q = 0; q < 4; ++q) {  // (16-head chunk, d_v half)
          const int h0 = hb + 16 * (q >> 1), half = q & 1;
          const uint32_t tc = tl + O_COL + 64 * half + h0;
          uint32_t o[16];
          if (k > 0 || had) {
            tmem_ld32_x16(tc, o);
            tc_wait_ld();
          }
          if (k == 0) {
            const float* w = red_al + half * kH + h0;
#pragma unroll
            for (int i = 0; i < 16; ++i) o[i] = f2u(had ? w[i] * u2f(o[i]) : 0.0f);
          } else {
            const uint8_t* r = smem + (slot(pr, half) - sbase) + tr * 256;
            const float* w = red_wk + (half * kMaxParts + k - 1) * kH + h0;
#pragma unroll
            for (int i = 0; i < 16; i += 4) {
              const float4 x = *reinterpret_cast<const float4*>(r + 16 * ((((h0 + i) >> 2) ^ tr) & 15));
              o[i] = f2u(fmaf(w[i], x.x, u2f(o[i])));
              o[i + 1] = f2u(fmaf(w[i + 1], x.y, u2f(o[i + 1])));
              o[i + 2] = f2u(fmaf(w[i + 2], x.z, u2f(o[i + 2])));
              o[i + 3] = f2u(fmaf(w[i + 3], x.w, u2f(o[i + 3])));
            }
          }
          if (k == np) {
#pragma unroll
            for (int i = 0; i < 16; ++i) stage[(h0 + i) * kD + 128 * half + tr] = __bfloat16_as_ushort(__float2bfloat16_rn(u2f(o[i])));
          } else {
            tmem_st32_x16(tc, o);
          }
        }
        if (k < np) tc_wait_st();  // the next step reads these columns back
        if (k >= 1 && k + 2 <= np) {
          // every warp has read this slot pair: refill it with part k + 2
          if (xsync(false) < 0) {
            okm = false;
            break;
          }
          if (sid == 0) {
            fence_proxy_async_smem();
            fetch_part(k + 2);
          }
        }
      }
      if (!okm) break;
      if (xsync(false) < 0) break;
      // every softmax warp has read the parts: clear their publish flags, so that the workspace
      // holds no set flag after the call (a later call that carries the same tag, such as a
      // replay of a recorded launch, then never mistakes this call's flags for its own)
      for (int f = sid; f < np * kNSM; f += 32 * kNSM) p.flags[8 * (b + 1 + f / kNSM) + f % kNSM] = 0;
      {
        uint16_t* orow = p.out + t * p.out_st;
#pragma unroll 4
        for (int j = 0; j < 2048 / (32 * kNSM); ++j) {
          const int q = sid + 32 * kNSM * j, h = q >> 5, gq = q & 31;
          *reinterpret_cast<uint4*>(orow + (int64_t)h * p.out_sh + gq * 8) =
              *reinterpret_cast<const uint4*>(stage + h * kD + gq * 8);
        }
      }
      // the staging area is a P buffer: every warp's copy-out reads complete before a next
      // tile's pass writes P
      if (xsync(false) < 0) break;
      tc_fence_before();
    }
  } else {
    // ================================================= row loaders (warps 3, 12-15) ====
    // Row pairs (2p, 2p + 1) of each K tile go to loader p % 5 (lanes 0-15 row 2p, 16-31 row
    // 2p + 1; lane il copies 16-byte granule il), in the 128-byte-swizzled K-major layout (row r,
    // granule q of chunk c at c * 16 KB + r * 128 + ((q ^ (r & 7)) << 4)). A row that starts
    // 16-byte aligned (even slot) takes 16-byte copies, the others 8-byte copies; rows past the
    // tile's valid count are zero-filled (a zero row keeps 0 * V finite). The two scales of a
    // row go to the stage's scale array. Each thread's copies signal the stage's full barrier
    // when they land.
    const int li = warp == 3 ? 0 : warp - 11;  // loader index 0-4
    const int npairs = (kBN / 2 - li + kNLD - 1) / kNLD;
    const int hl = lane >> 4, il = lane & 15;
    const int cc = il >> 3, gg = il & 7;
    uint32_t mc = 0, g = 0;
    while (!*abort_flag) {
      const int st = mc % kMST;
      if (!wait(m_full(st), (mc / kMST) & 1)) break;
      const MetaHdr* mh = reinterpret_cast<const MetaHdr*>(smem + META_OFF + st * META_BYTES);
      const int type = mh->type;
      if (type != kTile) {
        // a segment end: pull the next segment's query into L2 (the softmax warps split it when
        // they reach this entry, some tiles later)
        const int next = type == kSegEnd ? mh->next_token : -1;
        __syncwarp();
        if (lane == 0) mbar_arrive(m_empty(st));
        ++mc;
        if (li == 0 && next >= 0) prefetch_q(next);
        if (type == kDone) break;
        continue;
      }
      // lane j holds the slot of row 2 (li + 5 (j >> 1)) + (j & 1), or -1 past the valid rows
      const int n = mh->n_valid;
      const int* slots = reinterpret_cast<const int*>(reinterpret_cast<const uint8_t*>(mh) + META_HDR);
      const int rj = 2 * (li + kNLD * (lane >> 1)) + (lane & 1);
      const int slr = (lane < 2 * npairs && rj < n) ? slots[rj] : -1;
      __syncwarp();
      if (lane == 0) mbar_arrive(m_empty(st));
      ++mc;
      const int ks = g % kKST;
      if (g >= (uint32_t)kKST && !wait(k_empty(ks), ((g / kKST) & 1) ^ 1)) break;
      const uint32_t kt = sbase + KT_OFF + ks * KT_BYTES + cc * (kBN * 128);
      const uint32_t scs = sbase + SC_OFF + ks * SC_BYTES;
#pragma unroll 1
      for (int k = 0; k < npairs; ++k) {
        const int r = 2 * (li + kNLD * k) + hl;
        const int sl = __shfl_sync(0xffffffffu, slr, 2 * k + hl);
        const uint32_t dst = kt + r * 128 + ((gg ^ (r & 7)) << 4);
        const uint8_t* row = p.cache + (int64_t)(sl >= 0 ? sl : 0) * kRB;
        if (sl >= 0 && (sl & 1) == 0) {
          asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(row + 16 * il) : "memory");
        } else if (sl >= 0) {
          asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(row + 16 * il) : "memory");
          asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst + 8), "l"(row + 16 * il + 8) : "memory");
        } else {
          asm volatile("cp.async.cg.shared.global [%0], [%1], 16, 0;" ::"r"(dst), "l"(row) : "memory");
        }
        if (il == 0)
          asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;" ::"r"(scs + r * 8), "l"(row + kD),
                       "r"(sl >= 0 ? 8 : 0)
                       : "memory");
      }
      asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(k_full(ks)) : "memory");
      ++g;
    }
    // drain this thread's outstanding cp.async copies before the CTA can finish
    asm volatile("cp.async.wait_all;" ::: "memory");
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace f8

cudaError_t f8_set_attributes() {
  return cudaFuncSetAttribute(f8::attn_f8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, f8::SMEM_BYTES);
}

dsa_status_t launch_attn_f8(const dsa_attn_args_t* a, const DeviceInfo& dev, cudaStream_t stream) {
  using namespace f8;
  Params p{};
  p.cache = static_cast<const uint8_t*>(a->cache);
  p.num_slots = a->num_slots;
  p.q = static_cast<const uint16_t*>(a->q);
  p.q_st = a->q_stride_t;
  p.q_sh = a->q_stride_h;
  p.idx = a->indices;
  p.idx_stride = a->idx_stride_t;
  p.topk = a->topk;
  p.bt = a->block_table;
  p.bt_stride = a->bt_stride;
  p.page_size = a->block_table ? a->page_size : 1;
  p.max_pages = a->block_table ? a->max_pages : 0;
  {
    // round-up reciprocal: with l = ceil(log2 d) and m = ceil(2^(31+l) / d) < 2^32,
    // floor(x * m / 2^(31+l)) == floor(x / d) for every 0 <= x < 2^31
    const uint64_t d = (uint64_t)p.page_size;
    int l = 0;
    while ((1ull << l) < d) ++l;
    p.pg_mul = (uint32_t)(((1ull << (31 + l)) + d - 1) / d);
    p.pg_shift = 31 + l;
  }
  p.req = a->req_of_token;
  p.c_log2 = a->sm_scale * 1.4426950408889634f;
  p.out = static_cast<uint16_t*>(a->out);
  p.out_st = a->out_stride_t;
  p.out_sh = a->out_stride_h;
  p.lse = a->lse;
  const AttnWorkspace ws = attn_ws_layout(a->workspace, dev.sm_count);
  p.ws_o = ws.o;
  p.ws_ml = ws.ml;
  p.flags = ws.flags;
  p.err = a->error_word;
  p.epoch = next_attn_epoch(a->workspace);
  p.T = a->T;
  UnitSplit us;
  dsa_status_t st = plan_unit_split(a, dev, ws, stream, &us);
  if (st != DSA_OK) return st;
  p.NT = us.NT;
  p.U = us.U;
  p.G = us.G;
  p.bounds = us.bounds;
  p.split_gap = us.gap;

  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)p.G);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, attn_f8_kernel, p);
  return e == cudaSuccess ? DSA_OK : cuda_fail(e);
}

}  // namespace dsa
