// dsa_attn_ctl.cu - DSA sparse MLA attention forward over the packed scaled-FP8 cache of the
// 512+64 control geometry on sm_103a, with keys as the MMA M dimension and 8-bit operands.
//
// What is computed (sglang PR #38547 "Enable zero-RoPE TileLang DSA on gfx950", Summary,
// Contract table rows "scaled FP8 cache row", "HIP FP8 main width" and "HIP FP8 RoPE tail"):
// for every query token t and head h, gather the 656-byte rows named by t's top-k list (entries
// < 0 masked): 512 e4m3 codes with one fp32 scale per 128-column tile, then 64 bf16 RoPE
// values. k = (code * scale, rope), s_j = sm_scale * q[t,h].k_j, softmax over j, and the output
// is sum_j p_j * (code * scale)_j over the 512 NoPE columns (d_v = 512) in bf16, with the
// natural-log sum of exp(s_j) as an optional second output.
//
// Kernel design (the 256+0 kernel of dsa_attn_f8.cu, widened):
//  * A work unit is (token, half of the 64 heads, 128-position window): with 32 heads as the
//    MMA N dimension the five score accumulators of a key (four scale tiles and the RoPE part)
//    and O^T over all 512 output columns fit the 512 TMEM columns, double-buffered scores
//    included (2 x 160 + 128 + 64). Each key row is gathered by both head halves' CTAs (the
//    43 MB control cache is L2-resident).
//  * K tiles stay 8-bit in shared memory: 128 keys x 512 codes (four 128-byte-swizzled chunks
//    of 16 KB, one per scale tile), two stages; the RoPE part (128 keys x 64 bf16) has one
//    buffer, released as soon as the tile's score products complete. Rows are 16-byte aligned
//    (656 = 41 x 16), so every copy is a 16-byte cp.async.
//  * Scores: per scale tile t, S_t += K_t Q_t^T with tcgen05 kind::f8f6f4, the bf16 query of
//    each head split exactly into two e4m3 terms per tile (q = 2^e (hi + lo), hi the top four
//    significant bits); S_r += K_r Q_r^T with kind::f16 on the bf16 RoPE values. The score is
//    x = sum_t sc_t c 2^e_t S_t + c S_r (exp2 domain, c = sm_scale log2 e).
//  * Softmax per key (thread = TMEM lane), lazy running maxima per head: m of x (row sums) and
//    m'_t of x + log2 sc_t (output quarter t). P_t = 2^(x + log2 sc_t - m'_t + 4) < 2^8.5 is
//    written as two e4m3 terms; one P buffer, whose stores wait for the previous tile's output
//    products.
//  * Output O^T += V_t^T P_t^T per quarter t (M = 128 output columns, MN-major V from code chunk
//    t, N = 32 heads), hi then lo term.
//  * Persistent cooperative launch, one CTA per SM, units split into equal contiguous ranges; a
//    unit sequence cut by a range boundary is merged in-kernel by the CTA holding its first
//    tiles (parts bulk-copied into idle shared memory, added in a fixed order into its O columns
//    of tensor memory; no atomics on data).
//  * Warp roles: 0 producer, 1 score-MMA issuer, 2 output-MMA issuer, 4-11 softmax, query split
//    and epilogue (two warps per TMEM lane quarter, 16 heads each), 3 and 12-15 row loaders.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "dsa_attn_common.h"
#include "dsa_host.h"
#include "dsa_ptx.cuh"

namespace dsa {
namespace ctl {

constexpr int kH = 32;          // heads per unit: MMA N
constexpr int kD = 512;         // codes (= d_v)
constexpr int kDR = 64;         // RoPE values
constexpr int kRB = 656;        // packed row bytes
constexpr int kNT = 4;          // scale tiles = output quarters
constexpr int kBN = 128;        // gathered keys per tile: MMA M
constexpr int kKST = 2;         // code stages
constexpr int kMST = 4;         // meta ring depth
constexpr int kWarps = 16;
constexpr int kThreads = 32 * kWarps;
constexpr int kNSM = 8;         // softmax warps 4-11 (two per TMEM lane quarter, 16 heads each)
constexpr int kNLD = 5;         // loader warps 3, 12-15
constexpr int kMaxParts = 16;   // most parts of one split unit sequence (the launch guarantees it)
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr float kTau = 4.5f;     // lazy maxima of the output quarters: a tile may exceed them by 2^4.5
constexpr float kTauL = 20.0f;   // lazy maximum of the row sums
constexpr int kPShift = 4;       // P weights carry an extra 2^4 ...
constexpr float kPMax = 400.0f;  // ... and stay below 2^8.5 (e4m3 tops at 448)

// shared memory carve-up (offsets from a 1024-aligned base)
constexpr int Q_OFF = 0;                 // per tile t at t * 8 KB: hi [32 heads][128 B], lo 4 KB further
constexpr int QR_OFF = Q_OFF + 32768;    // RoPE query [32 heads][64 bf16]
constexpr int KT_OFF = QR_OFF + 4096;    // code stages: stage s at s * 64 KB, chunk t at t * 16 KB
constexpr int KT_BYTES = kBN * kD;
constexpr int KR_OFF = KT_OFF + kKST * KT_BYTES;  // RoPE rows [128 keys][64 bf16]
constexpr int P_OFF = KR_OFF + kBN * 128;         // P: quarters (0, 1) rows, then (2, 3) rows, 16 KB each
constexpr int P_BYTES = 2 * kBN * 128;
constexpr int SC_OFF = P_OFF + P_BYTES;           // per stage: the four tile scales of each row
constexpr int SC_BYTES = kBN * 16;
constexpr int SQ_OFF = SC_OFF + kKST * SC_BYTES;  // [32 heads][4 tiles] c * 2^e
constexpr int META_OFF = SQ_OFF + kH * kNT * 4;
constexpr int META_HDR = 48;
constexpr int META_BYTES = META_HDR + 4 * kBN;
constexpr int CMP_OFF = META_OFF + kMST * META_BYTES;
constexpr int RED_OFF = CMP_OFF + 4 * 256;
// m[32], m'[4][32], r[32][4], alpha[5][32], part[4][32] + lg[4 quarters][4 tiles], -m[32], votes[2][8]
constexpr int RED_FLOATS = kH + 4 * kH + 4 * kH + 5 * kH + 4 * kH + 16 + kH + 2 * kNSM;
enum : int {
  B_QFULL = 0, B_QEMPTY = 1, B_KFULL = 2, B_KEMPTY = B_KFULL + kKST, B_REMPTY = B_KEMPTY + kKST,
  B_RFULL = B_REMPTY + 1, B_MFULL = B_RFULL + 1, B_MEMPTY = B_MFULL + kMST, B_SFULL = B_MEMPTY + kMST, B_SEMPTY = B_SFULL + 2,
  B_PFULL = B_SEMPTY + 2, B_PVDONE = B_PFULL + 1, B_XBAR = B_PVDONE + 2, B_DRAIN = B_XBAR + 1,
  B_RANGE = B_DRAIN + 2, B_MERGE = B_RANGE + 1, NBARS = B_MERGE + 3
};
constexpr int BAR_OFF = RED_OFF + ((RED_FLOATS * 4 + 15) & ~15);
constexpr int MISC_OFF = BAR_OFF + 8 * NBARS;
constexpr int SMEM_BYTES = MISC_OFF + 48 + 1024;  // + alignment slack
// tensor memory columns
constexpr int S_COLS = 160;             // per S buffer (two): S_t at +32 t, S_r at +128
constexpr int O_COL = 2 * S_COLS;       // O^T quarter t (output columns 128 t ..) at O_COL + 32 t
constexpr int L_COL = O_COL + 128;      // per-lane partial row sums, two buffers of 32 columns
constexpr int TMEM_COLS = 512;
static_assert(L_COL + 64 <= TMEM_COLS, "TMEM budget");
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(KT_OFF % 1024 == 0 && KR_OFF % 1024 == 0 && P_OFF % 1024 == 0 && QR_OFF % 1024 == 0, "operand alignment");
static_assert(kNSM <= 8, "one publish flag per softmax warp, eight per CTA");
static_assert(kRB == kD + 4 * kNT + 2 * kDR && 2 * kDR == 128, "row layout: codes, scales, 128 RoPE bytes");
static_assert(kMaxParts * kNT * kH * 4 <= kBN * 128, "merge weights fit the RoPE buffer");
static_assert(kMaxParts * 6 * kH * 4 <= 32768, "parts' running values fit the Q buffer");

enum : int { kTile = 1, kSegEnd = 2, kDone = 3 };
enum : int { kComplete = 0, kHead = 1, kPart = 2 };

struct MetaHdr {
  int type;
  int token;       // unit sequence: 2 * token + head half
  int n_valid;
  int first;
  int kind;
  int had_tiles;
  int merge_last;
  int seg;
  int next_token;
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
  uint32_t pg_mul;
  int pg_shift;
  const int32_t* req;
  float c_log2;
  uint16_t* out;
  int64_t out_st, out_sh;
  float* lse;
  float* ws_o;   // [G][512 dv][32 heads] partial O^T (quarter t relative to 2^(m'_t - kPShift))
  float* ws_ml;  // [G][6][32] partial m, l, m'_0 .. m'_3
  int* flags;    // [G][8]
  int epoch;
  int32_t* err;
  int64_t VT;    // unit sequences: 2 per token
  int NT;
  int64_t U;
  int G;
};

__device__ __forceinline__ void set_err(int32_t* err, int bits) {
  if (err) atomicOr(err, bits);
}
__device__ __forceinline__ int64_t unit_begin(int64_t b, int64_t U, int G) { return (b * U) / G; }
__device__ __forceinline__ float u2f(uint32_t u) { return __uint_as_float(u); }
__device__ __forceinline__ uint32_t f2u(float f) { return __float_as_uint(f); }
__device__ __forceinline__ int ilog2f(float w) {
  const uint32_t b = __float_as_uint(w);
  return b >= 0x800000u ? (int)(b >> 23) - 127 : (31 - __clz((int)b)) - 149;
}
__device__ __forceinline__ float pow2i(int k) { return __uint_as_float((uint32_t)(k + 127) << 23); }
__device__ __forceinline__ float trunc4(float v) { return __uint_as_float(__float_as_uint(v) & 0xFFF00000u); }
__device__ __forceinline__ void split4(float a, float b, float c, float d, uint32_t& hi, uint32_t& lo) {
  const float ha = trunc4(a), hb = trunc4(b), hc = trunc4(c), hd = trunc4(d);
  hi = (uint32_t)f32x2_to_e4m3x2(ha, hb) | ((uint32_t)f32x2_to_e4m3x2(hc, hd) << 16);
  lo = (uint32_t)f32x2_to_e4m3x2(a - ha, b - hb) | ((uint32_t)f32x2_to_e4m3x2(c - hc, d - hd) << 16);
}
__device__ __forceinline__ void tmem_ld32_x8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32_x8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
               "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}

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

// Query split of unit sequence vt (token vt / 2, heads 32 (vt % 2) ..): softmax warp sm takes
// its heads 4 sm .. 4 sm + 3. For each head, lane l holds columns 16l .. 16l + 15 of the 512
// NoPE columns (tile l / 8): e = the binary exponent of the tile's largest |q| minus 7,
// x = q * 2^-e exactly, hi = x truncated to four significant bits, lo = x - hi; the terms go to
// the K-major 128-byte-swizzled Q operand of that tile and c * 2^e to sq[head][tile]. Lanes 0-7
// copy the head's 64 RoPE values (bf16, exact) into the RoPE operand.
static __device__ __forceinline__ void split_query(const Params& p, int64_t vt, uint8_t* smem, float* sq, int sm,
                                                   int lane) {
  const int64_t t = vt >> 1;
  const int hh = (int)(vt & 1);
  const int tile = lane >> 3, gq = lane & 7;
#pragma unroll 1
  for (int i = 0; i < 4; ++i) {
    const int h = 4 * sm + i;
    const uint16_t* qrow = p.q + t * p.q_st + (int64_t)(kH * hh + h) * p.q_sh;
    const uint4 v0 = __ldg(reinterpret_cast<const uint4*>(qrow + 16 * lane));
    const uint4 v1 = __ldg(reinterpret_cast<const uint4*>(qrow + 16 * lane + 8));
    const uint4 vr = lane < 8 ? __ldg(reinterpret_cast<const uint4*>(qrow + kD + 8 * lane)) : make_uint4(0u, 0u, 0u, 0u);
    const uint32_t wd[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    float f[16];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      f[2 * j] = u2f(wd[j] << 16);
      f[2 * j + 1] = u2f(wd[j] & 0xFFFF0000u);
    }
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(f[j]));
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    int e = amax > 0.0f ? ilog2f(amax) - 7 : 0;
    e = e < -120 ? -120 : (e > 120 ? 120 : e);
    const float inv = pow2i(-e);
#pragma unroll
    for (int j = 0; j < 16; ++j) f[j] *= inv;
    uint32_t hw[4], lw[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) split4(f[4 * j], f[4 * j + 1], f[4 * j + 2], f[4 * j + 3], hw[j], lw[j]);
    const int off = Q_OFF + tile * 8192 + h * 128 + ((gq ^ (h & 7)) << 4);
    *reinterpret_cast<uint4*>(smem + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    *reinterpret_cast<uint4*>(smem + off + 4096) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
    if (gq == 0) sq[h * kNT + tile] = pow2i(e) * p.c_log2;
    if (lane < 8) *reinterpret_cast<uint4*>(smem + QR_OFF + h * 128 + ((lane ^ (h & 7)) << 4)) = vr;
  }
}

__global__ void __launch_bounds__(kThreads, 1) attn_ctl_kernel(const __grid_constant__ Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const uint32_t bar0 = sbase + BAR_OFF;
  auto bar = [&](int i) { return bar0 + 8 * i; };
  const uint32_t q_full = bar(B_QFULL), q_empty = bar(B_QEMPTY);
  auto k_full = [&](int s) { return bar(B_KFULL + s); };
  auto k_empty = [&](int s) { return bar(B_KEMPTY + s); };
  const uint32_t r_empty = bar(B_REMPTY);  // the RoPE buffer: the score products that read it are complete
  const uint32_t r_full = bar(B_RFULL);    // the RoPE buffer holds the current tile's rows
  auto m_full = [&](int s) { return bar(B_MFULL + s); };
  auto m_empty = [&](int s) { return bar(B_MEMPTY + s); };
  auto s_full = [&](int i) { return bar(B_SFULL + i); };
  auto s_empty = [&](int i) { return bar(B_SEMPTY + i); };
  const uint32_t p_full = bar(B_PFULL);
  auto pv_done = [&](int i) { return bar(B_PVDONE + i); };
  const uint32_t xbar = bar(B_XBAR);
  const uint32_t mma_drain = bar(B_DRAIN);
  const uint32_t range_ready = bar(B_RANGE);
  auto merge_bar = [&](int i) { return bar(B_MERGE + i); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + MISC_OFF + 4);
  int64_t* range = reinterpret_cast<int64_t*>(smem + MISC_OFF + 8);
  float* sq = reinterpret_cast<float*>(smem + SQ_OFF);

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int s = 0; s < kKST; ++s) {
      mbar_init(k_full(s), 32 * kNLD);
      mbar_init(k_empty(s), 1);
    }
    mbar_init(r_empty, 1);
    mbar_init(r_full, 32 * kNLD);
    for (int s = 0; s < kMST; ++s) {
      mbar_init(m_full(s), 1);
      mbar_init(m_empty(s), 2 + kNSM + kNLD);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(s_full(i), 1);
      mbar_init(s_empty(i), kNSM);
      mbar_init(pv_done(i), 1);
    }
    mbar_init(p_full, kNSM);
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

  if (warp == 0) {
    // =========================================================== producer (one warp) ====
    // Walks this CTA's unit range, one segment per unit sequence vt (token vt / 2): index
    // window reads two steps ahead, masking, page translation, compaction into dense 128-key
    // tiles (as in the 256+0 kernels).
    uint32_t mc = 0;
    const int64_t u0 = unit_begin(b, p.U, p.G);
    const int64_t u1 = unit_begin(b + 1, p.U, p.G);
    if (lane == 0) {
      range[0] = u0;
      range[1] = u1;
      mbar_arrive(range_ready);
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
    int64_t vt = u0 / p.NT;
    int j0 = (int)(u0 - vt * p.NT);
    int seg = 0;
    while (u < u1 && !*abort_flag) {
      const int j1 = (int)((int64_t)(p.NT - j0) < u1 - u ? p.NT : j0 + (u1 - u));
      const int64_t uend = u + (j1 - j0);
      const int kind = j0 > 0 ? kPart : (j1 < p.NT ? kHead : kComplete);
      const int64_t t = vt >> 1;
      const int64_t req = p.req ? p.req[t] : 0;
      const int32_t* irow = p.idx + t * p.idx_stride;
      const int32_t* btrow = p.bt ? p.bt + req * p.bt_stride : nullptr;
      const int e0 = j0 * kBN, e1 = min(j1 * kBN, p.topk);
      {
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
          mh->token = (int)vt;
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
            slot = -2;
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
          me->token = (int)vt;
          me->kind = kind;
          me->had_tiles = had ? 1 : 0;
          me->seg = seg;
          me->next_token = uend < u1 ? (int)(vt + 1) : -1;
          int last = b;
          if (kind == kHead) {
            const int64_t L1 = (vt + 1) * p.NT;
            const int64_t c = (L1 * p.G + p.U - 1) / p.U - 1;
            last = (int)(c < p.G - 1 ? c : p.G - 1);
          }
          me->merge_last = last;
        }
        emit_end(st2);
      }
      u = uend;
      ++vt;
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
    if (lane == 0) {
      constexpr uint32_t idS = idesc_e4m3(128, kH, 0, 0);    // A = K chunk (K-major), B = Q term (K-major)
      constexpr uint32_t idR = idesc_bf16(128, kH, 0, 0);    // A = RoPE rows, B = RoPE query (bf16, K-major)
      constexpr uint32_t idPV = idesc_e4m3(128, kH, 1, 1);   // A = V_t^T (MN-major), B = P_t^T term (MN-major)
      const uint32_t k_hi = (uint32_t)(sw128_desc(0, 16, 1024) >> 32);
      const uint32_t mn_hi = (uint32_t)(sw128_desc(0, 16384, 1024) >> 32);
      const uint32_t q_lo = (uint32_t)sw128_desc(sbase + Q_OFF, 16, 1024);
      const uint32_t qr_lo = (uint32_t)sw128_desc(sbase + QR_OFF, 16, 1024);
      const uint32_t kr_lo = (uint32_t)sw128_desc(sbase + KR_OFF, 16, 1024);
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
          // ---- scores: per scale tile t, four K-steps of 32 codes, Q's hi term then its lo
          // term into S_t; then the RoPE part, four K-steps of 16 bf16 into S_r
          if (first && !wait(q_full, seg & 1)) break;
          if (g >= 2 && !wait(s_empty(g & 1), ((g >> 1) & 1) ^ 1)) break;
          if (!wait(k_full(ks), (g / kKST) & 1)) break;
          fence_proxy_async_smem();
          tc_fence_after();
          const uint32_t k_lo = (uint32_t)sw128_desc(sbase + KT_OFF + ks * KT_BYTES, 16, 1024);
          const uint32_t d0 = tmem + (g & 1) * S_COLS;
#pragma unroll
          for (int t = 0; t < kNT; ++t) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint32_t ka = k_lo + (uint32_t)((t * (kBN * 128) + 32 * kk) >> 4);
              const uint32_t qa = q_lo + (uint32_t)((t * 8192 + 32 * kk) >> 4);
              if (kk == 0) mma_f8_lohi<0>(d0 + 32 * t, ka, k_hi, qa, k_hi, idS);
              else mma_f8_lohi<1>(d0 + 32 * t, ka, k_hi, qa, k_hi, idS);
              mma_f8_lohi<1>(d0 + 32 * t, ka, k_hi, qa + (4096 >> 4), k_hi, idS);
            }
          }
          if (!wait(r_full, g & 1)) break;
          fence_proxy_async_smem();
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            if (kk == 0) mma_bf16_lohi<0>(d0 + 128, kr_lo, k_hi, qr_lo, k_hi, idR);
            else mma_bf16_lohi<1>(d0 + 128, kr_lo + 2 * kk, k_hi, qr_lo + 2 * kk, k_hi, idR);
          }
          mma_commit(s_full(g & 1));
          mma_commit(r_empty);
        } else {
          // ---- output: quarter t takes P_t, hi term then lo term (32 bytes further)
          if (!wait(p_full, g & 1)) break;
          tc_fence_after();
          const uint32_t v_lo = (uint32_t)sw128_desc(sbase + KT_OFF + ks * KT_BYTES, 16384, 1024);
          const uint32_t p_lo = (uint32_t)sw128_desc(sbase + P_OFF, 16384, 1024);
#pragma unroll
          for (int t = 0; t < kNT; ++t) {
            const uint32_t d = tmem + O_COL + 32 * t;
            const uint32_t va = v_lo + (uint32_t)((t * (kBN * 128)) >> 4);
            const uint32_t pa = p_lo + (uint32_t)(((t >> 1) * (kBN * 128) + (t & 1) * 64) >> 4);
            mma_f8_lohi_rt(d, va, mn_hi, pa, mn_hi, idPV, first ? 0u : 1u);
            mma_f8_lohi<1>(d, va, mn_hi, pa + (32 >> 4), mn_hi, idPV);
#pragma unroll
            for (int kk = 1; kk < kBN / 32; ++kk) {
              mma_f8_lohi<1>(d, va + ((4096 * kk) >> 4), mn_hi, pa + ((4096 * kk) >> 4), mn_hi, idPV);
              mma_f8_lohi<1>(d, va + ((4096 * kk) >> 4), mn_hi, pa + ((4096 * kk + 32) >> 4), mn_hi, idPV);
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
    // take heads 0-15 and 16-31 of the unit, in two groups of eight. Running maxima per head:
    // m (of x) and m'_t (of x + log2 sc_t, reference of output quarter t); P_t = p sc_t r_t with
    // p = 2^(x - m), r_t = 2^(m - m'_t + kPShift). A vote checks P_t <= kPMax and x - m <= kTauL;
    // else (and on a segment's first tile) the exact path recomputes the maxima.
    const int sm = warp - 4;
    const int qd = warp & 3;
    const int hb = 16 * (sm >> 2);
    const int tr = 32 * qd + lane;
    const int sid = 32 * sm + lane;
    const uint32_t tl = tmem + ((uint32_t)(32 * qd) << 16);
    float* red = reinterpret_cast<float*>(smem + RED_OFF);
    float* red_m = red;                     // [32]
    float* red_mt = red + kH;               // [4][32]
    float* red_r = red + 5 * kH;            // [32][4]
    float* red_al = red + 9 * kH;           // [5][32] (sums, O quarters 0-3); epilogue: own weights per quarter
    float* red_part = red + 14 * kH;        // [4 lane quarters][32]; then lg [4 lane quarters][4 tiles]
    float* red_lg = red + 18 * kH;          // [4][4]
    float* red_nm = red + 18 * kH + 16;     // [32] -m
    int* votes = reinterpret_cast<int*>(red + 19 * kH + 16);  // [2][8]
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
    auto pv_wait = [&](int64_t last) -> bool {
      if (last < 0) return true;
      return mbar_wait(pv_done((uint32_t)last & 1), ((uint32_t)last >> 1) & 1, kWaitNs);
    };
    auto make_q = [&](int64_t vt) -> bool {
      if (qs > 0 && !wait_all(mbar_wait(q_empty, (qs - 1) & 1, kWaitNs))) return false;
      split_query(p, vt, smem, sq, sm, lane);
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
        if (!wait_all(ok)) break;
        tc_fence_after();
        const bool valid = tr < n_valid;
        const float4 sc = *reinterpret_cast<const float4*>(smem + SC_OFF + ks * SC_BYTES + tr * 16);
        const float scv[4] = {sc.x, sc.y, sc.z, sc.w};
        const uint32_t sa = tl + (g & 1) * S_COLS + hb;
        const uint32_t lcur = tl + L_COL + 32 * lb + hb, lnxt = tl + L_COL + 32 * (lb ^ 1) + hb;
        uint8_t* prow = smem + P_OFF + tr * 128;
        bool p_free = false;  // the previous tile's output products have read P
        bool exact = first != 0, bad = false;
        for (;;) {
          bool resc = false;
          if (exact) {
            // per-head maxima of x over the tile's keys and each tile's largest log2 sc_t
            if (hb == 0) {
#pragma unroll
              for (int t = 0; t < kNT; ++t) {
                const int l = redux_max_s32(f2ord(valid && scv[t] > 0.0f ? __log2f(scv[t]) : -INFINITY));
                if (lane == 0) red_lg[qd * 4 + t] = ord2f(l);
              }
            }
#pragma unroll 1
            for (int g8 = 0; g8 < 2; ++g8) {
              uint32_t a[5][8];
#pragma unroll
              for (int t = 0; t < 5; ++t) tmem_ld32_x8(sa + 32 * t + 8 * g8, a[t]);
              tc_wait_ld();
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const int h = hb + 8 * g8 + i;
                float x = u2f(a[4][i]) * p.c_log2;
#pragma unroll
                for (int t = 0; t < kNT; ++t) x = fmaf(u2f(a[t][i]), scv[t] * sq[h * kNT + t], x);
                const int mx = redux_max_s32(f2ord(valid ? x : -INFINITY));
                if (lane == 0) red_part[qd * kH + h] = ord2f(mx);
              }
            }
            if (xsync(false) < 0) { bad = true; break; }
            bool grow_any = false;
            if (sid < kH) {
              const float mt = fmaxf(fmaxf(red_part[sid], red_part[kH + sid]), fmaxf(red_part[2 * kH + sid], red_part[3 * kH + sid]));
              const float mo = first ? -INFINITY : red_m[sid];
              const bool gl = first || mt > mo + kTauL;
              const float mn = gl ? mt : mo;
              red_al[sid] = gl ? ex2_approx(mo - mn) : 1.0f;
              red_m[sid] = mn;
              red_nm[sid] = -mn;
              grow_any = gl && !first;
#pragma unroll
              for (int t = 0; t < kNT; ++t) {
                const float LG = fmaxf(fmaxf(red_lg[t], red_lg[4 + t]), fmaxf(red_lg[8 + t], red_lg[12 + t]));
                const float cand = mt + LG;
                const float to = first ? -INFINITY : red_mt[t * kH + sid];
                const bool gt = first || cand > to + kTau;
                float tn = gt ? cand : to;
                if (tn == -INFINITY) tn = mn;
                red_al[(1 + t) * kH + sid] = (gt && to != -INFINITY) ? ex2_approx(to - tn) : 1.0f;
                red_mt[t * kH + sid] = tn;
                red_r[sid * 4 + t] = exp2f(mn - tn + (float)kPShift);
                grow_any |= gt && !first;
              }
            }
            const int r = xsync(grow_any);
            if (r < 0) { bad = true; break; }
            resc = r != 0;
          }
          if (resc) {
            // rare: a maximum grew; scale the O^T columns of those heads per quarter and the
            // partial sums the pass reads next (every issued output product complete)
            if (!wait_all(pv_wait((int64_t)g - 1))) { bad = true; break; }
            tc_fence_after();
#pragma unroll 1
            for (int g8 = 0; g8 < 2; ++g8) {
              uint32_t lv[8];
              tmem_ld32_x8(lcur + 8 * g8, lv);
              tc_wait_ld();
#pragma unroll
              for (int i = 0; i < 8; ++i) lv[i] = f2u(u2f(lv[i]) * red_al[hb + 8 * g8 + i]);
              tmem_st32_x8(lcur + 8 * g8, lv);
#pragma unroll 1
              for (int t = 0; t < kNT; ++t) {
                uint32_t o[8];
                tmem_ld32_x8(tl + O_COL + 32 * t + hb + 8 * g8, o);
                tc_wait_ld();
#pragma unroll
                for (int i = 0; i < 8; ++i) o[i] = f2u(u2f(o[i]) * red_al[(1 + t) * kH + hb + 8 * g8 + i]);
                tmem_st32_x8(tl + O_COL + 32 * t + hb + 8 * g8, o);
              }
            }
            tc_wait_st();
          }
          // the pass: p = 2^(x - m), partial row sums into the other TMEM buffer, and
          // P_t = p sc_t r_t as e4m3 hi/lo terms into this key's rows
          float xm = -INFINITY, pm = 0.0f;
#pragma unroll 1
          for (int g8 = 0; g8 < 2; ++g8) {
            uint32_t a[5][8], l[8];
#pragma unroll
            for (int t = 0; t < 5; ++t) tmem_ld32_x8(sa + 32 * t + 8 * g8, a[t]);
            if (!first) tmem_ld32_x8(lcur + 8 * g8, l);
            tc_wait_ld();
            if (first) {
#pragma unroll
              for (int i = 0; i < 8; ++i) l[i] = 0u;
            }
            uint32_t hw[4][2], lw[4][2];  // [quarter][four heads]
            if (valid) {
#pragma unroll
              for (int hq = 0; hq < 2; ++hq) {  // four heads at a time
                float w[4][4];  // [quarter][head]
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  const int i = 4 * hq + j, h = hb + 8 * g8 + i;
                  const float4 A = *reinterpret_cast<const float4*>(sq + h * kNT);
                  const float4 R = *reinterpret_cast<const float4*>(red_r + h * 4);
                  float x = fmaf(u2f(a[4][i]), p.c_log2, red_nm[h]);
                  x = fmaf(u2f(a[0][i]), scv[0] * A.x, x);
                  x = fmaf(u2f(a[1][i]), scv[1] * A.y, x);
                  x = fmaf(u2f(a[2][i]), scv[2] * A.z, x);
                  x = fmaf(u2f(a[3][i]), scv[3] * A.w, x);
                  xm = fmaxf(xm, x);
                  const float pp = ex2_approx(x);
                  l[i] = f2u(u2f(l[i]) + pp);
                  w[0][j] = pp * (scv[0] * R.x);
                  w[1][j] = pp * (scv[1] * R.y);
                  w[2][j] = pp * (scv[2] * R.z);
                  w[3][j] = pp * (scv[3] * R.w);
                  pm = fmaxf(pm, fmaxf(fmaxf(w[0][j], w[1][j]), fmaxf(w[2][j], w[3][j])));
                }
#pragma unroll
                for (int t = 0; t < kNT; ++t) split4(w[t][0], w[t][1], w[t][2], w[t][3], hw[t][hq], lw[t][hq]);
              }
            } else {
#pragma unroll
              for (int t = 0; t < kNT; ++t) hw[t][0] = hw[t][1] = lw[t][0] = lw[t][1] = 0u;
            }
            tmem_st32_x8(lnxt + 8 * g8, l);
            if (!p_free) {
              if (!wait_all(pv_wait((int64_t)g - 1))) {
                bad = true;
                break;
              }
              p_free = true;
            }
            // quarter t: row group t / 2; hi bytes of heads hb .. at logical byte 64 (t % 2) + hb,
            // lo 32 bytes further; this group's eight heads are the 8-byte half 8 g8 of the granule
            const int bo = 8 * g8;
#pragma unroll
            for (int t = 0; t < kNT; ++t) {
              uint8_t* row = prow + (t >> 1) * (kBN * 128);
              const uint32_t ch = (uint32_t)(4 * (t & 1) + (hb >> 4));
              *reinterpret_cast<uint2*>(row + ((ch ^ sw) << 4) + bo) = make_uint2(hw[t][0], hw[t][1]);
              *reinterpret_cast<uint2*>(row + (((ch + 2) ^ sw) << 4) + bo) = make_uint2(lw[t][0], lw[t][1]);
            }
          }
          if (bad) break;
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
          mbar_arrive(p_full);
          mbar_arrive(s_empty(g & 1));
        }
        ++g;
        continue;
      }
      // ====================================================== kSegEnd: epilogue ====
      const int64_t vt = mh->token;
      const int kind = mh->kind, had = mh->had_tiles, last = mh->merge_last, next = mh->next_token;
      __syncwarp();
      if (lane == 0) mbar_arrive(m_empty(st));
      ++mc;
      if (next >= 0) {
        if (xsync(false) < 0) break;
        if (!make_q(next)) break;
      }
      const uint32_t lfin = tl + L_COL + 32 * lb + hb;
      {
        // row sums: a reduce-scatter over the lanes (keys) of the warp's 16 heads leaves head
        // hb + (lane >> 1) in lanes 2i and 2i + 1; the four lane quarters are added by thread h
        uint32_t l0[8], l1[8];
        if (had) {
          tmem_ld32_x8(lfin, l0);
          tmem_ld32_x8(lfin + 8, l1);
          tc_wait_ld();
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) l0[i] = l1[i] = 0u;
        }
        float v8[8], v4[4], v2[2];
        const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4, b1 = lane & 2;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float lo = u2f(l0[i]), hi = u2f(l1[i]);
          v8[i] = (b4 ? hi : lo) + __shfl_xor_sync(0xffffffffu, b4 ? lo : hi, 16);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) v4[i] = (b3 ? v8[i + 4] : v8[i]) + __shfl_xor_sync(0xffffffffu, b3 ? v8[i] : v8[i + 4], 8);
#pragma unroll
        for (int i = 0; i < 2; ++i) v2[i] = (b2 ? v4[i + 2] : v4[i]) + __shfl_xor_sync(0xffffffffu, b2 ? v4[i] : v4[i + 2], 4);
        float v1 = (b1 ? v2[1] : v2[0]) + __shfl_xor_sync(0xffffffffu, b1 ? v2[0] : v2[1], 2);
        v1 += __shfl_xor_sync(0xffffffffu, v1, 1);
        if ((lane & 1) == 0) red_part[qd * kH + hb + (lane >> 1)] = v1;
      }
      if (xsync(false) < 0) break;
      float lsum = 0.0f, mrow = -INFINITY, mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      if (sid < kH && had) {
        lsum = (red_part[sid] + red_part[kH + sid]) + (red_part[2 * kH + sid] + red_part[3 * kH + sid]);
        mrow = red_m[sid];
#pragma unroll
        for (int t = 0; t < kNT; ++t) mq[t] = red_mt[t * kH + sid];
      }
      if (xsync(false) < 0) break;
      if (had) {
        if (!wait_all(pv_wait((int64_t)g - 1))) break;
        tc_fence_after();
      }
      float* wsml = p.ws_ml;  // [G][6][32]: m, l, m'_0 .. m'_3
      if (kind == kPart) {
        if (sid < kH) {
          wsml[((int64_t)b * 6 + 0) * kH + sid] = mrow;
          wsml[((int64_t)b * 6 + 1) * kH + sid] = lsum;
#pragma unroll
          for (int t = 0; t < kNT; ++t) wsml[((int64_t)b * 6 + 2 + t) * kH + sid] = mq[t];
        }
        if (had) {
          // row dv = 128 t + tr of O^T (128 bytes: 32 heads); the 16-byte granule of heads
          // 4q .. 4q + 3 at position q ^ (tr & 7)
#pragma unroll 1
          for (int t = 0; t < kNT; ++t) {
            float* wr = p.ws_o + ((int64_t)b * kD + 128 * t + tr) * kH;
            uint32_t o0[8], o1[8];
            tmem_ld32_x8(tl + O_COL + 32 * t + hb, o0);
            tmem_ld32_x8(tl + O_COL + 32 * t + hb + 8, o1);
            tc_wait_ld();
#pragma unroll
            for (int i = 0; i < 8; i += 4) {
              const int p0 = 4 * ((((hb + i) >> 2) ^ tr) & 7), p1 = 4 * ((((hb + 8 + i) >> 2) ^ tr) & 7);
              *reinterpret_cast<float4*>(wr + p0) = make_float4(u2f(o0[i]), u2f(o0[i + 1]), u2f(o0[i + 2]), u2f(o0[i + 3]));
              *reinterpret_cast<float4*>(wr + p1) = make_float4(u2f(o1[i]), u2f(o1[i + 1]), u2f(o1[i + 2]), u2f(o1[i + 3]));
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
      // Parts come into the idle buffers of this CTA's finished last segment by bulk copies:
      // their running values into the Q buffer, their O^T (64 KB each) into code stage
      // (k - 1) % 2, two in flight; the merge weights go to the RoPE buffer.
      auto fetch_part = [&](int k) {
        const uint32_t mb = merge_bar(1 + ((k - 1) & 1));
        mbar_arrive_expect_tx(mb, kD * kH * 4);
        bulk_g2s(sbase + KT_OFF + ((k - 1) & 1) * KT_BYTES, p.ws_o + (int64_t)(b + k) * kD * kH, kD * kH * 4, mb);
      };
      float* red_wk = reinterpret_cast<float*>(smem + KR_OFF);  // [4 quarters][kMaxParts][32]
      if (np > 0 && sid == 0) {
        asm volatile("fence.proxy.async.global;" ::: "memory");
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(merge_bar(0), np * 6 * kH * 4);
        bulk_g2s(sbase + Q_OFF, wsml + (int64_t)(b + 1) * 6 * kH, np * 6 * kH * 4, merge_bar(0));
        fetch_part(1);
        if (np >= 2) fetch_part(2);
      }
      if (sid < kH) {
        const float* pml = reinterpret_cast<const float*>(smem + Q_OFF);  // [np][6][32]
        if (np > 0 && !mbar_wait(merge_bar(0), 0, kWaitNs)) fail(DSA_DEVERR_TIMEOUT);
        float M = mrow;
        for (int k = 1; k <= np; ++k) M = fmaxf(M, pml[(k - 1) * 6 * kH + sid]);
        float L = lsum > 0.0f ? exp2f(mrow - M) * lsum : 0.0f;
        for (int k = 1; k <= np; ++k) {
          const float mk = pml[((k - 1) * 6 + 0) * kH + sid];
          const float lk = pml[((k - 1) * 6 + 1) * kH + sid];
          if (lk > 0.0f) L += exp2f(mk - M) * lk;
        }
        const float inv = L > 0.0f ? 1.0f / L : 0.0f;
        const float base = M + (float)kPShift;
#pragma unroll
        for (int t = 0; t < kNT; ++t) red_al[(1 + t) * kH + sid] = lsum > 0.0f ? exp2f(mq[t] - base) * inv : 0.0f;
        for (int k = 1; k <= np; ++k) {
          const bool live = pml[((k - 1) * 6 + 1) * kH + sid] > 0.0f;
#pragma unroll
          for (int t = 0; t < kNT; ++t)
            red_wk[(t * kMaxParts + k - 1) * kH + sid] = live ? exp2f(pml[((k - 1) * 6 + 2 + t) * kH + sid] - base) * inv : 0.0f;
        }
        if (p.lse) {
          const int64_t tok = vt >> 1;
          p.lse[tok * kAttnHeads + kH * (vt & 1) + sid] = L > 0.0f ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
        }
      }
      if (xsync(false) < 0) break;
      // O accumulates in TMEM: own O times its weights, then each part as it lands; the last
      // step writes bf16 [32 heads][512 columns] to the P buffer (idle: every output product
      // of this segment is complete)
      uint16_t* stage = reinterpret_cast<uint16_t*>(smem + P_OFF);
      bool okm = true;
      for (int k = 0; k <= np && okm; ++k) {
        const int pr = (k - 1) & 1;
        if (k > 0 && !wait_all(mbar_wait(merge_bar(1 + pr), ((k - 1) >> 1) & 1, kWaitNs))) {
          okm = false;
          break;
        }
#pragma unroll 1
        for (int q = 0; q < 2 * kNT; ++q) {  // (output quarter, group of eight heads)
          const int t = q >> 1, h0 = hb + 8 * (q & 1);
          const uint32_t tc = tl + O_COL + 32 * t + h0;
          uint32_t o[8];
          if (k > 0 || had) {
            tmem_ld32_x8(tc, o);
            tc_wait_ld();
          }
          if (k == 0) {
            const float* w = red_al + (1 + t) * kH + h0;
#pragma unroll
            for (int i = 0; i < 8; ++i) o[i] = f2u(had ? w[i] * u2f(o[i]) : 0.0f);
          } else {
            const uint8_t* r = smem + KT_OFF + pr * KT_BYTES + (128 * t + tr) * 128;
            const float* w = red_wk + (t * kMaxParts + k - 1) * kH + h0;
#pragma unroll
            for (int i = 0; i < 8; i += 4) {
              const float4 x = *reinterpret_cast<const float4*>(r + 16 * ((((h0 + i) >> 2) ^ tr) & 7));
              o[i] = f2u(fmaf(w[i], x.x, u2f(o[i])));
              o[i + 1] = f2u(fmaf(w[i + 1], x.y, u2f(o[i + 1])));
              o[i + 2] = f2u(fmaf(w[i + 2], x.z, u2f(o[i + 2])));
              o[i + 3] = f2u(fmaf(w[i + 3], x.w, u2f(o[i + 3])));
            }
          }
          if (k == np) {
#pragma unroll
            for (int i = 0; i < 8; ++i) stage[(h0 + i) * kD + 128 * t + tr] = __bfloat16_as_ushort(__float2bfloat16_rn(u2f(o[i])));
          } else {
            tmem_st32_x8(tc, o);
          }
        }
        if (k < np) tc_wait_st();
        if (k >= 1 && k + 2 <= np) {
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
      for (int f = sid; f < np * kNSM; f += 32 * kNSM) p.flags[8 * (b + 1 + f / kNSM) + f % kNSM] = 0;
      {
        // copy out: 32 heads x 1024 bytes, 2048 16-byte granules, eight per thread
        uint16_t* orow = p.out + (vt >> 1) * p.out_st + (int64_t)(kH * (vt & 1)) * p.out_sh;
#pragma unroll 4
        for (int j = 0; j < 2048 / (32 * kNSM); ++j) {
          const int q = sid + 32 * kNSM * j, h = q >> 6, gq = q & 63;
          *reinterpret_cast<uint4*>(orow + (int64_t)h * p.out_sh + gq * 8) =
              *reinterpret_cast<const uint4*>(stage + h * kD + gq * 8);
        }
      }
      if (xsync(false) < 0) break;
      tc_fence_before();
    }
  } else {
    // ================================================= row loaders (warps 3, 12-15) ====
    // Row k of a tile goes to loader k % 5, whose lane k / 5 holds its slot. Per tile, first the
    // codes into the free stage (one instruction per row: granule l of the row goes to chunk
    // l / 8, position l % 8) and the four scales of each row (one instruction for all the warp's
    // rows), signalled on k_full; then, once the previous tile's score products have read the
    // RoPE buffer, the 128 RoPE bytes of each row (four rows per instruction), signalled on
    // r_full. The codes of the next tile thus stream in while the current one is scored. Rows
    // past the tile's valid count are zero-filled.
    const int li = warp == 3 ? 0 : warp - 11;
    const int nrow = (kBN - li + kNLD - 1) / kNLD;  // rows li + 5 k, k < nrow
    uint32_t mc = 0, g = 0;
    bool stop = false;
    while (!stop && !*abort_flag) {
      const int st = mc % kMST;
      if (!wait(m_full(st), (mc / kMST) & 1)) break;
      const MetaHdr* mh = reinterpret_cast<const MetaHdr*>(smem + META_OFF + st * META_BYTES);
      const int type = mh->type;
      int n = 0, slr = -1;
      const int rt = li + kNLD * lane;
      if (type == kTile) {
        n = mh->n_valid;
        const int* slots = reinterpret_cast<const int*>(reinterpret_cast<const uint8_t*>(mh) + META_HDR);
        if (lane < nrow && rt < n) slr = slots[rt];
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(m_empty(st));
      ++mc;
      if (type == kDone) break;
      if (type != kTile) continue;
      const int ks = g % kKST;
      if (g >= (uint32_t)kKST && !wait(k_empty(ks), ((g / kKST) & 1) ^ 1)) break;
      const uint32_t kt = sbase + KT_OFF + ks * KT_BYTES;
      const uint32_t kr = sbase + KR_OFF;
      const uint32_t scs = sbase + SC_OFF + ks * SC_BYTES;
#pragma unroll 2
      for (int k = 0; k < nrow; ++k) {
        const int r = li + kNLD * k;
        const int sl = __shfl_sync(0xffffffffu, slr, k);
        const uint8_t* row = p.cache + (int64_t)(sl >= 0 ? sl : 0) * kRB;
        const uint32_t dst = kt + (lane >> 3) * (kBN * 128) + r * 128 + (((lane & 7) ^ (r & 7)) << 4);
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(row + 16 * lane), "r"(sl >= 0 ? 16 : 0)
                     : "memory");
      }
      if (lane < nrow) {
        const uint8_t* row = p.cache + (int64_t)(slr >= 0 ? slr : 0) * kRB;
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(scs + rt * 16), "l"(row + kD),
                     "r"(slr >= 0 ? 16 : 0)
                     : "memory");
      }
      asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(k_full(ks)) : "memory");
      if (g >= 1 && !wait(r_empty, (g - 1) & 1)) break;  // the RoPE buffer's previous tile is scored
      // four rows per instruction: lane 8 j + i copies granule i of row 4 k4 + j
#pragma unroll 1
      for (int k4 = 0; k4 < nrow; k4 += 4) {
        const int k = k4 + (lane >> 3), gi = lane & 7;
        const int sl = __shfl_sync(0xffffffffu, slr, k & 31);
        if (k < nrow) {
          const int r = li + kNLD * k;
          const uint8_t* row = p.cache + (int64_t)(sl >= 0 ? sl : 0) * kRB;
          asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(kr + r * 128 + ((gi ^ (r & 7)) << 4)),
                       "l"(row + kD + 16 + 16 * gi), "r"(sl >= 0 ? 16 : 0)
                       : "memory");
        }
      }
      asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(r_full) : "memory");
      ++g;
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace ctl

cudaError_t ctl_set_attributes() {
  return cudaFuncSetAttribute(ctl::attn_ctl_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, ctl::SMEM_BYTES);
}

dsa_status_t launch_attn_ctl(const dsa_attn_args_t* a, const DeviceInfo& dev, cudaStream_t stream) {
  using namespace ctl;
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
  p.VT = 2 * a->T;
  p.NT = (a->topk + kBN - 1) / kBN;
  p.U = p.VT * (int64_t)p.NT;
  // equal unit ranges, one CTA per SM, at least two units each, and few enough CTAs that a unit
  // sequence spans at most kMaxParts + 1 of them
  int64_t G = (p.U + 1) / 2;
  if (G > dev.sm_count) G = dev.sm_count;
  while (G > 1) {
    const int64_t upc = p.U / G;
    if ((p.NT + upc - 1) / upc + 1 <= kMaxParts + 1) break;
    --G;
  }
  p.G = (int)G;

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
  cudaError_t e = cudaLaunchKernelEx(&cfg, attn_ctl_kernel, p);
  return e == cudaSuccess ? DSA_OK : cuda_fail(e);
}

}  // namespace dsa
