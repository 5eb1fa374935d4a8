// dsa_attn_k128.cu - DSA sparse MLA attention forward for the 256+0 latent geometry on sm_103a,
// with the gathered keys as the MMA M dimension.
//
// What is computed (sglang PR #38547 "Enable zero-RoPE TileLang DSA on gfx950", Summary and
// Direct GLM geometry coverage list): for every query token t and head h, gather the latent
// rows named by t's top-k index list (entries < 0 masked), score s_j = sm_scale * q[t,h].k_j,
// softmax over j and return sum_j p_j * k_j (all 256 columns: d_v = d_nope, zero RoPE) in
// bf16. The cache holds bf16 rows or the packed scaled-FP8 rows of the Contract table (256
// e4m3 codes, then one fp32 scale per 128-column tile).
//
// This file holds the bf16-cache kernel; packed FP8 rows run in dsa_attn_f8.cu.
//
// Kernel design (GB300-first, not the pages' TileLang/HIP kernels):
//  * Transposed products. Scores: S^T[key, head] = K Q^T with M = 128 gathered keys, N = 64
//    heads, K-dim 256; output: O^T[dv, head] += V^T P^T in two M = 128 halves of d_v, V^T read
//    MN-major from the same K tile and P^T MN-major (one 128-byte row of 64 head weights per
//    key). tcgen05 kind::f16, bf16 operands, fp32 accumulators in tensor memory with lane =
//    key (scores) or lane = output column (O). M = 128 keeps the tensor core at full width,
//    where heads as M (M = 64) would use half of it.
//  * Softmax per key: one thread per TMEM lane holds its key's scores of 32 heads (two warps
//    per TMEM lane quarter). The running max of each head (exp2 domain) lives in shared memory
//    and is raised only when a tile exceeds it by more than 2^8 (a vote of the eight softmax
//    warps); the first tile of a segment takes exact per-head maxima with warp max-reductions.
//    Partial row sums per lane accumulate in TMEM and are reduced across lanes once per token.
//  * Persistent cooperative launch, one CTA per SM; (token, 128-position tile) units split into
//    contiguous ranges per CTA; a token cut by a range boundary is merged in-kernel by the CTA
//    holding its first tiles (fixed order, no atomics on data), from the other parts' partial
//    results brought into shared memory by bulk copies.
//  * Warp roles: 0 producer (index read, -1 compaction into dense 128-key tiles, page
//    translation, Q loads by TMA), 1 score-MMA issuer, 2 output-MMA issuer, 4-11 softmax and
//    epilogue, 3 and 12-15 row loaders (16-byte cp.async copies straight into the K tile,
//    loaded and released in two column halves).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>
#include <type_traits>

#include "dsa_attn_common.h"
#include "dsa_host.h"
#include "dsa_ptx.cuh"

namespace dsa {
namespace k128 {

constexpr int kH = kAttnHeads;  // heads: MMA N
constexpr int kD = 256;         // latent width (= d_v)
constexpr int kBN = 128;        // gathered keys per tile: MMA M
constexpr int kKST = 2;         // K tile stages
constexpr int kMST = 8;         // meta ring depth
constexpr int kWarps = 16;
constexpr int kThreads = 32 * kWarps;
constexpr int kMaxParts = 16;     // most parts of one split token (the launch guarantees it)
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr int kSplitMaxCtas = 192;  // most CTAs of a work-balanced split (its bounds live in shared memory)
constexpr int kSplitSlices = 32;    // unit slices per CTA counted by the split pre-pass
// Work of a token beyond its tiles, in key equivalents: its first tile takes the exact-maximum
// path and its segment end the epilogue (row sums, merge, output). Clock traces of CTAs that
// hold one-tile and sixteen-tile tokens put that at about 5.5 full tiles.
constexpr int kSegmentWeight = 704;

struct Cfg {
  static constexpr int RB = 512;  // cache row bytes (256 bf16)
  // Warp roles: 0 producer, 1 score-MMA issuer, 2 output-MMA issuer, 4-11 softmax (warp w takes
  // TMEM lane quarter w % 4; the two warps of a quarter split the heads), 3 and 12-15 loaders.
  static constexpr int NSM = 8;
  static constexpr int NLD = 5;
  static constexpr int HW = kH * 4 / NSM;  // heads per softmax warp
  static constexpr int CH = HW / 16;       // 16-head chunks per softmax warp
  static constexpr int NR = (kBN + NLD - 1) / NLD;  // most rows of a tile per loader warp
  // loader index of a warp, -1 for other warps
  static __device__ __forceinline__ int loader_index(int warp) { return warp == 3 ? 0 : (warp >= 12 ? warp - 11 : -1); }
  static constexpr int PBUF = 2;  // P buffers
  static constexpr int P_BYTES = kBN * 128;
  // shared memory carve-up (offsets from a 1024-aligned base)
  static constexpr int Q_OFF = 0;
  static constexpr int Q_BYTES = kH * kD * 2;
  static constexpr int KT_OFF = Q_OFF + Q_BYTES;
  static constexpr int KT_BYTES = kBN * kD * 2;
  static constexpr int P_OFF = KT_OFF + kKST * KT_BYTES;
  static constexpr int META_OFF = P_OFF + PBUF * P_BYTES;
  static constexpr int META_BYTES = 32 + 4 * kBN;
  static constexpr int CMP_OFF = META_OFF + kMST * META_BYTES;  // producer: one step's valid slots
  static constexpr int RED_OFF = CMP_OFF + 4 * 256;
  // m[64], alpha[64], spare[128], part[4][64], wk[kMaxParts][64], votes[2][8]
  static constexpr int RED_FLOATS = 8 * kH + kMaxParts * kH + 2 * NSM;
  static constexpr int SPLIT_OFF = RED_OFF + ((RED_FLOATS * 4 + 15) & ~15);  // producer: range bounds
  static constexpr int BAR_OFF = SPLIT_OFF + 8 * (kSplitMaxCtas + 1);
  static constexpr int NBARS = 2 + 4 * kKST + 2 * kMST + 8 + 3 + 3;
  static constexpr int MISC_OFF = BAR_OFF + 8 * NBARS;
  static constexpr int SMEM_BYTES = MISC_OFF + 16 + 1024;  // + alignment slack
  // tensor memory columns
  static constexpr int S_COLS = 64;          // per S buffer (two buffers)
  static constexpr int O_COL = 2 * S_COLS;   // O^T halves: dv 0-127 at O_COL, dv 128-255 at O_COL + 64
  static constexpr int L_COL = O_COL + 128;  // per-lane partial row sums, two buffers of 64 columns
  static constexpr int TMEM_COLS = 512;
  static_assert(L_COL + 128 <= TMEM_COLS, "TMEM budget");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
  static_assert(KT_OFF % 1024 == 0 && P_OFF % 1024 == 0 && KT_BYTES % 1024 == 0, "operand alignment");
  static_assert(CH == 2, "two 16-head chunks per softmax warp");
};

// meta ring entry types and segment kinds
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
  int pad;
};

struct Params {
  const uint8_t* cache;
  int64_t num_slots;
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
  float* ws_o;   // [G][256 dv][64 heads] partial O^T (unnormalised, relative to its max)
  float* ws_ml;  // [G][2][64] partial max (exp2 domain) and row sum
  int* flags;    // [G][8] partial published (holds the call's epoch), one per softmax warp
  int epoch;
  int32_t* err;
  int64_t T;
  int NT;     // 128-position tiles per token (over the index width)
  int64_t U;  // total units = T * NT
  int G;      // CTAs
  // work-balanced split (null: CTA b takes units [b U / G, (b + 1) U / G)): the first unit of
  // each CTA's range by work, G + 1 values, and the fewest units a range may hold
  const int64_t* bounds;
  int split_gap;
};

__device__ __forceinline__ void set_err(int32_t* err, int bits) {
  if (err) atomicOr(err, bits);
}
__device__ __forceinline__ int64_t unit_begin(int64_t b, int64_t U, int G) { return (b * U) / G; }
__device__ __forceinline__ float u2f(uint32_t u) { return __uint_as_float(u); }
__device__ __forceinline__ uint32_t f2u(float f) { return __float_as_uint(f); }

// Exchange among the softmax warps (one arrival each on `xbar`, phase `n` of it; `sm` is the
// warp's softmax index): returns the OR of `v` over the warps, with every warp's earlier
// shared-memory writes visible, or -1 when a warp did not arrive within the time limit.
template <int NSM>
static __device__ __noinline__ int softmax_exchange(uint32_t xbar, int* votes, uint32_t n, int sm, int v) {
  const int lane = threadIdx.x & 31;
  const int slot = n & 1;
  const bool any = __any_sync(0xffffffffu, v != 0);
  if (lane == 0) votes[slot * NSM + sm] = any ? 1 : 0;
  __syncwarp();
  if (lane == 0) mbar_arrive(xbar);
  const bool ok = mbar_wait(xbar, n & 1, kWaitNs);
  if (!__all_sync(0xffffffffu, ok)) return -1;
  int r = 0;
#pragma unroll
  for (int w = 0; w < NSM; ++w) r |= votes[slot * NSM + w];
  return r ? 1 : 0;
}

__global__ void __launch_bounds__(kThreads, 1)
    attn_k128_kernel(const __grid_constant__ Params p, const __grid_constant__ CUtensorMap tmap_q) {
  using C = Cfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const uint32_t bar0 = sbase + C::BAR_OFF;
  const uint32_t q_full = bar0, q_empty = bar0 + 8;
  // K stage s, column half h (codes / columns 0-127, 128-255): written, and free again
  auto k_full = [&](int s, int h) { return bar0 + 16 + 8 * (2 * s + h); };
  auto k_empty = [&](int s, int h) { return bar0 + 16 + 8 * (2 * kKST + 2 * s + h); };
  auto m_full = [&](int s) { return bar0 + 16 + 8 * (4 * kKST + s); };
  auto m_empty = [&](int s) { return bar0 + 16 + 8 * (4 * kKST + kMST + s); };
  const uint32_t x0 = bar0 + 16 + 8 * (4 * kKST + 2 * kMST);
  auto s_full = [&](int i) { return x0 + 8 * i; };
  auto s_empty = [&](int i) { return x0 + 16 + 8 * i; };
  auto p_full = [&](int i) { return x0 + 32 + 8 * i; };
  auto pv_done = [&](int i) { return x0 + 48 + 8 * i; };
  const uint32_t xbar = x0 + 64;        // softmax-warp exchange (one arrival per softmax warp)
  const uint32_t mma_drain = x0 + 72;   // every MMA of an issuer complete (x0 + 72: scores, + 80: output)
  // a head's merge: the other parts' (m, l) rows (+0) and their O^T halves, two parts in flight
  auto merge_bar = [&](int i) { return x0 + 88 + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::MISC_OFF + 4);

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int s = 0; s < kKST; ++s) {
      for (int h = 0; h < 2; ++h) {
        mbar_init(k_full(s, h), 32 * C::NLD);  // one cp.async arrive per loader thread
        mbar_init(k_empty(s, h), 1);
      }
    }
    for (int s = 0; s < kMST; ++s) {
      mbar_init(m_full(s), 1);
      mbar_init(m_empty(s), 2 + C::NSM + C::NLD);  // 2 MMA threads, softmax warps, loader warps
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(s_full(i), 1);
      mbar_init(s_empty(i), C::NSM);
      mbar_init(p_full(i), C::NSM);
      mbar_init(pv_done(i), 1);
    }
    mbar_init(xbar, C::NSM);
    mbar_init(mma_drain, 1);
    mbar_init(mma_drain + 8, 1);
    for (int i = 0; i < 3; ++i) mbar_init(merge_bar(i), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) prefetch_tmap(&tmap_q);
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
    // Walks this CTA's unit range segment by segment. The index window of a segment is read 256
    // entries per step (two steps ahead, block-table rows one step ahead); entries < 0 are
    // dropped and the valid ones packed, in index order, into dense 128-key tiles, so runs of
    // padding cost only their index reads and every emitted tile but a segment's last is full.
    uint32_t mc = 0, qc = 0;
    // range bounds of every CTA. A work-balanced split comes with a bound per CTA by valid
    // entries; they are spaced to at least split_gap units (so that a token spans few CTAs)
    // by a running maximum of bounds[c] - c * gap, capped at U - (G - c) * gap.
    int64_t* sb = reinterpret_cast<int64_t*>(smem + C::SPLIT_OFF);
    if (p.bounds) {
      const int64_t gap = p.split_gap;
      constexpr int kPer = (kSplitMaxCtas + 32) / 32;  // bounds per lane, in order
      int64_t v[kPer];
      int64_t run = INT64_MIN;
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const int c = kPer * lane + i;
        v[i] = c <= p.G ? p.bounds[c] - c * gap : INT64_MIN;
        run = v[i] > run ? v[i] : run;
        v[i] = run;
      }
      int64_t pre = INT64_MIN;  // running maximum of the lanes below
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
    auto emit_begin = [&](int& st) -> MetaHdr* {
      st = mc % kMST;
      if (mc >= (uint32_t)kMST) wait(m_empty(st), ((mc / kMST) & 1) ^ 1);
      return reinterpret_cast<MetaHdr*>(smem + C::META_OFF + st * C::META_BYTES);
    };
    auto emit_end = [&](int st) {
      __syncwarp();
      if (lane == 0) mbar_arrive(m_full(st));
      ++mc;
    };
    const int64_t pos_limit = p.bt ? (int64_t)p.max_pages * p.page_size : p.num_slots;
    int64_t u = u0;
    int64_t t = u0 / p.NT;       // token and tile of the CTA's first unit; later segments start
    int j0 = (int)(u0 - t * p.NT);  // at tile 0 of the next token
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
        if (!had) {  // Q of this segment, loaded with its first tile
          if (qc > 0) wait(q_empty, (qc - 1) & 1);
          if (lane == 0) mbar_arrive_expect_tx(q_full, C::Q_BYTES);
          __syncwarp();
          if (lane < kD / 64)
            tma_load_3d(sbase + C::Q_OFF + lane * (kH * 128), &tmap_q, 64 * lane, 0, (int)t, q_full);
          ++qc;
        }
        mh = emit_begin(st);
        slots = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(mh) + 32);
        if (lane == 0) {
          mh->type = kTile;
          mh->token = (int)t;
          mh->first = had ? 0 : 1;
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
      int* cbuf = reinterpret_cast<int*>(smem + C::CMP_OFF);
      for (int pos = e0; pos < e1 && !*abort_flag; pos += 32 * V) {
        int ic[V], pb[V];
        load_step(pos + 64 * V, ic);
        page_of(ib, pb);
        // compact this step's valid slots, in index order, into cbuf
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
        // move them into dense tiles of kBN keys
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
          int last = b;
          if (kind == kHead) {
            // the last CTA c whose range starts at or before the token's last unit L
            const int64_t L1 = (t + 1) * p.NT;
            if (p.bounds) {
              int lo = b, hi = p.G - 1;  // sb[lo] <= L1 - 1 holds; find the largest such c
              while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (sb[mid] <= L1 - 1) lo = mid;
                else hi = mid - 1;
              }
              last = lo;
            } else {
              // floor(c * U / G) <= L  <=>  c <= ceil((L + 1) * G / U) - 1
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
      j0 = 0;
    }
    {
      int st;
      MetaHdr* mh = emit_begin(st);
      if (lane == 0) mh->type = kDone;
      emit_end(st);
    }
    // no Q copy may still be in flight when the CTA exits
    if (qc > 0) mbar_wait(q_full, (qc - 1) & 1, kWaitNs);
  } else if (warp == 1 || warp == 2) {
    // ======================================================= MMA issuers (2 threads) ====
    // Warp 1 issues the score products, warp 2 the output products. Each is a short blocking
    // loop over the meta ring, so a tile whose probabilities are ready never waits behind the
    // next tile's score product (the tensor core takes both streams; their accumulators are
    // disjoint). Every MMA is straight-line code: one 32-bit add on each descriptor's low word.
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16(128, kH, 0, 0);   // A = K tile (K-major), B = Q (K-major)
      constexpr uint32_t idPV = idesc_bf16(128, kH, 1, 1);  // A = V^T (MN-major), B = P^T (MN-major)
      const uint64_t dq = sw128_desc(sbase + C::Q_OFF, 16, 1024);
      const uint32_t q_lo = (uint32_t)dq, q_hi = (uint32_t)(dq >> 32);
      const uint32_t k_hi = (uint32_t)(sw128_desc(0, 16, 1024) >> 32);
      const uint32_t mn_hi = (uint32_t)(sw128_desc(0, kBN * 128, 1024) >> 32);
      uint32_t mc = 0, g = 0, qc = 0;
      for (;;) {
        const int st = mc % kMST;
        if (!wait(m_full(st), (mc / kMST) & 1)) break;
        const MetaHdr* mh = reinterpret_cast<const MetaHdr*>(smem + C::META_OFF + st * C::META_BYTES);
        const int type = mh->type;
        const int first = mh->first, had = mh->had_tiles;
        mbar_arrive(m_empty(st));
        ++mc;
        if (type == kDone) break;
        if (type == kSegEnd) {
          // the segment's score products are all issued: its Q buffer is free once they complete
          if (warp == 1 && had) mma_commit(q_empty);
          continue;
        }
        const int ks = g % kKST;
        if (warp == 1) {
          // ---- scores S^T = K Q^T for tile g
          if (first) {
            if (!wait(q_full, qc & 1)) break;
            ++qc;
          }
          if (g >= 2 && !wait(s_empty(g & 1), ((g >> 1) & 1) ^ 1)) break;
          const uint32_t k_lo = (uint32_t)sw128_desc(sbase + C::KT_OFF + ks * C::KT_BYTES, 16, 1024);
          const uint32_t d0 = tmem + (g & 1) * C::S_COLS;
          // 16-column step kk: chunk kk/4 of 64 columns, 32 bytes per step inside the chunk
          auto step = [&](int kk) {
            const uint32_t ka = (uint32_t)((kk >> 2) * ((kBN * 128) >> 4) + (kk & 3) * 2);
            const uint32_t qa = (uint32_t)((kk >> 2) * ((kH * 128) >> 4) + (kk & 3) * 2);
            if (kk == 0) mma_bf16_lohi<0>(d0, k_lo + ka, k_hi, q_lo + qa, q_hi, idS);
            else mma_bf16_lohi<1>(d0, k_lo + ka, k_hi, q_lo + qa, q_hi, idS);
          };
          // the first column half's products start while the loaders write the second half
          if (!wait(k_full(ks, 0), (g / kKST) & 1)) break;
          // rows arrive by cp.async (generic proxy): order them before the tensor core reads
          fence_proxy_async_smem();
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kD / 32; ++kk) step(kk);
          if (!wait(k_full(ks, 1), (g / kKST) & 1)) break;
          fence_proxy_async_smem();
          tc_fence_after();
#pragma unroll
          for (int kk = kD / 32; kk < kD / 16; ++kk) step(kk);
          mma_commit(s_full(g & 1));
        } else {
          // ---- output O^T += V^T P^T for tile g, once its probabilities are written
          if (!wait(p_full(g % C::PBUF), (g / C::PBUF) & 1)) break;
          tc_fence_after();
          // V^T: 64-column groups of the K tile are 128 * 128 bytes apart (LBO), 8-key groups 1024
          const uint32_t v_lo = (uint32_t)sw128_desc(sbase + C::KT_OFF + ks * C::KT_BYTES, kBN * 128, 1024);
          const uint32_t p_lo = (uint32_t)sw128_desc(sbase + C::P_OFF + (g % C::PBUF) * C::P_BYTES, kBN * 128, 1024);
          // output columns 128h .. 128h + 127 (V^T two 64-column groups further); 16 keys per
          // step (16 rows of 128 bytes)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t d = tmem + C::O_COL + 64 * h;
            const uint32_t va = v_lo + h * ((2 * kBN * 128) >> 4);
            const uint32_t pa = p_lo;
            // the first step of a segment's first tile overwrites the accumulator
            mma_bf16(d, ((uint64_t)mn_hi << 32) | va, ((uint64_t)mn_hi << 32) | pa, idPV, first ? 0u : 1u);
#pragma unroll
            for (int j = 1; j < kBN / 16; ++j) mma_bf16_lohi<1>(d, va + 128 * j, mn_hi, pa + 128 * j, mn_hi, idPV);
            // d_v half h has read columns 128h .. 128h + 127 of the K tile: that half is free
            mma_commit(k_empty(ks, h));
          }
          mma_commit(pv_done(g & 1));
        }
        ++g;
      }
      // drain: every MMA issued by this thread completes before TMEM can be released
      const uint32_t drain = warp == 1 ? mma_drain : mma_drain + 8;
      mma_commit(drain);
      mbar_wait(drain, 0, kWaitNs);
    }
    __syncwarp();
  } else if (warp >= 4 && warp < 4 + C::NSM) {  // (softmax)
    // ============================================= softmax + epilogue (8 warps) ====
    // Thread = key of the tile = TMEM lane (quarter warp % 4); the two warps of a quarter take
    // heads 0-31 and 32-63. Per tile one pass computes, with the running max m_h of each head,
    // x = c * score - m_h, p = 2^x, the per-lane partial row sums (TMEM, two buffers: the pass
    // reads one and writes the other) and the probability rows of P. A vote of the warps
    // then checks that no x exceeded 8; if one did (rare after a segment's first tile), the
    // tile takes exact per-head maxima, raises m_h where it grew by more than 2^8, rescales O
    // and the partial sums of those heads, and is redone. A segment's first tile starts there.
    const int sm = warp - 4;                                 // softmax warp index
    const int qd = warp & 3;                                 // TMEM lane quarter
    const int hb = C::HW * (sm >> 2);                          // first head of this warp
    const int tr = 32 * qd + lane;                           // key row of the tile / dv row of O^T
    const int sid = 32 * sm + lane;                          // softmax thread index
    const uint32_t tl = tmem + ((uint32_t)(32 * qd) << 16);  // this warp's lanes
    float* red = reinterpret_cast<float*>(smem + C::RED_OFF);
    float* red_m = red;           // running max per head (exp2 domain)
    float* red_alpha = red + 64;  // rescale factor per head; epilogue: weight of own partial
    float* red_part = red + 256;  // [4 lane quarters][64 heads]
    float* red_wk = red + 512;    // [kMaxParts][64]: merge weights of the other parts
    int* votes = reinterpret_cast<int*>(red + 512 + kMaxParts * kH);  // [2][C::NSM]
    uint32_t mc = 0, g = 0, xc = 0, lb = 0;
    auto xsync = [&](bool v) -> int {
      const int r = softmax_exchange<C::NSM>(xbar, votes, xc++, sm, v ? 1 : 0);
      if (r < 0) fail(DSA_DEVERR_TIMEOUT);
      return r;
    };
    auto wait_all = [&](bool ok) -> bool {
      if (__all_sync(0xffffffffu, ok)) return true;
      fail(DSA_DEVERR_TIMEOUT);
      return false;
    };
    // every PV product up to tile `last` (inclusive) complete
    auto pv_wait = [&](int64_t last) -> bool {
      if (last < 0) return true;
      return mbar_wait(pv_done((uint32_t)last & 1), ((uint32_t)last >> 1) & 1, kWaitNs);
    };
    for (;;) {
      const int st = mc % kMST;
      if (!wait_all(mbar_wait(m_full(st), (mc / kMST) & 1, kWaitNs))) break;
      const MetaHdr* mh = reinterpret_cast<const MetaHdr*>(smem + C::META_OFF + st * C::META_BYTES);
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
        bool ok = mbar_wait(s_full(g & 1), (g >> 1) & 1, kWaitNs);
        // the P buffer must be free: the PV product that read it last is complete
        ok = ok && pv_wait((int64_t)g - C::PBUF);
        if (!wait_all(ok)) break;
        tc_fence_after();
        const bool valid = tr < n_valid;
        const float c0 = p.c_log2;
        const uint32_t sa = tl + (g & 1) * C::S_COLS + hb;
        const uint32_t lcur = tl + C::L_COL + 64 * lb + hb, lnxt = tl + C::L_COL + 64 * (lb ^ 1) + hb;
        uint8_t* prow = smem + C::P_OFF + (g % C::PBUF) * C::P_BYTES + tr * 128;
        const int sw = tr & 7;
        // score of head i of a chunk, exp2 domain, before subtracting the running max
        auto score = [&](const uint32_t (&a)[16], int i) -> float { return u2f(a[i]) * c0; };
        bool exact = first != 0, bad = false;
        for (;;) {
          bool resc = false;
          if (exact) {
            // exact per-head maximum of this tile: warp max-reductions over the keys, then
            // across the four lane quarters
#pragma unroll 1
            for (int ch = 0; ch < C::CH; ++ch) {
              uint32_t a[16];
              tmem_ld32_x16(sa + 16 * ch, a);
              tc_wait_ld();
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const int mx = redux_max_s32(f2ord(valid ? score(a, i) : -INFINITY));
                if (lane == ((16 * ch + i) & 31)) red_part[qd * 64 + hb + 16 * ch + i] = ord2f(mx);
              }
            }
            if (xsync(false) < 0) { bad = true; break; }
            bool grow_any = false;
            if (sid < kH) {
              const float mt = fmaxf(fmaxf(red_part[sid], red_part[64 + sid]), fmaxf(red_part[128 + sid], red_part[192 + sid]));
              const float mo = first ? -INFINITY : red_m[sid];
              const bool grow = first || mt > mo + 8.0f;
              const float mn = grow ? mt : mo;
              red_alpha[sid] = grow ? ex2_approx(mo - mn) : 1.0f;
              red_m[sid] = mn;
              grow_any = grow && !first;
            }
            const int r = xsync(grow_any);
            if (r < 0) { bad = true; break; }
            resc = r != 0;
          }
          if (resc) {
            // rare: some head's max grew; scale its O^T columns (every issued PV complete)
            if (!wait_all(pv_wait((int64_t)g - 1))) { bad = true; break; }
            tc_fence_after();
#pragma unroll 1
            for (int ch = 0; ch < C::CH; ++ch) {
              uint32_t o0[16], o1[16], lv[16];
              tmem_ld32_x16(tl + C::O_COL + hb + 16 * ch, o0);
              tmem_ld32_x16(tl + C::O_COL + 64 + hb + 16 * ch, o1);
              tmem_ld32_x16(lcur + 16 * ch, lv);
              tc_wait_ld();
              const float* al = red_alpha + hb + 16 * ch;
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                o0[i] = f2u(u2f(o0[i]) * al[i]);
                o1[i] = f2u(u2f(o1[i]) * al[i]);
                lv[i] = f2u(u2f(lv[i]) * al[i]);
              }
              tmem_st32_x16(tl + C::O_COL + hb + 16 * ch, o0);
              tmem_st32_x16(tl + C::O_COL + 64 + hb + 16 * ch, o1);
              tmem_st32_x16(lcur + 16 * ch, lv);  // the partial sums the pass reads next
            }
            tc_wait_st();
          }
          // the pass: p = 2^(c * score - m) (one FFMA and one MUFU ex2 per score), partial row
          // sums into the other TMEM buffer (a rescale has already scaled the buffer it reads),
          // and P as bf16 into this key's 128-byte row
          float xm = -INFINITY;
#pragma unroll 1
          for (int ch = 0; ch < C::CH; ++ch) {
            float mv[16];  // running maxima of the chunk's heads, read ahead of the TMEM wait
#pragma unroll
            for (int i = 0; i < 16; i += 4)
              *reinterpret_cast<float4*>(mv + i) = *reinterpret_cast<const float4*>(red_m + hb + 16 * ch + i);
            uint32_t a[16], l[16];
            tmem_ld32_x16(sa + 16 * ch, a);
            if (!first) tmem_ld32_x16(lcur + 16 * ch, l);
            tc_wait_ld();
            float pr[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float x = score(a, i) - mv[i];
              xm = fmaxf(xm, valid ? x : -INFINITY);
              pr[i] = valid ? ex2_approx(x) : 0.0f;
              float lv = pr[i];
              if (!first) lv = u2f(l[i]) + pr[i];
              l[i] = f2u(lv);
            }
            tmem_st32_x16(lnxt + 16 * ch, l);
            const int g0 = (hb >> 3) + 2 * ch;  // 16-byte granules of this chunk's 16 heads
            uint32_t w[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) w[i] = f32x2_to_bf16x2(pr[2 * i], pr[2 * i + 1]);
            *reinterpret_cast<uint4*>(prow + ((g0 ^ sw) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
            *reinterpret_cast<uint4*>(prow + (((g0 + 1) ^ sw) << 4)) = make_uint4(w[4], w[5], w[6], w[7]);
          }
          if (exact) break;
          const int r = xsync(xm > 8.0f);
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
          mbar_arrive(p_full(g % C::PBUF));
          mbar_arrive(s_empty(g & 1));
        }
        ++g;
        continue;
      }
      // ====================================================== kSegEnd: token epilogue ====
      const int64_t t = mh->token;
      const int kind = mh->kind, had = mh->had_tiles, last = mh->merge_last;
      __syncwarp();
      if (lane == 0) mbar_arrive(m_empty(st));
      ++mc;
      // the row sums need only the partial-sum buffer the last pass wrote (this warp's own
      // TMEM stores, complete before it signalled P): they run while the last output product
      // may still be in flight, and O is read only after it
      const uint32_t lfin = tl + C::L_COL + 64 * lb + hb;  // the buffer the last pass wrote
      // row sums: per warp, a reduce-scatter over the lanes (keys) of each 16-head chunk leaves
      // the warp's sum of head 16 ch + (lane >> 1) in lanes 2i and 2i + 1 (each round halves the
      // values a lane holds: it keeps one half, adds its partner's copy of that half, and hands
      // over the other); lane 2i writes it to red_part[quarter][head], and thread h < 64 adds
      // up the quarters
#pragma unroll 1
      for (int ch = 0; ch < C::CH; ++ch) {
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
      float lsum = 0.0f, mrow = -INFINITY;
      if (sid < kH && had) {
        lsum = (red_part[sid] + red_part[64 + sid]) + (red_part[128 + sid] + red_part[192 + sid]);
        mrow = red_m[sid];
      }
      // the quarter sums are read before a next tile's exact path rewrites them: a part publishes
      // and moves on, so it needs its own exchange here; the other kinds pass the weights'
      // exchange below after their last read
      if (kind == kPart && xsync(false) < 0) break;
      if (had) {
        if (!wait_all(pv_wait((int64_t)g - 1))) break;
        tc_fence_after();
      }
      if (kind == kPart) {
        // publish (O^T, m, l) of this part in workspace slot b
        if (sid < kH) {
          p.ws_ml[((int64_t)b * 2 + 0) * kH + sid] = mrow;
          p.ws_ml[((int64_t)b * 2 + 1) * kH + sid] = lsum;
        }
        if (had) {
          // rows dv = tr and 128 + tr of O^T; the 16-byte granule of heads 4q .. 4q + 3 sits at
          // position q ^ (tr & 15) of its 256-byte row, so that the merge reads the rows from
          // shared memory without bank conflicts
          float* w0 = p.ws_o + ((int64_t)b * kD + tr) * kH;
          float* w1 = p.ws_o + ((int64_t)b * kD + 128 + tr) * kH;
#pragma unroll 1
          for (int ch = 0; ch < C::CH; ++ch) {
            uint32_t o0[16], o1[16];
            tmem_ld32_x16(tl + C::O_COL + hb + 16 * ch, o0);
            tmem_ld32_x16(tl + C::O_COL + 64 + hb + 16 * ch, o1);
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
      // every publish flag of parts b+1 .. last, one per lane (a warp vote ends the wait); the
      // warp barrier then orders every lane's reads of the parts after the acquiring loads
      for (int f0 = 0; f0 < nparts * C::NSM && okp; f0 += 32) {
        const int f = f0 + lane;
        const bool mine = f < nparts * C::NSM;
        const int* fp = p.flags + 8 * (b + 1 + f / C::NSM) + f % C::NSM;
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
      // (the launch keeps nparts <= kMaxParts; more would overrun the weight table)
      const int np = (okp && nparts <= kMaxParts) ? nparts : 0;
      // The parts' rows come into shared memory by bulk copies: their (m, l) rows (consecutive
      // workspace slots b+1 .. b+np) into the Q buffer, and their O^T halves into two slot
      // pairs of the K stages, two parts in flight. A head segment is its CTA's last, so none of
      // these buffers is in use any more: every output product is complete, and no further Q
      // load or row load follows.
      auto slot = [&](int pair, int half) -> uint32_t { return sbase + C::KT_OFF + (2 * pair + half) * (128 * kH * 4); };
      auto fetch_part = [&](int u) {  // one thread: fill u = part u % np + 1 into slot pair u & 1
        const uint32_t mb = merge_bar(1 + (u & 1));
        const float* src = p.ws_o + (int64_t)(b + 1 + u % np) * kD * kH;
        mbar_arrive_expect_tx(mb, kD * kH * 4);
        bulk_g2s(slot(u & 1, 0), src, 128 * kH * 4, mb);
        bulk_g2s(slot(u & 1, 1), src + 128 * kH, 128 * kH * 4, mb);
      };
      if (np > 0 && sid == 0) {
        // the flags were acquired by this warp; order the parts' data (read by the async proxy)
        // after them, and the buffers' earlier uses before the copies
        asm volatile("fence.proxy.async.global;" ::: "memory");
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(merge_bar(0), np * 2 * kH * 4);
        bulk_g2s(sbase + C::Q_OFF, p.ws_ml + (int64_t)(b + 1) * 2 * kH, np * 2 * kH * 4, merge_bar(0));
        fetch_part(0);
        if (np >= 2) fetch_part(1);
      }
      if (sid < kH) {
        const float* pml = reinterpret_cast<const float*>(smem + C::Q_OFF);  // [np][2][64]
        if (np > 0 && !mbar_wait(merge_bar(0), 0, kWaitNs)) fail(DSA_DEVERR_TIMEOUT);
        float M = mrow;
        for (int k = 1; k <= np; ++k) M = fmaxf(M, pml[(k - 1) * 2 * kH + sid]);
        const float w_own = lsum > 0.0f ? exp2f(mrow - M) : 0.0f;
        float L = w_own * lsum;
        for (int k = 1; k <= np; ++k) {
          const float mk = pml[((k - 1) * 2 + 0) * kH + sid];
          const float lk = pml[((k - 1) * 2 + 1) * kH + sid];
          const float wk = lk > 0.0f ? exp2f(mk - M) : 0.0f;
          red_wk[(k - 1) * kH + sid] = wk;
          L += wk * lk;
        }
        const float inv = L > 0.0f ? 1.0f / L : 0.0f;
        red_alpha[sid] = w_own * inv;
        for (int k = 1; k <= np; ++k) red_wk[(k - 1) * kH + sid] *= inv;
        if (p.lse) p.lse[t * kH + sid] = L > 0.0f ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
      }
      if (xsync(false) < 0) break;
      // combine: this CTA's O (TMEM) and the parts in order, then stage the bf16 block
      // [64 heads][256 columns] in the (idle) P buffers
      uint16_t* stage = reinterpret_cast<uint16_t*>(smem + C::P_OFF);
      // One 16-head chunk at a time (32 accumulators): the parts stream through the two slot
      // pairs in order, and with more than two parts the second chunk fetches them again.
      bool okm = true;
      int uses = 0;  // slot-pair fills consumed so far (fill u is part (u % np) + 1 in pair u & 1)
#pragma unroll 1
      for (int ch = 0; ch < C::CH && okm; ++ch) {
        const int h0 = hb + 16 * ch;
        if (np <= 2) uses = 0;  // both parts stay in their slot pairs for the second chunk
        float acc0[16], acc1[16];
        const float* wo = red_alpha + h0;
        if (had) {
          uint32_t o0[16], o1[16];
          tmem_ld32_x16(tl + C::O_COL + h0, o0);
          tmem_ld32_x16(tl + C::O_COL + 64 + h0, o1);
          tc_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            acc0[i] = wo[i] * u2f(o0[i]);
            acc1[i] = wo[i] * u2f(o1[i]);
          }
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) acc0[i] = acc1[i] = 0.0f;
        }
        for (int k = 1; k <= np; ++k, ++uses) {
          const int pr = uses & 1;
          if (!wait_all(mbar_wait(merge_bar(1 + pr), (uses >> 1) & 1, kWaitNs))) {
            okm = false;
            break;
          }
          const uint8_t* r0 = smem + (slot(pr, 0) - sbase) + tr * 256;
          const uint8_t* r1 = smem + (slot(pr, 1) - sbase) + tr * 256;
          const float* wk = red_wk + (k - 1) * kH + h0;
#pragma unroll
          for (int i = 0; i < 16; i += 4) {
            const int pos = 16 * ((((h0 + i) >> 2) ^ tr) & 15);
            const float4 x = *reinterpret_cast<const float4*>(r0 + pos);
            const float4 y = *reinterpret_cast<const float4*>(r1 + pos);
            acc0[i] += wk[i] * x.x;
            acc0[i + 1] += wk[i + 1] * x.y;
            acc0[i + 2] += wk[i + 2] * x.z;
            acc0[i + 3] += wk[i + 3] * x.w;
            acc1[i] += wk[i] * y.x;
            acc1[i + 1] += wk[i + 1] * y.y;
            acc1[i + 2] += wk[i + 2] * y.z;
            acc1[i + 3] += wk[i + 3] * y.w;
          }
          // the fill two ahead: the next part of this chunk's pass, or of the second chunk's
          const int ahead = uses + 2, total = np > 2 ? C::CH * np : np;
          if (ahead < total) {
            // every warp has read this slot pair: refill it
            if (xsync(false) < 0) {
              okm = false;
              break;
            }
            if (sid == 0) {
              fence_proxy_async_smem();
              fetch_part(ahead);
            }
          }
        }
        if (!okm) break;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          stage[(h0 + i) * kD + tr] = __bfloat16_as_ushort(__float2bfloat16_rn(acc0[i]));
          stage[(h0 + i) * kD + 128 + tr] = __bfloat16_as_ushort(__float2bfloat16_rn(acc1[i]));
        }
      }
      if (!okm) break;
      if (xsync(false) < 0) break;
      // every softmax warp has read the parts: clear their publish flags, so that the workspace
      // holds no set flag after the call (a later call that carries the same tag, such as a
      // replay of a recorded launch, then never mistakes this call's flags for its own)
      for (int f = sid; f < np * C::NSM; f += 32 * C::NSM) p.flags[8 * (b + 1 + f / C::NSM) + f % C::NSM] = 0;
      // copy out: 2048 16-byte granules (64 rows of 512 bytes), 8 per thread, row-contiguous
      {
        uint16_t* orow = p.out + t * p.out_st;
#pragma unroll 4
        for (int j = 0; j < 2048 / (32 * C::NSM); ++j) {
          const int q = sid + 32 * C::NSM * j, h = q >> 5, gq = q & 31;
          *reinterpret_cast<uint4*>(orow + (int64_t)h * p.out_sh + gq * 8) =
              *reinterpret_cast<const uint4*>(stage + h * kD + gq * 8);
        }
      }
      tc_fence_before();
    }
  } else if (C::loader_index(warp) >= 0) {
    // ================================================= row loaders (5 warps) ====
    // Warp dw fills rows dw + C::NLD * k (k < nk) of each K tile in the 128-byte-swizzled K-major
    // layout (row r, 16-byte granule q of 64-column chunk c at c*128*128 + r*128 + ((q ^ (r&7)) << 4)).
    // A tile is written in two column halves, columns 0-127 (chunks 0-1) and 128-255 (chunks
    // 2-3), each with its own full and empty barrier: the score product starts on the first half
    // while the second is written, and a stage's first half is refilled as soon as the output
    // product's first d_v half has read it. Rows are taken in pairs (lanes 0-15: row 2p,
    // 16-31: row 2p + 1); lane il of a half warp handles 16-byte granule 16h + il of its row, so
    // the eight lanes of a quarter warp store to eight different 16-byte positions.
    // Rows past n_valid are zero (their keys are masked: a zero row keeps 0 * V finite).
    const int dw = C::loader_index(warp);
    const int nk = (kBN - dw + C::NLD - 1) / C::NLD;  // rows of this warp per tile: dw + C::NLD * k, k < nk
    // lane t holds the slot of row dw + NLD * t
    static_assert(C::NR <= 32, "a warp's rows of a tile fit its lanes");
    const int hl = lane >> 4, il = lane & 15;
    uint32_t mc = 0, g = 0;
    auto next_tile = [&](bool block, int& st_out) -> int {
      while (!*abort_flag) {
        const int st = mc % kMST;
        if (!block && !mbar_test(m_full(st), (mc / kMST) & 1)) return -1;
        if (!wait(m_full(st), (mc / kMST) & 1)) return 0;
        const MetaHdr* mh = reinterpret_cast<const MetaHdr*>(smem + C::META_OFF + st * C::META_BYTES);
        const int type = mh->type;
        if (type == kTile) {
          st_out = st;
          return 1;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(m_empty(st));
        ++mc;
        if (type == kDone) return 0;
      }
      return 0;
    };
    // tile in meta slot st: row count and lane t's slot of row dw + C::NLD * t (-1 past the
    // valid rows). Everything the loader needs of the entry is then in registers: the caller
    // releases the meta stage right away, and a copy takes the slot of row k from lane k by a
    // shuffle.
    auto take = [&](int st, int& n, int& slr) {
      const MetaHdr* mh = reinterpret_cast<const MetaHdr*>(smem + C::META_OFF + st * C::META_BYTES);
      n = mh->n_valid;
      const int* slots = reinterpret_cast<const int*>(reinterpret_cast<const uint8_t*>(mh) + 32);
      const int rt = dw + C::NLD * lane;
      slr = -1;
      if (lane < nk && rt < n) slr = slots[rt];
    };
    auto release = [&]() {
      __syncwarp();
      if (lane == 0) mbar_arrive(m_empty(mc % kMST));
      ++mc;
    };
    {
      // 16-byte cp.async straight into the tile, one row pair per instruction; each thread's
      // copies of a half signal that half's full barrier when they land
      int st = 0, n = 0, slr = -1;
      bool bad = false;
      while (!bad && next_tile(true, st) == 1) {
        take(st, n, slr);
        release();
        const int ks = g % kKST;
        uint8_t* kt = smem + C::KT_OFF + ks * C::KT_BYTES;
        for (int h = 0; h < 2; ++h) {
          if (g >= (uint32_t)kKST && !wait(k_empty(ks, h), ((g / kKST) & 1) ^ 1)) {
            bad = true;
            break;
          }
          const int G = 16 * h + il;
#pragma unroll
          for (int pp = 0; pp < (C::NR + 1) / 2; ++pp) {
            const int k = 2 * pp + hl;
            const int sl = __shfl_sync(0xffffffffu, slr, k);
            if (k < nk) {
              const int r = dw + C::NLD * k;
              const uint8_t* src = p.cache + (sl >= 0 ? (int64_t)sl : 0) * C::RB + 16 * G;
              const uint32_t dst = smem_u32(kt + (G >> 3) * (kBN * 128) + r * 128 + (((G & 7) ^ (r & 7)) << 4));
              asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(sl >= 0 ? 16 : 0)
                           : "memory");
            }
          }
          asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(k_full(ks, h)) : "memory");
        }
        ++g;
      }
    }
    // drain this thread's outstanding cp.async copies before the CTA can finish
    asm volatile("cp.async.wait_all;" ::: "memory");
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ------------------------------------------------------------- work-balanced split --
// Units (token, 128-entry window) carry very different work when the index lists are uneven
// (causal prefill: the early tokens' windows are mostly padding). Two small kernels turn the
// lists into per-CTA range bounds by work (non-empty tiles plus a fixed amount per token), so
// that every CTA gets about the same work. Both read only the index lists; the bounds depend on nothing else, so a split
// (and so the result) is the same on every call.

// Work of units u0 .. u0 + 7 (unit u: window [128 j, 128 j + 128) of token u / NT): a full tile
// if any entry is >= 0 (a token's valid entries are packed into dense tiles, and a tile costs the
// same however full), plus the token's fixed work on its first unit; 0 past u1. The warp reads
// each window's 128 entries (four per lane), all eight windows' loads in flight at once.
constexpr int kUnitBatch = 8;
__device__ __forceinline__ void unit_work8(const int32_t* idx, int64_t idx_stride, int topk, int NT, int64_t u0,
                                           int64_t u1, int lane, int (&w)[kUnitBatch]) {
  int v[kUnitBatch][4];
#pragma unroll
  for (int q = 0; q < kUnitBatch; ++q) {
    const int64_t u = u0 + q;
    const int64_t t = u / NT;
    const int j = (int)(u - t * NT);
    const int32_t* row = idx + t * idx_stride;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int e = kBN * j + 32 * k + lane;
      v[q][k] = (u < u1 && e < topk) ? __ldg(row + e) : -1;
    }
  }
#pragma unroll
  for (int q = 0; q < kUnitBatch; ++q) {
    const int64_t u = u0 + q;
    const int64_t t = u / NT;
    const int j = (int)(u - t * NT);
    const bool any = (v[q][0] & v[q][1] & v[q][2] & v[q][3]) >= 0;  // not every sign bit set: some entry >= 0
    const bool hit = __any_sync(0xffffffffu, any);
    w[q] = u < u1 ? (hit ? kBN : 0) + (j == 0 ? kSegmentWeight : 0) : 0;
  }
}

// warp s: work of slice s = units [s U / S, (s + 1) U / S)
__global__ void __launch_bounds__(1024) split_count_kernel(const int32_t* __restrict__ idx, int64_t idx_stride, int topk,
                                                           int NT, int64_t U, int S, int64_t* __restrict__ tot) {
  const int lane = threadIdx.x & 31;
  const int s = blockIdx.x * 32 + (threadIdx.x >> 5);
  if (s >= S) return;
  const int64_t u0 = (int64_t)s * U / S, u1 = (int64_t)(s + 1) * U / S;
  int64_t c = 0;
  for (int64_t u = u0; u < u1; u += kUnitBatch) {
    int w[kUnitBatch];
    unit_work8(idx, idx_stride, topk, NT, u, u1, lane, w);
#pragma unroll
    for (int q = 0; q < kUnitBatch; ++q) c += w[q];
  }
  if (lane == 0) tot[s] = c;
}

// block b: bounds[b] = the first unit u with G * (work of the units before u) >= b * W (W: all
// the work); bounds[0] = 0, bounds[G] = U
__global__ void __launch_bounds__(256) split_bounds_kernel(const int32_t* __restrict__ idx, int64_t idx_stride, int topk,
                                                           int NT, int64_t U, int S, int G,
                                                           const int64_t* __restrict__ tot, int64_t* __restrict__ bounds) {
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (b == 0 || b == G) {
    if (tid == 0) bounds[b] = b == 0 ? 0 : U;
    return;
  }
  __shared__ int64_t part[256];
  __shared__ int64_t sel_slice, sel_base;
  // each thread takes a run of consecutive slices; an exclusive scan of the run sums gives
  // every slice's prefix
  const int per = (S + 255) / 256, s0 = min(S, tid * per), s1 = min(S, s0 + per);
  int64_t mine = 0;
  for (int s = s0; s < s1; ++s) mine += tot[s];
  part[tid] = mine;
  __syncthreads();
  if (tid == 0) {
    int64_t run = 0;
    for (int i = 0; i < 256; ++i) {
      const int64_t x = part[i];
      part[i] = run;
      run += x;
    }
    sel_base = run;  // W for now
    sel_slice = S;
  }
  __syncthreads();
  const int64_t W = sel_base, target = (int64_t)b * W;
  __syncthreads();
  // the slice holding the crossing: the first s with G * (prefix through s) >= b W
  {
    int64_t pre = part[tid];
    for (int s = s0; s < s1; ++s) {
      const int64_t after = pre + tot[s];
      if ((int64_t)G * after >= target) {
        atomicMin(reinterpret_cast<unsigned long long*>(&sel_slice), (unsigned long long)s);
        break;
      }
      pre = after;
    }
  }
  __syncthreads();
  const int64_t s = sel_slice;
  if (warp != 0) return;
  if (s >= S) {  // no crossing (W == 0): every unit counts the same
    if (lane == 0) bounds[b] = (int64_t)b * U / G;
    return;
  }
  // prefix before slice s, then walk its units
  int64_t cum = 0;
  {
    const int per_s = (S + 31) / 32;
    for (int i = lane * per_s; i < min(S, (lane + 1) * per_s) && i < s; ++i) cum += tot[i];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cum += __shfl_xor_sync(0xffffffffu, cum, o);
  }
  const int64_t u0 = s * U / S, u1 = (s + 1) * U / S;
  int64_t bound = u1;
  for (int64_t ub = u0; ub < u1; ub += 32) {  // 32 units a round; lane i then holds unit ub + i's work
    const int64_t u = ub + lane;
    int c = 0;
#pragma unroll 1
    for (int b8 = 0; b8 < 32; b8 += kUnitBatch) {
      int w[kUnitBatch];
      unit_work8(idx, idx_stride, topk, NT, ub + b8, u1, lane, w);
#pragma unroll
      for (int q = 0; q < kUnitBatch; ++q)
        if (lane == b8 + q) c = w[q];
    }
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int x = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += x;
    }
    const unsigned hit = __ballot_sync(0xffffffffu, u < u1 && (int64_t)G * (cum + incl - c) >= target);
    if (hit) {
      bound = ub + __ffs(hit) - 1;
      break;
    }
    cum += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) bounds[b] = bound;
}

}  // namespace k128

dsa_status_t plan_unit_split(const dsa_attn_args_t* a, const DeviceInfo& dev, const AttnWorkspace& ws,
                             cudaStream_t stream, UnitSplit* out) {
  using namespace k128;
  UnitSplit r;
  r.NT = (a->topk + kBN - 1) / kBN;
  r.U = a->T * (int64_t)r.NT;
  // one persistent CTA per SM, with at least 4 units per CTA (a small batch spreads over
  // several CTAs per token, whose parts the head CTA merges from bulk copies in shared memory:
  // four units each measured faster than two for 8 and 17 tokens, fewer parts to merge against
  // two more tiles), and few enough CTAs that a token spans at most kMaxParts + 1 of them
  int64_t G = (r.U + 3) / 4;
  if (G > dev.sm_count) G = dev.sm_count;
  {
    // when every token can have the same whole number of CTAs, the ranges fall on token
    // boundaries: no CTA holds the end of one token and the start of the next (two epilogues)
    const int64_t k = r.NT / 4 > 0 ? r.NT / 4 : 1;
    if (a->T * k <= dev.sm_count) G = a->T * k;
  }
  while (G > 1) {
    const int64_t upc = r.U / G;  // fewest units any CTA holds
    if ((r.NT + upc - 1) / upc + 1 <= kMaxParts + 1) break;
    --G;
  }
  r.G = (int)G;
  // Work-balanced split when CTAs hold many units (long, possibly uneven index lists): two small
  // kernels on the same stream turn the lists into range bounds by work. Ranges keep at
  // least ceil(NT / (kMaxParts - 1)) units, so that a token still spans at most kMaxParts CTAs.
  r.bounds = nullptr;
  r.gap = 1;
  const int64_t gap = (r.NT + kMaxParts - 2) / (kMaxParts - 1);
  if (r.G > 1 && r.G <= kSplitMaxCtas && r.U / r.G >= 64 && r.U >= (int64_t)r.G * gap) {
    const int S = kSplitSlices * r.G;
    int64_t* tot = ws.split;
    int64_t* bnd = ws.split + S;
    split_count_kernel<<<r.G, 1024, 0, stream>>>(a->indices, a->idx_stride_t, a->topk, r.NT, r.U, S, tot);
    split_bounds_kernel<<<r.G + 1, 256, 0, stream>>>(a->indices, a->idx_stride_t, a->topk, r.NT, r.U, S, r.G, tot,
                                                     bnd);
    const cudaError_t le = cudaGetLastError();
    if (le != cudaSuccess) return cuda_fail(le);
    r.bounds = bnd;
    r.gap = (int)gap;
  }
  *out = r;
  return DSA_OK;
}

namespace k128 {

static dsa_status_t launch(const dsa_attn_args_t* a, const DeviceInfo& dev, cudaStream_t stream) {
  using C = Cfg;
  CUtensorMap tq;
  dsa_status_t st = encode_q_tensor_map(a, kD, &tq);
  if (st != DSA_OK) return st;

  Params p{};
  p.cache = static_cast<const uint8_t*>(a->cache);
  p.num_slots = a->num_slots;
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
  st = plan_unit_split(a, dev, ws, stream, &us);
  if (st != DSA_OK) return st;
  p.NT = us.NT;
  p.U = us.U;
  p.G = us.G;
  p.bounds = us.bounds;
  p.split_gap = us.gap;

  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)p.G);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, attn_k128_kernel, p, tq);
  return e == cudaSuccess ? DSA_OK : cuda_fail(e);
}

}  // namespace k128

cudaError_t k128_set_attributes() {
  return cudaFuncSetAttribute(k128::attn_k128_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              k128::Cfg::SMEM_BYTES);
}

dsa_status_t launch_attn_k128(const dsa_attn_args_t* a, const DeviceInfo& dev, cudaStream_t stream) {
  if (a->kind == DSA_CACHE_BF16) return k128::launch(a, dev, stream);
  return launch_attn_f8(a, dev, stream);
}

}  // namespace dsa
