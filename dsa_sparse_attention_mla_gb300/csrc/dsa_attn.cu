// dsa_attn.cu - DSA sparse MLA attention forward for sm_103a (tcgen05 + TMEM + TMA): the
// entry points (argument checks, dispatch, workspace, fixed-scratch variant), the host pieces
// shared with the other attention files, and the kernel of the 512+64 control geometry over a
// bf16 cache. The 256+0 geometry runs in dsa_attn_k128.cu (bf16) and dsa_attn_f8.cu (FP8), the
// 512+64 geometry over the packed FP8 cache in dsa_attn_ctl.cu.
//
// What is computed (sglang PR #38547 "Enable zero-RoPE TileLang DSA on gfx950", Summary and
// Direct GLM geometry coverage list): for every query token t and head h, gather the latent
// rows named by t's top-k index list (entries < 0 masked), score s_j = sm_scale * q[t,h].k_j,
// softmax over j and return sum_j p_j * k_j[0:d_v] in bf16. The cache holds bf16 rows or the
// packed scaled-FP8 rows of the Contract table (codes * per-128-tile fp32 scale).
//
// 512+64 bf16 kernel design:
//  * Heads are the MMA M dimension (M = 64), gathered keys are N: S = Q K^T (K-dim = d) and
//    O += P V (K-dim = keys, V = the first d_v columns of the same gathered rows) are dense
//    tcgen05 kind::f16 contractions with fp32 accumulators in tensor memory. The M = 64
//    accumulator occupies TMEM lanes 32*w + [0,16) of each sub-partition w. d_v = 512 runs as
//    two 256-column passes (TMEM holds O for 256 columns at a time).
//  * One persistent CTA per SM, launched cooperatively. The (token, key-tile) units are split
//    into equal contiguous ranges, one per CTA ("stream-K"); a token cut by a range boundary
//    is finished by the CTA holding its first tiles, which merges the other CTAs' partial
//    (o, max, sum) from the workspace in a fixed order (deterministic, no atomics on data).
//  * Warp roles: warp 0 producer (index read, -1 compaction, page translation, L2 prefetch of
//    index / block-table rows, Q loads by TMA), warp 1 MMA issuer, warps 2-3 idle (they only
//    follow the meta ring), warps 4-7 softmax + epilogue (one per TMEM sub-partition, 16 heads
//    each), warps 8-15 row loaders: cp.async 16-byte copies of bf16 rows into the
//    128-byte-swizzled K-major tile.
//  * Online softmax in the exp2 domain with a lazy rescale (O and the running sum are only
//    rescaled when the running max grows by more than 2^8).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>
#include <unordered_map>

#include "dsa_attn_common.h"
#include "dsa_host.h"
#include "dsa_ptx.cuh"

namespace dsa {

constexpr int kHeads = 64;

template <int KIND_, int D_NOPE_, int D_ROPE_, int DV_SPLIT_, int BN_, int KSTAGES_>
struct AttnCfg {
  static constexpr int KIND = KIND_;
  static constexpr int D_NOPE = D_NOPE_, D_ROPE = D_ROPE_, DK = D_NOPE + D_ROPE;
  static constexpr int DV_SPLIT = DV_SPLIT_;       // 256-wide output slices per token
  static constexpr int DVC = 256;                  // output columns per CTA pass
  static constexpr int BN = BN_;                   // gathered keys per tile (MMA N of S)
  static constexpr int KSTAGES = KSTAGES_;
  static constexpr int MSTAGES = DK > 256 ? 4 : 8;  // meta ring depth (smem-limited for 512+64)
  static constexpr int KCH = DK / 64;              // 128-byte chunks along d
  static constexpr int PCH = (BN + 63) / 64;       // 128-byte chunks of P along keys
  static constexpr int HALF = BN / 2;              // keys per softmax thread
  static_assert(KIND == DSA_CACHE_BF16, "the packed FP8 cache has its own kernels");
  static constexpr int NDEQ = 8;                   // loader warps (cp.async rows)
  static constexpr int WARPS = 8 + NDEQ;
  static constexpr int THREADS = 32 * WARPS;
  static constexpr int IDX_PER_LANE = (BN + 31) / 32;
  // shared memory carve-up (offsets from a 1024-aligned base)
  static constexpr int Q_BYTES = kHeads * DK * 2;
  static constexpr int KT_BYTES = BN * DK * 2;
  static constexpr int P_BYTES = PCH * kHeads * 128;
  static constexpr int Q_OFF = 0;
  static constexpr int KT_OFF = Q_OFF + Q_BYTES;
  static constexpr int P_OFF = KT_OFF + KSTAGES * KT_BYTES;
  static constexpr int META_BYTES = 32 + 4 * BN;
  static constexpr int META_OFF = P_OFF + P_BYTES;
  static constexpr int BAR_OFF = META_OFF + MSTAGES * META_BYTES;
  static constexpr int NBARS = 2 + 2 * KSTAGES + 2 * MSTAGES + 4 + 2;
  static constexpr int MISC_OFF = BAR_OFF + 8 * NBARS;
  static constexpr int SMEM_BYTES = MISC_OFF + 16 + 1024;  // + alignment slack
  // tensor memory columns
  static constexpr int S_COL = 0;
  static constexpr int O_COL = 2 * BN;
  static constexpr int TMEM_COLS = 512;
  static_assert(O_COL + DVC <= TMEM_COLS, "TMEM budget");
  static_assert(BN % 16 == 0 && HALF % 8 == 0 && BN <= 256, "tile shape");
  static_assert(KT_BYTES % 1024 == 0 && Q_BYTES % 1024 == 0, "alignment");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

// meta ring entry types
enum : int { kTile = 1, kSegEnd = 2, kDone = 3 };
// segment kinds
enum : int { kComplete = 0, kHead = 1, kPart = 2 };

struct MetaHdr {
  int type;
  int vtoken;     // virtual token = t * DV_SPLIT + dv slice
  int n_valid;    // kTile: valid rows in this tile
  int first;      // kTile: first non-empty tile of its segment
  int kind;       // kSegEnd: segment kind
  int had_tiles;  // kSegEnd: the segment had at least one non-empty tile
  int merge_last; // kSegEnd / kHead: last CTA holding a part of this token
  int pad;
};

struct AttnParams {
  const uint8_t* cache;
  int64_t num_slots;
  const int32_t* idx;
  int64_t idx_stride;
  int topk;
  const int32_t* bt;
  int64_t bt_stride;
  int page_size;
  int max_pages;
  const int32_t* req;
  float c_log2;  // sm_scale * log2(e)
  uint16_t* out;
  int64_t out_st, out_sh;
  float* lse;
  float* ws_o;    // [G][64][256] partial o (unnormalised, relative to its max)
  float* ws_ml;   // [G][2][64] partial max (log2 domain) and sum
  int* flags;     // [G][4] partial published (holds the call's epoch), one per softmax warp
  int epoch;      // this call's tag for the flags (never 0); stale flags from older calls differ
  int32_t* err;
  int64_t T;
  int NT;         // key tiles per token (over the index width)
  int64_t U;      // total units = T * DV_SPLIT * NT
  int G;          // CTAs
};

__device__ __forceinline__ void set_err(int32_t* err, int bits) {
  if (err) atomicOr(err, bits);
}

__device__ __forceinline__ int64_t unit_begin(int64_t b, int64_t U, int G) { return (b * U) / G; }

// ------------------------------------------------------------------------------ kernel --
template <class C>
__global__ void __launch_bounds__(C::THREADS, 1)
    dsa_attn_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ CUtensorMap tmap_q) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  const uint32_t bar0 = smem_u32(bars);
  // barrier addresses
  const uint32_t q_full = bar0, q_empty = bar0 + 8;
  auto k_full = [&](int s) { return bar0 + 16 + 8 * s; };
  auto k_empty = [&](int s) { return bar0 + 16 + 8 * (C::KSTAGES + s); };
  auto m_full = [&](int s) { return bar0 + 16 + 8 * (2 * C::KSTAGES + s); };
  auto m_empty = [&](int s) { return bar0 + 16 + 8 * (2 * C::KSTAGES + C::MSTAGES + s); };
  const uint32_t sx0 = bar0 + 16 + 8 * (2 * C::KSTAGES + 2 * C::MSTAGES);
  auto s_full = [&](int b) { return sx0 + 8 * b; };
  auto s_empty = [&](int b) { return sx0 + 16 + 8 * b; };
  const uint32_t p_full = sx0 + 32, pv_done = sx0 + 40;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::MISC_OFF + 4);

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int s = 0; s < C::KSTAGES; ++s) {
      mbar_init(k_full(s), 32 * C::NDEQ);  // one cp.async arrive per loader thread
      mbar_init(k_empty(s), 1);
    }
    for (int s = 0; s < C::MSTAGES; ++s) {
      mbar_init(m_full(s), 1);
      mbar_init(m_empty(s), 1 + 2 + 4 + C::NDEQ);  // MMA thread, warps 2-3, 4 softmax, loader warps
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(s_full(b), 1);
      mbar_init(s_empty(b), 4);
    }
    mbar_init(p_full, 4);
    mbar_init(pv_done, 1);
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
    if (mbar_wait(bar, par)) return true;
    fail(DSA_DEVERR_TIMEOUT);
    return false;
  };

  if (warp == 0) {
    // =========================================================== producer (one warp) ====
    // Walks this CTA's unit range segment by segment. Per key tile it reads the tile's index
    // window, masks entries < 0, translates logical positions through the block table, and
    // emits a meta entry with the compacted slot list. The index loads run two tiles ahead and
    // the block-table loads one tile ahead, so a tile (or a run of empty tiles) costs no
    // round trip of its own; both index rows and block-table rows are pulled into L2 at the
    // segment start.
    uint32_t mc = 0, qc = 0;
    const int64_t u0 = unit_begin(b, p.U, p.G), u1 = unit_begin(b + 1, p.U, p.G);
    auto emit_begin = [&](int& st) -> MetaHdr* {
      st = mc % C::MSTAGES;
      if (mc >= (uint32_t)C::MSTAGES) wait(m_empty(st), ((mc / C::MSTAGES) & 1) ^ 1);
      return reinterpret_cast<MetaHdr*>(smem + C::META_OFF + st * C::META_BYTES);
    };
    auto emit_end = [&](int st) {
      __syncwarp();
      if (lane == 0) mbar_arrive(m_full(st));
      ++mc;
    };
    const int64_t pos_limit = p.bt ? (int64_t)p.max_pages * p.page_size : p.num_slots;
    int64_t u = u0;
    while (u < u1 && !*abort_flag) {
      const int64_t vt = u / p.NT;
      const int j0 = (int)(u - vt * p.NT);
      const int64_t uend = (vt + 1) * p.NT < u1 ? (vt + 1) * p.NT : u1;
      const int j1 = (int)(uend - vt * p.NT);
      const int64_t t = vt / C::DV_SPLIT;
      const int kind = j0 > 0 ? kPart : (j1 < p.NT ? kHead : kComplete);
      const int64_t req = p.req ? p.req[t] : 0;
      const int32_t* irow = p.idx + t * p.idx_stride;
      const int32_t* btrow = p.bt ? p.bt + req * p.bt_stride : nullptr;
      {  // pull this segment's index window and the request's block-table row into L2
        const int e0 = j0 * C::BN, e1 = min(j1 * C::BN, p.topk);
        const uintptr_t a0 = reinterpret_cast<uintptr_t>(irow + e0) & ~uintptr_t(127);
        const uintptr_t a1 = reinterpret_cast<uintptr_t>(irow + e1);
        for (uintptr_t a = a0 + 128 * lane; a < a1; a += 32 * 128)
          asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
        if (btrow) {
          const uintptr_t c0 = reinterpret_cast<uintptr_t>(btrow) & ~uintptr_t(127);
          const uintptr_t c1 = reinterpret_cast<uintptr_t>(btrow + p.max_pages);
          for (uintptr_t a = c0 + 128 * lane; a < c1; a += 32 * 128)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
        }
      }
      // The segment's index window [e0, e1) is read 256 entries per step (entry pos + 32k + lane
      // in lane `lane`, slot k). Index loads run two steps ahead and block-table loads one step
      // ahead. Valid entries are packed, in index order, into dense tiles of BN rows, so runs of
      // -1 padding cost only their index reads and every emitted tile but the segment's last
      // is full.
      constexpr int V = 8;
      const int e0 = j0 * C::BN, e1 = min(j1 * C::BN, p.topk);
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
          else pg[k] = btrow ? __ldg(btrow + x[k] / p.page_size) : x[k];
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
          if (lane < C::KCH)
            tma_load_3d(sbase + C::Q_OFF + lane * (kHeads * 128), &tmap_q, 64 * lane, 0, (int)t, q_full);
          ++qc;
        }
        mh = emit_begin(st);
        slots = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(mh) + 32);
        if (lane == 0) {
          mh->type = kTile;
          mh->vtoken = (int)vt;
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
      for (int pos = e0; pos < e1 && !*abort_flag; pos += 32 * V) {
        int ic[V], pb[V];
        load_step(pos + 64 * V, ic);
        page_of(ib, pb);
        int bad = 0;
#pragma unroll
        for (int k = 0; k < V; ++k) {
          int64_t slot = -1;
          if (pa[k] >= 0) {
            if (btrow) {
              slot = (int64_t)pa[k] * p.page_size + ia[k] % p.page_size;
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
          if (bal == 0u) continue;
          if (!open) open_tile();
          const int n = __popc(bal);
          const int my = cnt + __popc(bal & ((1u << lane) - 1u));
          if (ok && my < C::BN) slots[my] = (int)slot;
          if (cnt + n >= C::BN) {  // this group fills the tile (and may spill into the next one)
            close_tile(C::BN);
            const int rest = cnt + n - C::BN;
            if (rest > 0) {
              open_tile();
              if (ok && my >= C::BN) slots[my - C::BN] = (int)slot;
              cnt = rest;
            }
          } else {
            cnt += n;
          }
        }
        if (bad) set_err(p.err, DSA_DEVERR_INDEX_OUT_OF_RANGE);
#pragma unroll
        for (int k = 0; k < V; ++k) {
          ia[k] = ib[k];
          ib[k] = ic[k];
          pa[k] = pb[k];
        }
      }
      if (open) close_tile(cnt);
      {
        int st;
        MetaHdr* mh = emit_begin(st);
        if (lane == 0) {
          mh->type = kSegEnd;
          mh->vtoken = (int)vt;
          mh->kind = kind;
          mh->had_tiles = had ? 1 : 0;
          int last = b;
          if (kind == kHead) {
            const int64_t last_unit = (vt + 1) * p.NT - 1;
            while (last + 1 < p.G && unit_begin(last + 1, p.U, p.G) <= last_unit) ++last;
          }
          mh->merge_last = last;
        }
        emit_end(st);
      }
      u = uend;
    }
    {
      int st;
      MetaHdr* mh = emit_begin(st);
      if (lane == 0) mh->type = kDone;
      emit_end(st);
    }
  } else if (warp == 1) {
    // ============================================================== MMA issuer ====
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16(64, C::BN, 0, 0);
      constexpr uint32_t idPV = idesc_bf16(64, C::DVC, 0, 1);
      uint32_t mc = 0, g = 0, qc = 0;
      // Descriptors are built once; the k-step offsets are compile-time adds on the 16-byte
      // address field (every operand stays below 256 KB of shared memory).
      const uint64_t dQ = sw128_desc(sbase + C::Q_OFF, 16, 1024);
      const uint64_t dP = sw128_desc(sbase + C::P_OFF, 16, 1024);
      auto issue_pv = [&](uint32_t gg, int first, int dvh) {
        if (!wait(p_full, gg & 1)) return;
        tc_fence_after();
        const int ks = gg % C::KSTAGES;
        const uint64_t dV = sw128_desc(sbase + C::KT_OFF + ks * C::KT_BYTES + dvh * (C::DVC / 64) * (C::BN * 128),
                                       C::BN * 128, 1024);
#pragma unroll
        for (int kk = 0; kk < C::BN / 16; ++kk) {
          const uint64_t pa = (uint64_t)(((kk >> 2) * (kHeads * 128) + (kk & 3) * 32) >> 4);
          const uint64_t vb = (uint64_t)((kk * 16 * 128) >> 4);
          mma_bf16(tmem + C::O_COL, dP + pa, dV + vb, idPV, (first && kk == 0) ? 0u : 1u);
        }
        mma_commit(k_empty(ks));
        mma_commit(pv_done);
      };
      // Event-driven issue: poll (without blocking) for the oldest tile whose P is ready and for
      // the next tile whose K stage, S buffer (and Q) are ready; issue whichever is ready,
      // PV first since it frees a K stage. Meta entries are consumed as S advances (segment
      // ends release the Q buffer once the segment's S products are issued).
      uint32_t gP = 0;             // PV products issued (gP <= g, the S products issued)
      int t_first[4] = {0, 0, 0, 0}, t_dvh[4] = {0, 0, 0, 0};
      bool done = false, have = false, q_ok = false;
      int cur_first = 0, cur_dvh = 0;
      uint64_t last_progress = globaltimer_ns();
      auto try_pv = [&](uint32_t limit) -> bool {  // issue PV(gP) if its P is ready
        if (gP < limit && mbar_test(p_full, gP & 1)) {
          issue_pv(gP, t_first[gP & 3], t_dvh[gP & 3]);
          ++gP;
          return true;
        }
        return false;
      };
      auto issue_s = [&](uint32_t gg) {
        const int ks = gg % C::KSTAGES;
        // bf16 rows arrive by cp.async, i.e. through the generic proxy: order them before the
        // tensor core reads
        fence_proxy_async_smem();
        tc_fence_after();
        const uint64_t dK = sw128_desc(sbase + C::KT_OFF + ks * C::KT_BYTES, 16, 1024);
        // four k-steps at a time, so that a PV whose P became ready is not queued behind the
        // whole S product
#pragma unroll
        for (int kk = 0; kk < C::DK / 16; ++kk) {
          const uint64_t qa = (uint64_t)(((kk >> 2) * (kHeads * 128) + (kk & 3) * 32) >> 4);
          const uint64_t ka = (uint64_t)(((kk >> 2) * (C::BN * 128) + (kk & 3) * 32) >> 4);
          mma_bf16(tmem + C::S_COL + (gg & 1) * C::BN, dQ + qa, dK + ka, idS, kk > 0 ? 1u : 0u);
          if ((kk & 3) == 3 && kk + 1 < C::DK / 16) try_pv(gg);
        }
        mma_commit(s_full(gg & 1));
      };
      while (!*abort_flag && (!done || gP < g)) {
        bool progress = false;
        if (try_pv(g)) {
          progress = true;
        } else if (!done) {
          if (!have) {
            const int st = mc % C::MSTAGES;
            if (mbar_test(m_full(st), (mc / C::MSTAGES) & 1)) {
              const MetaHdr* mh = reinterpret_cast<const MetaHdr*>(smem + C::META_OFF + st * C::META_BYTES);
              const int type = mh->type;
              if (type == kTile) {
                cur_first = mh->first;
                cur_dvh = mh->vtoken % C::DV_SPLIT;
                have = true;
              } else if (type == kSegEnd) {
                if (mh->had_tiles) mma_commit(q_empty);
              } else {
                done = true;
              }
              mbar_arrive(m_empty(st));
              ++mc;
              progress = true;
            }
          }
          if (have) {
            if (cur_first && !q_ok && mbar_test(q_full, qc & 1)) {
              q_ok = true;
              ++qc;
            }
            if ((!cur_first || q_ok) && mbar_test(k_full(g % C::KSTAGES), (g / C::KSTAGES) & 1) &&
                (g < 2 || mbar_test(s_empty(g & 1), ((g >> 1) & 1) ^ 1))) {
              issue_s(g);
              t_first[g & 3] = cur_first;
              t_dvh[g & 3] = cur_dvh;
              ++g;
              have = false;
              q_ok = false;
              progress = true;
            }
          }
        }
        if (progress) {
          last_progress = globaltimer_ns();
        } else if (globaltimer_ns() - last_progress > 2000000000ull) {
          fail(DSA_DEVERR_TIMEOUT);
          break;
        }
      }
      // drain: wait for every MMA this thread issued before TMEM can be released
      if (g > 0) mbar_wait(pv_done, (g - 1) & 1);
    }
    __syncwarp();
  } else if (warp == 2 || warp == 3) {
    // ========================================================= idle (2 warps) ====
    // These warps only follow the meta ring (its release counts them), so that they leave the
    // loop with the others.
    uint32_t mc = 0;
    while (!*abort_flag) {
      const int st = mc % C::MSTAGES;
      if (!wait(m_full(st), (mc / C::MSTAGES) & 1)) break;
      const MetaHdr* mh = reinterpret_cast<const MetaHdr*>(smem + C::META_OFF + st * C::META_BYTES);
      const int type = mh->type;
      __syncwarp();
      if (lane == 0) mbar_arrive(m_empty(st));
      ++mc;
      if (type == kDone) break;
    }
  } else if (warp >= 4 && warp < 8) {
    // =============================================== softmax + epilogue (4 warps) ====
    const int sp = warp & 3;                 // TMEM sub-partition
    const int h = 16 * sp + (lane & 15);     // head of this thread
    const int hf = lane >> 4;                // key half (S) / column half (O)
    const uint32_t trow = tmem + ((uint32_t)(32 * sp) << 16);
    const float c = p.c_log2;
    uint32_t mc = 0, g = 0;
    float m_run = -INFINITY, l_part = 0.0f;
    while (!*abort_flag) {
      const int st = mc % C::MSTAGES;
      if (!wait(m_full(st), (mc / C::MSTAGES) & 1)) break;
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
        if (first) {
          m_run = -INFINITY;
          l_part = 0.0f;
        }
        if (!wait(s_full(g & 1), (g >> 1) & 1)) break;
        tc_fence_after();
        float s[C::HALF];
        {
          const uint32_t ta = trow + C::S_COL + (g & 1) * C::BN;
          uint32_t r[C::HALF];
          // all column chunks of this thread's key half, then a single wait
#pragma unroll
          for (int c0 = 0; c0 + 32 <= C::HALF; c0 += 32)
            tmem_ld16x2_x32<C::HALF>(ta + c0, *reinterpret_cast<uint32_t(*)[32]>(r + c0));
          constexpr int TAIL = C::HALF % 32, T0 = C::HALF - TAIL;
          if constexpr (TAIL >= 16) tmem_ld16x2_x16<C::HALF>(ta + T0, r + T0);
          if constexpr (TAIL % 16 == 8) tmem_ld16x2_x8<C::HALF>(ta + T0 + (TAIL & 16), r + T0 + (TAIL & 16));
          tc_wait_ld();
#pragma unroll
          for (int i = 0; i < C::HALF; ++i) s[i] = __uint_as_float(r[i]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(s_empty(g & 1));
        // mask keys past n_valid (only a partially filled tile has any), then the row max with
        // four independent chains; the two threads of a head hold its two key halves
        const int kbase = hf * C::HALF;
        if (n_valid < C::BN) {
#pragma unroll
          for (int i = 0; i < C::HALF; ++i)
            if (kbase + i >= n_valid) s[i] = -INFINITY;
        }
        float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int i = 0; i < C::HALF; ++i) mx4[i & 3] = fmaxf(mx4[i & 3], s[i]);
        float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        const float m_tile = mx * c;  // finite: every tile has at least one valid key
        const bool grow = m_tile > m_run + 8.0f;
        const float m_new = grow ? m_tile : m_run;
        const float alpha = grow ? ex2_approx(m_run - m_new) : 1.0f;  // exp2(-inf) = 0 on the first tile
        // p = 2^(s*c - m): one FFMA and one MUFU ex2 per score; masked keys of a partially filled
        // tile get p = 0 explicitly (a zero scale would turn -inf * 0 into NaN)
        float rs4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        uint32_t pk[C::HALF / 2];
        if (n_valid < C::BN) {
#pragma unroll
          for (int i = 0; i < C::HALF; i += 2) {
            const float p0 = kbase + i < n_valid ? ex2_approx(fmaf(s[i], c, -m_new)) : 0.0f;
            const float p1 = kbase + i + 1 < n_valid ? ex2_approx(fmaf(s[i + 1], c, -m_new)) : 0.0f;
            rs4[(i >> 1) & 3] += p0 + p1;
            pk[i / 2] = f32x2_to_bf16x2(p0, p1);
          }
        } else {
#pragma unroll
          for (int i = 0; i < C::HALF; i += 2) {
            const float p0 = ex2_approx(fmaf(s[i], c, -m_new));
            const float p1 = ex2_approx(fmaf(s[i + 1], c, -m_new));
            rs4[(i >> 1) & 3] += p0 + p1;
            pk[i / 2] = f32x2_to_bf16x2(p0, p1);
          }
        }
        const float rs = (rs4[0] + rs4[1]) + (rs4[2] + rs4[3]);
        l_part = l_part * alpha + rs;
        // P buffer reuse and O rescale need the previous PV to be complete
        if (g > 0 && !wait(pv_done, (g - 1) & 1)) break;
        tc_fence_after();
        // tcgen05.ld/st are warp-collective: the warp rescales if any of its heads grew, each
        // thread with its own factor (1 for heads that did not grow)
        if (__any_sync(0xffffffffu, grow && !first)) {
          const uint32_t oa = trow + C::O_COL;
          uint32_t r[32];
#pragma unroll 1
          for (int c0 = 0; c0 < C::DVC / 2; c0 += 32) {
            tmem_ld16x2_x32<128>(oa + c0, r);
            tc_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
            tmem_st16x2_x32<128>(oa + c0, r);
          }
          tc_wait_st();
        }
        m_run = m_new;
        // write P (bf16, K-major, 128-byte swizzle): row h, keys [kbase, kbase + HALF)
#pragma unroll
        for (int gq = 0; gq < C::HALF / 8; ++gq) {
          const int key0 = kbase + 8 * gq;
          const int ch = key0 >> 6, gr = (key0 & 63) >> 3;
          uint8_t* dst = smem + C::P_OFF + ch * (kHeads * 128) + h * 128 + ((gr ^ (h & 7)) << 4);
          *reinterpret_cast<uint4*>(dst) = make_uint4(pk[4 * gq], pk[4 * gq + 1], pk[4 * gq + 2], pk[4 * gq + 3]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full);
        ++g;
      } else {  // kSegEnd: epilogue for this (virtual) token
        const int vt = mh->vtoken, kind = mh->kind, had = mh->had_tiles, last = mh->merge_last;
        __syncwarp();
        if (lane == 0) mbar_arrive(m_empty(st));
        if (had) {
          if (!wait(pv_done, (g - 1) & 1)) break;
          tc_fence_after();
        }
        const float l_row = l_part + __shfl_xor_sync(0xffffffffu, l_part, 16);
        const float m_row = had ? m_run : -INFINITY;
        const float l_own = had ? l_row : 0.0f;
        const int64_t t = vt / C::DV_SPLIT;
        const int dvh = vt % C::DV_SPLIT;
        const uint32_t oa = trow + C::O_COL;
        if (kind == kPart) {
          // publish (o, m, l) of this part in workspace slot b
          float* wo = p.ws_o + ((int64_t)b * kHeads + h) * C::DVC + hf * (C::DVC / 2);
          if (had) {
            uint32_t r[32];
#pragma unroll 1
            for (int c0 = 0; c0 < C::DVC / 2; c0 += 32) {
              tmem_ld16x2_x32<128>(oa + c0, r);
              tc_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; i += 4)
                *reinterpret_cast<float4*>(wo + c0 + i) = make_float4(
                    __uint_as_float(r[i]), __uint_as_float(r[i + 1]), __uint_as_float(r[i + 2]), __uint_as_float(r[i + 3]));
            }
          }
          if (hf == 0) {
            p.ws_ml[((int64_t)b * 2 + 0) * kHeads + h] = m_row;
            p.ws_ml[((int64_t)b * 2 + 1) * kHeads + h] = l_own;
          }
          __threadfence();
          __syncwarp();
          if (lane == 0)
            asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p.flags + 4 * b + sp), "r"(p.epoch) : "memory");
        } else {
          // complete token, or the head of a split token: merge parts b+1..last in order
          const int nparts = kind == kHead ? last - b : 0;
          bool ok = true;
          for (int k = 1; k <= nparts && ok; ++k) {
            int v = 0;
            const uint64_t t0 = globaltimer_ns();
            for (;;) {
              asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p.flags + 4 * (b + k) + sp) : "memory");
              if (v == p.epoch || globaltimer_ns() - t0 > 2000000000ull) break;
              __nanosleep(64);
            }
            if (v != p.epoch) ok = false;
          }
          if (!ok) fail(DSA_DEVERR_TIMEOUT);
          float M = m_row;
          for (int k = 1; k <= nparts && ok; ++k) M = fmaxf(M, p.ws_ml[((int64_t)(b + k) * 2 + 0) * kHeads + h]);
          const float w_own = (l_own > 0.0f) ? exp2f(m_row - M) : 0.0f;
          float L = w_own * l_own;
          float wk[8];
          int nk = 0;
          for (int k = 1; k <= nparts && ok; ++k) {
            const float mk = p.ws_ml[((int64_t)(b + k) * 2 + 0) * kHeads + h];
            const float lk = p.ws_ml[((int64_t)(b + k) * 2 + 1) * kHeads + h];
            const float w = lk > 0.0f ? exp2f(mk - M) : 0.0f;
            if (nk < 8) wk[nk] = w;
            ++nk;
            L += w * lk;
          }
          const float inv = L > 0.0f ? 1.0f / L : 0.0f;
          uint16_t* orow = p.out + t * p.out_st + (int64_t)h * p.out_sh + dvh * C::DVC + hf * (C::DVC / 2);
          uint32_t r[32];
#pragma unroll 1
          for (int c0 = 0; c0 < C::DVC / 2; c0 += 32) {
            float acc[32];
            if (had) {  // warp-uniform: every thread of the warp saw the same meta entry
              tmem_ld16x2_x32<128>(oa + c0, r);
              tc_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i) acc[i] = w_own * __uint_as_float(r[i]);
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i) acc[i] = 0.0f;
            }
            for (int k = 1; k <= nparts && ok; ++k) {
              const float w = (k - 1 < 8) ? wk[k - 1]
                                          : (p.ws_ml[((int64_t)(b + k) * 2 + 1) * kHeads + h] > 0.0f
                                                 ? exp2f(p.ws_ml[((int64_t)(b + k) * 2 + 0) * kHeads + h] - M)
                                                 : 0.0f);
              if (w == 0.0f) continue;
              const float* src = p.ws_o + ((int64_t)(b + k) * kHeads + h) * C::DVC + hf * (C::DVC / 2) + c0;
#pragma unroll
              for (int i = 0; i < 32; i += 4) {
                const float4 v = *reinterpret_cast<const float4*>(src + i);
                acc[i] += w * v.x;
                acc[i + 1] += w * v.y;
                acc[i + 2] += w * v.z;
                acc[i + 3] += w * v.w;
              }
            }
            uint32_t pkd[16];
#pragma unroll
            for (int i = 0; i < 32; i += 2) pkd[i / 2] = f32x2_to_bf16x2(acc[i] * inv, acc[i + 1] * inv);
#pragma unroll
            for (int i = 0; i < 16; i += 4)
              *reinterpret_cast<uint4*>(orow + c0 + 2 * i) = make_uint4(pkd[i], pkd[i + 1], pkd[i + 2], pkd[i + 3]);
          }
          if (p.lse && dvh == 0 && hf == 0)
            p.lse[t * kHeads + h] = L > 0.0f ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
          // every lane of this warp has read the parts: clear their publish flags, so that the
          // workspace holds no set flag after the call (a later call that carries the same tag,
          // such as a replay of a recorded launch, then never mistakes them for its own)
          __syncwarp();
          if (ok && lane == 0)
            for (int k = 1; k <= nparts; ++k) p.flags[4 * (b + k) + sp] = 0;

        }
        tc_fence_before();
      }
      ++mc;
    }
  } else if (warp >= 8) {
    // ====================================================== row loaders (8 warps) ====
    // Warp dw fills rows dw, dw + 8, ... of each K tile in the 128-byte-swizzled K-major layout
    // (row r, 16-byte granule g of 64-element chunk c at c*BN*128 + r*128 + ((g ^ (r&7)) << 4)).
    // cp.async 16-byte copies (rows past n_valid zero-filled), completion counted on the stage
    // barrier per thread.
    const int dw = warp - 8;
    constexpr int RPW = C::BN / C::NDEQ;  // rows per warp per tile
    uint32_t mc = 0, g = 0;
    while (!*abort_flag) {
      const int st = mc % C::MSTAGES;
      if (!wait(m_full(st), (mc / C::MSTAGES) & 1)) break;
      const MetaHdr* mh = reinterpret_cast<const MetaHdr*>(smem + C::META_OFF + st * C::META_BYTES);
      const int type = mh->type;
      if (type != kTile) {
        __syncwarp();
        if (lane == 0) mbar_arrive(m_empty(st));
        ++mc;
        if (type == kDone) break;
        continue;
      }
      const int n_valid = mh->n_valid;
      const int* slots = reinterpret_cast<const int*>(reinterpret_cast<const uint8_t*>(mh) + 32);
      const int ks = g % C::KSTAGES;
      uint8_t* kt = smem + C::KT_OFF + ks * C::KT_BYTES;
      if (g >= (uint32_t)C::KSTAGES && !wait(k_empty(ks), ((g / C::KSTAGES) & 1) ^ 1)) break;
      constexpr int GR = C::DK / 8;  // 16-byte granules per row
#pragma unroll 2
      for (int k = 0; k < RPW; ++k) {
        const int r = dw + C::NDEQ * k;
        const bool v = r < n_valid;
        const uint8_t* row = p.cache + (v ? (int64_t)slots[r] : 0) * (2 * C::DK);
#pragma unroll
        for (int q0 = 0; q0 < GR; q0 += 32) {
          const int q = q0 + lane;
          if (q < GR) {
            const int ch = q >> 3, gr = q & 7;
            const uint32_t dst = smem_u32(kt + ch * (C::BN * 128) + r * 128 + ((gr ^ (r & 7)) << 4));
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(row + 16 * q),
                         "r"(v ? 16 : 0)
                         : "memory");
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(m_empty(st));
      ++mc;
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
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ------------------------------------------------------------------------------- host --
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static dsa_status_t get_encode_fn(EncodeTiledFn* fn) {
  static std::once_flag once;
  static EncodeTiledFn f = nullptr;
  static cudaError_t err = cudaSuccess;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q);
    if (err == cudaSuccess && q == cudaDriverEntryPointSuccess) f = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  if (!f) return cuda_fail(err != cudaSuccess ? err : cudaErrorNotSupported);
  *fn = f;
  return DSA_OK;
}

dsa_status_t encode_q_tensor_map(const dsa_attn_args_t* a, int dk, CUtensorMap* out) {
  EncodeTiledFn encode = nullptr;
  dsa_status_t st = get_encode_fn(&encode);
  if (st != DSA_OK) return st;
  const cuuint64_t dims[3] = {(cuuint64_t)dk, (cuuint64_t)kHeads, (cuuint64_t)a->T};
  const cuuint64_t strides[2] = {(cuuint64_t)a->q_stride_h * 2, (cuuint64_t)a->q_stride_t * 2};
  const cuuint32_t box[3] = {64, (cuuint32_t)kHeads, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  CUresult r = encode(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a->q), dims, strides, box, es,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DSA_OK : cuda_fail(cudaErrorInvalidValue);
}

static size_t attn_ws_split_bytes(int sm_count) { return ((size_t)(33 * sm_count + 1) * 8 + 255) & ~size_t(255); }

size_t attn_ws_bytes(int sm_count) {
  // partial o [G][64][256] fp32 + up to four running values per head [G][4][64] fp32 (max and
  // sum; the 8-bit-operand kernel adds one reference max per output half) + flags [G][8] int32
  // + the work-balanced split: entry counts of 32 unit slices per CTA and the G + 1 range
  // bounds (int64)
  const size_t o = (size_t)sm_count * kHeads * 256 * 4;
  const size_t ml = (size_t)sm_count * 4 * kHeads * 4;
  const size_t fl = ((size_t)sm_count * 32 + 255) & ~size_t(255);
  return o + ml + fl + attn_ws_split_bytes(sm_count);
}

AttnWorkspace attn_ws_layout(void* workspace, int sm_count) {
  uint8_t* w = static_cast<uint8_t*>(workspace);
  const size_t o_bytes = (size_t)sm_count * kHeads * 256 * 4;
  AttnWorkspace r;
  r.o = reinterpret_cast<float*>(w);
  r.ml = reinterpret_cast<float*>(w + o_bytes);
  r.flags = reinterpret_cast<int*>(w + o_bytes + (size_t)sm_count * 4 * kHeads * 4);
  r.split = reinterpret_cast<int64_t*>(w + o_bytes + (size_t)sm_count * 4 * kHeads * 4 +
                                       (((size_t)sm_count * 32 + 255) & ~size_t(255)));
  return r;
}

int next_attn_epoch(const void* workspace) {
  static std::mutex mu;
  static std::unordered_map<const void*, int> epochs;
  std::lock_guard<std::mutex> lock(mu);
  int& e = epochs[workspace];
  e = (e == 0x7FFFFFFF) ? 1 : e + 1;
  return e;
}

template <class C>
static dsa_status_t launch(const dsa_attn_args_t* a, const DeviceInfo& dev, cudaStream_t stream) {
  CUtensorMap tq;
  dsa_status_t st = encode_q_tensor_map(a, C::DK, &tq);
  if (st != DSA_OK) return st;

  AttnParams p{};
  p.cache = static_cast<const uint8_t*>(a->cache);
  p.num_slots = a->num_slots;
  p.idx = a->indices;
  p.idx_stride = a->idx_stride_t;
  p.topk = a->topk;
  p.bt = a->block_table;
  p.bt_stride = a->bt_stride;
  p.page_size = a->block_table ? a->page_size : 1;
  p.max_pages = a->block_table ? a->max_pages : 0;
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
  p.NT = (a->topk + C::BN - 1) / C::BN;
  p.U = a->T * C::DV_SPLIT * (int64_t)p.NT;
  // one persistent CTA per SM, but at least 4 units per CTA so that small batches split each
  // token into few parts (fewer partials to merge)
  const int64_t g_cap = (p.U + 3) / 4;
  p.G = (int)(g_cap < dev.sm_count ? g_cap : dev.sm_count);

  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)p.G);
  cfg.blockDim = dim3(C::THREADS);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, dsa_attn_kernel<C>, p, tq);
  return e == cudaSuccess ? DSA_OK : cuda_fail(e);
}

using CfgBf16_576 = AttnCfg<DSA_CACHE_BF16, 512, 64, 2, 64, 2>;

dsa_status_t prepare_attn_kernels(int device) {
  static std::mutex mu;
  static bool done[64] = {};
  if (device < 0 || device >= 64) return DSA_ERR_NO_DEVICE;
  std::lock_guard<std::mutex> lock(mu);
  if (done[device]) return DSA_OK;
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(dsa_attn_kernel<CfgBf16_576>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                CfgBf16_576::SMEM_BYTES)) != cudaSuccess ||

      (e = k128_set_attributes()) != cudaSuccess || (e = f8_set_attributes()) != cudaSuccess ||
      (e = ctl_set_attributes()) != cudaSuccess)
    return cuda_fail(e);
  done[device] = true;
  return DSA_OK;
}

static dsa_status_t validate(const dsa_attn_args_t* a) {
  if (!a) return DSA_ERR_INVALID_ARGUMENT;
  if (a->T < 0 || a->num_slots < 0) return DSA_ERR_INVALID_ARGUMENT;
  if (a->kind != DSA_CACHE_BF16 && a->kind != DSA_CACHE_FP8_SCALED) return DSA_ERR_INVALID_ARGUMENT;
  if (a->H != kHeads) return DSA_ERR_UNSUPPORTED;
  if (!((a->d_nope == 256 && a->d_rope == 0 && a->d_v == 256) || (a->d_nope == 512 && a->d_rope == 64 && a->d_v == 512)))
    return DSA_ERR_UNSUPPORTED;
  if (a->topk < 1 || a->topk > 16384) return DSA_ERR_INVALID_ARGUMENT;
  // any finite scale (a negative one reverses the ranking of the keys; the pages set no limit)
  if (!(a->sm_scale > -3.0e38f && a->sm_scale < 3.0e38f)) return DSA_ERR_INVALID_ARGUMENT;
  if (a->num_slots > 0x7FFFFFFELL) return DSA_ERR_UNSUPPORTED;
  if (a->T == 0) return DSA_OK;
  const int D = a->d_nope + a->d_rope;
  if (!a->q || !a->cache || !a->indices || !a->out || !a->workspace) return DSA_ERR_INVALID_ARGUMENT;
  if (a->num_slots < 1) return DSA_ERR_INVALID_ARGUMENT;
  if (!aligned(a->q, 16) || a->q_stride_h % 8 || a->q_stride_t % 8 || a->q_stride_h < D ||
      a->q_stride_t < (int64_t)kHeads * a->q_stride_h)
    return DSA_ERR_INVALID_ARGUMENT;
  if (a->idx_stride_t < a->topk) return DSA_ERR_INVALID_ARGUMENT;
  if (!aligned(a->out, 16) || a->out_stride_h % 8 || a->out_stride_t % 8 || a->out_stride_h < a->d_v ||
      a->out_stride_t < (int64_t)kHeads * a->out_stride_h)
    return DSA_ERR_INVALID_ARGUMENT;
  if (!aligned(a->cache, 16) || !aligned(a->workspace, 256)) return DSA_ERR_INVALID_ARGUMENT;
  if (a->block_table) {
    if (a->page_size <= 0 || a->max_pages <= 0 || a->bt_stride < a->max_pages) return DSA_ERR_INVALID_ARGUMENT;
  }
  if (a->lse && !aligned(a->lse, 4)) return DSA_ERR_INVALID_ARGUMENT;
  return DSA_OK;
}

}  // namespace dsa

using namespace dsa;

extern "C" {

dsa_status_t dsa_sparse_attn_workspace_size(const dsa_attn_args_t* a, size_t* bytes) {
  if (!a || !bytes) return DSA_ERR_INVALID_ARGUMENT;
  DeviceInfo dev;
  dsa_status_t st = current_device(&dev);
  if (st != DSA_OK) return st;
  *bytes = attn_ws_bytes(dev.sm_count);
  return DSA_OK;
}

dsa_status_t dsa_sparse_attn(const dsa_attn_args_t* a, void* stream) {
  dsa_status_t st = validate(a);
  if (st != DSA_OK || a->T == 0) return st;
  DeviceInfo dev;
  st = current_device(&dev);
  if (st != DSA_OK) return st;
  if (a->workspace_bytes < attn_ws_bytes(dev.sm_count)) return DSA_ERR_WORKSPACE_TOO_SMALL;
  st = prepare_attn_kernels(dev.device);
  if (st != DSA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (a->d_nope == 256) return launch_attn_k128(a, dev, s);
  if (a->kind == DSA_CACHE_FP8_SCALED) return launch_attn_ctl(a, dev, s);
  return launch<CfgBf16_576>(a, dev, s);
}

}  // extern "C"

// ------------------------------------------------------------- fixed-scratch entry point --
// Some callers cannot allocate device memory when they call the library: serving engines that
// reserve all device memory up front for their KV page pool, runtimes that work from a fixed
// memory plan, and latency-critical paths where an allocation could stall or synchronise the
// device. For them, dsa_sparse_attn_static_ws takes its scratch (split-token partials, their
// flags and the split bounds) from this file-scope device array instead of a caller-supplied
// workspace. It holds the partials of at most kStaticWsCtas CTAs (about 10.6 MB); every GPU that
// loads the library keeps it until the process exits.
namespace dsa {
constexpr int kStaticWsCtas = 160;
constexpr size_t kStaticWsBytes = (size_t)kStaticWsCtas * kHeads * 256 * 4 + (size_t)kStaticWsCtas * 4 * kHeads * 4 +
                                  (((size_t)kStaticWsCtas * 32 + 255) & ~size_t(255)) +
                                  (((size_t)(33 * kStaticWsCtas + 1) * 8 + 255) & ~size_t(255));
static __device__ __align__(256) uint8_t g_static_ws[kStaticWsBytes];

// Device address of g_static_ws for the current device, looked up once per device (the host
// name of the array is only a stand-in and must never be passed to a kernel).
static dsa_status_t static_ws_ptr(int device, void** out) {
  static std::mutex mu;
  static void* ptrs[64] = {};
  if (device < 0 || device >= 64) return DSA_ERR_NO_DEVICE;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[device]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_static_ws);
    if (e != cudaSuccess) return cuda_fail(e);
    ptrs[device] = p;
  }
  *out = ptrs[device];
  return DSA_OK;
}
}  // namespace dsa

extern "C" dsa_status_t dsa_sparse_attn_static_ws(const dsa_attn_args_t* a, void* stream) {
  if (!a) return DSA_ERR_INVALID_ARGUMENT;
  // the caller's workspace fields are ignored; the other arguments follow dsa_sparse_attn's
  // rules (the placeholder only satisfies the workspace check and is never dereferenced)
  dsa_attn_args_t b = *a;
  b.workspace = reinterpret_cast<void*>(uintptr_t(256));
  b.workspace_bytes = 0;
  dsa_status_t st = validate(&b);
  if (st != DSA_OK || b.T == 0) return st;
  DeviceInfo dev;
  st = current_device(&dev);
  if (st != DSA_OK) return st;
  // at most kStaticWsCtas persistent CTAs: their partials must fit in the fixed array
  DeviceInfo capped = dev;
  if (capped.sm_count > kStaticWsCtas) capped.sm_count = kStaticWsCtas;
  if (attn_ws_bytes(capped.sm_count) > kStaticWsBytes) return DSA_ERR_WORKSPACE_TOO_SMALL;
  void* ws = nullptr;
  st = static_ws_ptr(dev.device, &ws);
  if (st != DSA_OK) return st;
  st = prepare_attn_kernels(dev.device);
  if (st != DSA_OK) return st;
  b.workspace = ws;
  b.workspace_bytes = kStaticWsBytes;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // nothing needs clearing: the array starts zero-filled and each call tags its merge flags
  // with a fresh per-array epoch, so values left by an earlier call never match
  if (b.d_nope == 256) return launch_attn_k128(&b, capped, s);
  if (b.kind == DSA_CACHE_FP8_SCALED) return launch_attn_ctl(&b, capped, s);
  return launch<CfgBf16_576>(&b, capped, s);
}
