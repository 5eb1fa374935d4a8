// dsa_attn.cu - DSA sparse MLA attention forward for sm_103a (tcgen05 + TMEM + TMA).
//
// What is computed (sglang PR #38547 "Enable zero-RoPE TileLang DSA on gfx950", Summary and
// Direct GLM geometry coverage list): for every query token t and head h, gather the latent
// rows named by t's top-k index list (entries < 0 masked), score s_j = sm_scale * q[t,h].k_j,
// softmax over j and return sum_j p_j * k_j[0:d_v] in bf16. The cache holds bf16 rows or the
// packed scaled-FP8 rows of the Contract table (codes * per-128-tile fp32 scale).
//
// Kernel design (GB300-first, not the pages' TileLang/HIP kernels):
//  * Heads are the MMA M dimension (M = 64), gathered keys are N: S = Q K^T (K-dim = d) and
//    O += P V (K-dim = keys, V = the first d_v columns of the same gathered rows) are dense
//    tcgen05 kind::f16 contractions with fp32 accumulators in tensor memory. The M = 64
//    accumulator occupies TMEM lanes 32*w + [0,16) of each sub-partition w.
//  * One persistent CTA per SM, launched cooperatively. The (token, key-tile) units are split
//    into equal contiguous ranges, one per CTA ("stream-K"); a token cut by a range boundary
//    is finished by the CTA holding its first tiles, which merges the other CTAs' partial
//    (o, max, sum) from the workspace in a fixed order (deterministic, no atomics on data).
//  * Warp roles: warp 0 producer (index read, -1 compaction, page translation, TMA gathers
//    for bf16 rows / L2 prefetch for FP8 rows, Q loads), warp 1 MMA issuer, warps 4-7 softmax
//    + epilogue (one per TMEM sub-partition, 16 heads each), warps 8-15 (FP8 only) dequant:
//    they load packed rows and write bf16(code * scale) into the 128-byte-swizzled K tile.
//  * Online softmax in the exp2 domain with a lazy rescale (O and the running sum are only
//    rescaled when the running max grows by more than 2^8), zero-RoPE work compiled out.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

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
  static constexpr int MSTAGES = 4;
  static constexpr int KCH = DK / 64;              // 128-byte chunks along d
  static constexpr int PCH = (BN + 63) / 64;       // 128-byte chunks of P along keys
  static constexpr int HALF = BN / 2;              // keys per softmax thread
  static constexpr int RB = D_NOPE + 4 * (D_NOPE / 128) + 2 * D_ROPE;
  static constexpr int ROWB = KIND == DSA_CACHE_BF16 ? 2 * DK : RB;  // cache row bytes
  static constexpr int NDEQ = KIND == DSA_CACHE_FP8_SCALED ? 8 : 0;
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
  int* flags;     // [G][4] partial published, one flag per softmax warp (16 heads)
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
    dsa_attn_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ CUtensorMap tmap_q,
                    const __grid_constant__ CUtensorMap tmap_kv) {
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
      mbar_init(k_full(s), C::KIND == DSA_CACHE_BF16 ? 1 : C::NDEQ);
      mbar_init(k_empty(s), 1);
    }
    for (int s = 0; s < C::MSTAGES; ++s) {
      mbar_init(m_full(s), 1);
      mbar_init(m_empty(s), 1 + 4 + C::NDEQ);
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
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmap_q);
    if (C::KIND == DSA_CACHE_BF16) prefetch_tmap(&tmap_kv);
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
    if (mbar_wait(bar, par)) return true;
    fail(DSA_DEVERR_TIMEOUT);
    return false;
  };

  if (warp == 0) {
    // =========================================================== producer (one warp) ====
    uint32_t mc = 0, g = 0, qc = 0;
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
      bool had = false;
      for (int j = j0; j < j1 && !*abort_flag; ++j) {
        // --- read this tile's index window, mask, translate, compact
        int slot_k[C::IDX_PER_LANE];
        bool ok_k[C::IDX_PER_LANE];
        int bad = 0;
#pragma unroll
        for (int k = 0; k < C::IDX_PER_LANE; ++k) {
          const int e = j * C::BN + 32 * k + lane;
          ok_k[k] = false;
          slot_k[k] = 0;
          if (32 * k + lane < C::BN && e < p.topk) {
            const int64_t pos = irow[e];
            if (pos >= 0) {
              int64_t slot;
              if (!p.bt) {
                slot = pos < p.num_slots ? pos : -2;
              } else if (pos >= (int64_t)p.max_pages * p.page_size) {
                slot = -2;
              } else {
                const int64_t page = p.bt[req * p.bt_stride + pos / p.page_size];
                slot = page < 0 ? -2 : page * p.page_size + pos % p.page_size;
                if (slot >= p.num_slots) slot = -2;
              }
              if (slot >= 0) {
                ok_k[k] = true;
                slot_k[k] = (int)slot;
              } else {
                bad = 1;
              }
            }
          }
        }
        if (bad) set_err(p.err, DSA_DEVERR_INDEX_OUT_OF_RANGE);
        int n_valid = 0;
#pragma unroll
        for (int k = 0; k < C::IDX_PER_LANE; ++k) n_valid += __popc(__ballot_sync(0xffffffffu, ok_k[k]));
        if (n_valid == 0) continue;
        // --- Q of this segment (first non-empty tile)
        if (!had) {
          if (qc > 0) wait(q_empty, (qc - 1) & 1);
          if (lane == 0) mbar_arrive_expect_tx(q_full, C::Q_BYTES);
          __syncwarp();
          if (lane < C::KCH)
            tma_load_3d(sbase + C::Q_OFF + lane * (kHeads * 128), &tmap_q, 64 * lane, 0, (int)t, q_full);
          ++qc;
        }
        // --- meta entry with the compacted slot list
        int st;
        MetaHdr* mh = emit_begin(st);
        int* slots = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(mh) + 32);
        int cnt = 0;
#pragma unroll
        for (int k = 0; k < C::IDX_PER_LANE; ++k) {
          const uint32_t bal = __ballot_sync(0xffffffffu, ok_k[k]);
          if (ok_k[k]) {
            const int pos = cnt + __popc(bal & ((1u << lane) - 1u));
            slots[pos] = slot_k[k];
            if constexpr (C::KIND == DSA_CACHE_FP8_SCALED) {
              // pull the packed row into L2 ahead of the dequant warps' loads
              const uint8_t* row = p.cache + (int64_t)slot_k[k] * C::RB;
              const uintptr_t a = reinterpret_cast<uintptr_t>(row);
              const uintptr_t a0 = a & ~uintptr_t(15);
              uint32_t sz = (uint32_t)(((a + C::RB + 15) & ~uintptr_t(15)) - a0);
              const uintptr_t end = reinterpret_cast<uintptr_t>(p.cache) + (uintptr_t)p.num_slots * C::RB;
              if (a0 + sz > end) sz = (uint32_t)((end - a0) & ~uintptr_t(15));
              if (sz > 0)
                asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(a0), "r"(sz) : "memory");
            }
          }
          cnt += __popc(bal);
        }
        if (lane == 0) {
          mh->type = kTile;
          mh->vtoken = (int)vt;
          mh->n_valid = n_valid;
          mh->first = had ? 0 : 1;
        }
        had = true;
        emit_end(st);
        // --- bf16 rows: TMA gather straight into the swizzled K tile
        if constexpr (C::KIND == DSA_CACHE_BF16) {
          const int ks = g % C::KSTAGES;
          if (g >= (uint32_t)C::KSTAGES) wait(k_empty(ks), ((g / C::KSTAGES) & 1) ^ 1);
          if (lane == 0) mbar_arrive_expect_tx(k_full(ks), C::KT_BYTES);
          __syncwarp();
          const uint32_t kt = sbase + C::KT_OFF + ks * C::KT_BYTES;
          const int oob = (int)p.num_slots;  // rows past n_valid read out of bounds -> zeros
          for (int w = lane; w < (C::BN / 4) * C::KCH; w += 32) {
            const int q4 = w % (C::BN / 4), c = w / (C::BN / 4);
            const int r = 4 * q4;
            const int s0 = r + 0 < n_valid ? slots[r + 0] : oob;
            const int s1 = r + 1 < n_valid ? slots[r + 1] : oob;
            const int s2 = r + 2 < n_valid ? slots[r + 2] : oob;
            const int s3 = r + 3 < n_valid ? slots[r + 3] : oob;
            tma_gather4(kt + c * (C::BN * 128) + r * 128, &tmap_kv, 64 * c, s0, s1, s2, s3, k_full(ks));
          }
        }
        ++g;
      }
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
      int pend = -1, pend_first = 0, pend_dvh = 0;
      auto issue_pv = [&](uint32_t gg, int first, int dvh) {
        if (!wait(p_full, gg & 1)) return;
        tc_fence_after();
        const int ks = gg % C::KSTAGES;
        const uint32_t vbase = sbase + C::KT_OFF + ks * C::KT_BYTES + dvh * (C::DVC / 64) * (C::BN * 128);
        for (int kk = 0; kk < C::BN / 16; ++kk) {
          const uint32_t pa = sbase + C::P_OFF + (kk >> 2) * (kHeads * 128) + (kk & 3) * 32;
          const uint64_t ad = sw128_desc(pa, 16, 1024);
          const uint64_t bd = sw128_desc(vbase + kk * 16 * 128, C::BN * 128, 1024);
          mma_bf16(tmem + C::O_COL, ad, bd, idPV, (first && kk == 0) ? 0u : 1u);
        }
        mma_commit(k_empty(ks));
        mma_commit(pv_done);
      };
      while (!*abort_flag) {
        const int st = mc % C::MSTAGES;
        if (!wait(m_full(st), (mc / C::MSTAGES) & 1)) break;
        const MetaHdr* mh = reinterpret_cast<const MetaHdr*>(smem + C::META_OFF + st * C::META_BYTES);
        const int type = mh->type;
        if (type == kTile) {
          const int first = mh->first;
          const int dvh = mh->vtoken % C::DV_SPLIT;
          mbar_arrive(m_empty(st));
          if (first) {
            if (!wait(q_full, qc & 1)) break;
            ++qc;
          }
          const int ks = g % C::KSTAGES;
          if (!wait(k_full(ks), (g / C::KSTAGES) & 1)) break;
          if (g >= 2 && !wait(s_empty(g & 1), ((g >> 1) & 1) ^ 1)) break;
          tc_fence_after();
          const uint32_t kbase = sbase + C::KT_OFF + ks * C::KT_BYTES;
          for (int kk = 0; kk < C::DK / 16; ++kk) {
            const uint32_t qa = sbase + C::Q_OFF + (kk >> 2) * (kHeads * 128) + (kk & 3) * 32;
            const uint32_t ka = kbase + (kk >> 2) * (C::BN * 128) + (kk & 3) * 32;
            mma_bf16(tmem + C::S_COL + (g & 1) * C::BN, sw128_desc(qa, 16, 1024), sw128_desc(ka, 16, 1024), idS,
                     kk > 0 ? 1u : 0u);
          }
          mma_commit(s_full(g & 1));
          if (pend >= 0) issue_pv((uint32_t)pend, pend_first, pend_dvh);
          pend = (int)g;
          pend_first = first;
          pend_dvh = dvh;
          ++g;
        } else if (type == kSegEnd) {
          const int had = mh->had_tiles;
          mbar_arrive(m_empty(st));
          if (had) mma_commit(q_empty);
        } else {
          mbar_arrive(m_empty(st));
          ++mc;
          break;
        }
        ++mc;
      }
      if (pend >= 0 && !*abort_flag) issue_pv((uint32_t)pend, pend_first, pend_dvh);
      // drain: wait for every MMA this thread issued before TMEM can be released
      if (g > 0) mbar_wait(pv_done, (g - 1) & 1);
    }
    __syncwarp();
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
          uint32_t r[32];
#pragma unroll
          for (int c0 = 0; c0 < C::HALF; c0 += 32) {
            if (c0 + 32 <= C::HALF) {
              tmem_ld16x2_x32<C::HALF>(ta + c0, r);
            } else {
              // HALF not a multiple of 32: the last 24 / 16 / 8 columns
              if constexpr (C::HALF % 32 == 24) {
                tmem_ld16x2_x16<C::HALF>(ta + c0, r);
                tmem_ld16x2_x8<C::HALF>(ta + c0 + 16, r + 16);
              } else if constexpr (C::HALF % 32 == 16) {
                tmem_ld16x2_x16<C::HALF>(ta + c0, r);
              } else if constexpr (C::HALF % 32 == 8) {
                tmem_ld16x2_x8<C::HALF>(ta + c0, r);
              }
            }
            tc_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (c0 + i < C::HALF) s[c0 + i] = __uint_as_float(r[i]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(s_empty(g & 1));
        // mask and row max (the two threads of a head hold its two key halves)
        const int kbase = hf * C::HALF;
        float mx = -INFINITY;
#pragma unroll
        for (int i = 0; i < C::HALF; ++i) {
          if (kbase + i >= n_valid) s[i] = -INFINITY;
          mx = fmaxf(mx, s[i]);
        }
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        const float m_tile = mx * c;  // finite: every tile has at least one valid key
        const bool grow = m_tile > m_run + 8.0f;
        const float m_new = grow ? m_tile : m_run;
        const float alpha = grow ? exp2f(m_run - m_new) : 1.0f;  // exp2(-inf) = 0 on the first tile
        float rs = 0.0f;
        uint32_t pk[C::HALF / 2];
#pragma unroll
        for (int i = 0; i < C::HALF; i += 2) {
          const float p0 = (kbase + i < n_valid) ? exp2f(fmaf(s[i], c, -m_new)) : 0.0f;
          const float p1 = (kbase + i + 1 < n_valid) ? exp2f(fmaf(s[i + 1], c, -m_new)) : 0.0f;
          rs += p0 + p1;
          pk[i / 2] = f32x2_to_bf16x2(p0, p1);
        }
        l_part = l_part * alpha + rs;
        // P buffer reuse and O rescale need the previous PV to be complete
        if (g > 0 && !wait(pv_done, (g - 1) & 1)) break;
        tc_fence_after();
        if (grow && !first) {
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
            asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p.flags + 4 * b + sp), "r"(1) : "memory");
        } else {
          // complete token, or the head of a split token: merge parts b+1..last in order
          const int nparts = kind == kHead ? last - b : 0;
          bool ok = true;
          for (int k = 1; k <= nparts && ok; ++k) {
            int v = 0;
            for (uint32_t it = 0; it < (1u << 22); ++it) {
              asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p.flags + 4 * (b + k) + sp) : "memory");
              if (v) break;
              __nanosleep(64);
            }
            if (!v) ok = false;
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
            if (w_own > 0.0f) {
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
          if (nparts > 0) {
            __syncwarp();
            if (lane == 0)
              for (int k = 1; k <= nparts; ++k) p.flags[4 * (b + k) + sp] = 0;
          }
        }
        tc_fence_before();
      }
      ++mc;
    }
  } else if (warp >= 8) {
    // ==================================================== FP8 dequant (8 warps) ====
    if constexpr (C::KIND == DSA_CACHE_FP8_SCALED) {
      const int dw = warp - 8;
      constexpr int RPW = C::BN / C::NDEQ;  // rows per warp per tile
      constexpr int PARTS = C::D_NOPE / 256;
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
        uint2 codes[RPW][PARTS];
        float scl[RPW][PARTS];
        uint4 rope[RPW];
#pragma unroll
        for (int k = 0; k < RPW; ++k) {
          const int r = dw + C::NDEQ * k;
          if (r < n_valid) {
            const uint8_t* row = p.cache + (int64_t)slots[r] * C::RB;
#pragma unroll
            for (int pt = 0; pt < PARTS; ++pt) {
              const int d0 = 256 * pt + 8 * lane;
              codes[k][pt] = __ldg(reinterpret_cast<const uint2*>(row + d0));
              scl[k][pt] = __ldg(reinterpret_cast<const float*>(row + C::D_NOPE + 4 * (d0 / 128)));
            }
            if constexpr (C::D_ROPE > 0) {
              if (lane < C::D_ROPE / 8)
                rope[k] = __ldg(reinterpret_cast<const uint4*>(row + C::D_NOPE + 4 * (C::D_NOPE / 128)) + lane);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(m_empty(st));
        ++mc;
        const int ks = g % C::KSTAGES;
        if (g >= (uint32_t)C::KSTAGES && !wait(k_empty(ks), ((g / C::KSTAGES) & 1) ^ 1)) break;
        uint8_t* kt = smem + C::KT_OFF + ks * C::KT_BYTES;
#pragma unroll
        for (int k = 0; k < RPW; ++k) {
          const int r = dw + C::NDEQ * k;
          const bool v = r < n_valid;
#pragma unroll
          for (int pt = 0; pt < PARTS; ++pt) {
            const int d0 = 256 * pt + 8 * lane;
            uint4 o = make_uint4(0, 0, 0, 0);
            if (v) {
              const float sc = scl[k][pt];
              const uint32_t cw[2] = {codes[k][pt].x, codes[k][pt].y};
              uint32_t w[4];
#pragma unroll
              for (int q = 0; q < 2; ++q) {
                const float2 a = f16x2_to_f32x2(e4m3x2_to_f16x2((uint16_t)(cw[q] & 0xFFFFu)));
                const float2 bb = f16x2_to_f32x2(e4m3x2_to_f16x2((uint16_t)(cw[q] >> 16)));
                w[2 * q] = f32x2_to_bf16x2(__fmul_rn(a.x, sc), __fmul_rn(a.y, sc));
                w[2 * q + 1] = f32x2_to_bf16x2(__fmul_rn(bb.x, sc), __fmul_rn(bb.y, sc));
              }
              o = make_uint4(w[0], w[1], w[2], w[3]);
            }
            const int ch = d0 >> 6, gr = (d0 & 63) >> 3;
            *reinterpret_cast<uint4*>(kt + ch * (C::BN * 128) + r * 128 + ((gr ^ (r & 7)) << 4)) = o;
          }
          if constexpr (C::D_ROPE > 0) {
            if (lane < C::D_ROPE / 8) {
              const int ch = C::D_NOPE / 64 + (lane >> 3), gr = lane & 7;
              *reinterpret_cast<uint4*>(kt + ch * (C::BN * 128) + r * 128 + ((gr ^ (r & 7)) << 4)) =
                  v ? rope[k] : make_uint4(0, 0, 0, 0);
            }
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(k_full(ks));
        ++g;
      }
    }
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

struct Geometry {
  int d_nope, d_rope, d_v, dv_split;
};

static size_t ws_bytes_for(int sm_count) {
  // partial o [G][64][256] fp32 + (max, sum) [G][2][64] fp32 + flags [G][4] int32
  const size_t o = (size_t)sm_count * kHeads * 256 * 4;
  const size_t ml = (size_t)sm_count * 2 * kHeads * 4;
  const size_t fl = ((size_t)sm_count * 16 + 255) & ~size_t(255);
  return o + ml + fl;
}

template <class C>
static dsa_status_t launch(const dsa_attn_args_t* a, const DeviceInfo& dev, cudaStream_t stream) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(dsa_attn_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  });
  if (attr_err != cudaSuccess) return cuda_fail(attr_err);
  EncodeTiledFn encode;
  dsa_status_t st = get_encode_fn(&encode);
  if (st != DSA_OK) return st;

  CUtensorMap tq, tkv;
  {
    const cuuint64_t dims[3] = {(cuuint64_t)C::DK, (cuuint64_t)kHeads, (cuuint64_t)a->T};
    const cuuint64_t strides[2] = {(cuuint64_t)a->q_stride_h * 2, (cuuint64_t)a->q_stride_t * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)kHeads, 1};
    const cuuint32_t es[3] = {1, 1, 1};
    CUresult r = encode(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a->q), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cuda_fail(cudaErrorInvalidValue);
  }
  if (C::KIND == DSA_CACHE_BF16) {
    const cuuint64_t dims[2] = {(cuuint64_t)C::DK, (cuuint64_t)a->num_slots};
    const cuuint64_t strides[1] = {(cuuint64_t)C::DK * 2};
    const cuuint32_t box[2] = {64, 1};
    const cuuint32_t es[2] = {1, 1};
    CUresult r = encode(&tkv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(a->cache), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cuda_fail(cudaErrorInvalidValue);
  } else {
    tkv = tq;  // unused by the FP8 kernels
  }

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
  const size_t o_bytes = (size_t)dev.sm_count * kHeads * 256 * 4;
  p.ws_o = static_cast<float*>(a->workspace);
  p.ws_ml = reinterpret_cast<float*>(static_cast<uint8_t*>(a->workspace) + o_bytes);
  p.flags = reinterpret_cast<int*>(static_cast<uint8_t*>(a->workspace) + o_bytes + (size_t)dev.sm_count * 2 * kHeads * 4);
  p.err = a->error_word;
  p.T = a->T;
  p.NT = (a->topk + C::BN - 1) / C::BN;
  p.U = a->T * C::DV_SPLIT * (int64_t)p.NT;
  p.G = (int)(p.U < dev.sm_count ? p.U : dev.sm_count);

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
  cudaError_t e = cudaLaunchKernelEx(&cfg, dsa_attn_kernel<C>, p, tq, tkv);
  return e == cudaSuccess ? DSA_OK : cuda_fail(e);
}

using CfgBf16_256 = AttnCfg<DSA_CACHE_BF16, 256, 0, 1, 112, 3>;
using CfgFp8_256 = AttnCfg<DSA_CACHE_FP8_SCALED, 256, 0, 1, 112, 3>;
using CfgBf16_576 = AttnCfg<DSA_CACHE_BF16, 512, 64, 2, 64, 2>;
using CfgFp8_576 = AttnCfg<DSA_CACHE_FP8_SCALED, 512, 64, 2, 64, 2>;

static dsa_status_t validate(const dsa_attn_args_t* a) {
  if (!a) return DSA_ERR_INVALID_ARGUMENT;
  if (a->T < 0 || a->num_slots < 0) return DSA_ERR_INVALID_ARGUMENT;
  if (a->kind != DSA_CACHE_BF16 && a->kind != DSA_CACHE_FP8_SCALED) return DSA_ERR_INVALID_ARGUMENT;
  if (a->H != kHeads) return DSA_ERR_UNSUPPORTED;
  if (!((a->d_nope == 256 && a->d_rope == 0 && a->d_v == 256) || (a->d_nope == 512 && a->d_rope == 64 && a->d_v == 512)))
    return DSA_ERR_UNSUPPORTED;
  if (a->topk < 1 || a->topk > 16384) return DSA_ERR_INVALID_ARGUMENT;
  if (!(a->sm_scale >= 0.0f) || !(a->sm_scale < 3.0e38f)) return DSA_ERR_INVALID_ARGUMENT;
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
  *bytes = ws_bytes_for(dev.sm_count);
  return DSA_OK;
}

dsa_status_t dsa_sparse_attn(const dsa_attn_args_t* a, void* stream) {
  dsa_status_t st = validate(a);
  if (st != DSA_OK || a->T == 0) return st;
  DeviceInfo dev;
  st = current_device(&dev);
  if (st != DSA_OK) return st;
  if (a->workspace_bytes < ws_bytes_for(dev.sm_count)) return DSA_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (a->d_nope == 256) {
    if (a->kind == DSA_CACHE_BF16) return launch<CfgBf16_256>(a, dev, s);
    return launch<CfgFp8_256>(a, dev, s);
  }
  if (a->kind == DSA_CACHE_BF16) return launch<CfgBf16_576>(a, dev, s);
  return launch<CfgFp8_576>(a, dev, s);
}

}  // extern "C"
