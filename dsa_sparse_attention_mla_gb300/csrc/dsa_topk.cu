// dsa_topk.cu - top-k index selection for sm_103a: the step that turns each query token's
// index-logits into the top-k position list the sparse attention gathers.
//
// What is computed (FreeToken PR #270 "glm5_next: support GLM-5.3-Flash", Summary, the DSA
// key-pooling bullet: pooled keys are scored and the best-scoring positions are the ones the
// sparse kernels read; sglang PR #38547 "Enable zero-RoPE TileLang DSA on gfx950", Direct GLM
// geometry coverage list: top-k widths 2048 and 2112, lists padded with -1): for row t, over
// positions 0 .. n_t - 1, the positions of the min(K, n_t) largest scores, in descending score
// order with equal scores in ascending position order (-0.0 equals +0.0), then -1 up to K.
//
// Kernel: one CTA per row (1024 threads). Scores map to unsigned keys that order like the
// floats; a row whose keys fit in shared memory (beside the sort buffer) is read from HBM once,
// with 16-byte loads, and every later pass reads the shared copy. A four-pass radix select (8
// bits per pass, most significant first) finds the K-th largest key u*: per pass each warp counts
// into its own 256-entry histogram (scores bunch in a few top digits, and one shared histogram
// would serialise the whole CTA on them), the 32 histograms are summed and one warp picks the
// digit. The keys above u* and the first ties at u* are collected in position order from
// per-warp chunks (a count pass, a scan over the warps, a write pass), so the choice among equal
// scores is the lowest positions. The K selected (key, position) pairs are then sorted by a
// bitonic network on 64-bit words (~key << 32 | position), in registers with shuffles for the
// steps inside a warp and shared memory for the steps between warps, and written out. Rows that
// fit two to an SM run two per SM. Every decision is on integer keys: the result is the same on
// every run.
#include <cuda_runtime.h>

#include <mutex>

#include "dsa_host.h"

namespace dsa {
namespace topk {

constexpr int kThreads = 1024;
constexpr int kMaxK = 16384;
constexpr int kSmemMax = 225 * 1024;  // dynamic shared memory per CTA: sort buffer + cached keys
constexpr int kCandCap = 2048;        // keys left after two radix passes that the one-SM rows keep aside

// Unsigned key with the order of the float values (-0.0 maps as +0.0).
__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t b = __float_as_uint(f);
  if (b == 0x80000000u) b = 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
// Ascending order of the composite = descending key, then ascending position.
__device__ __forceinline__ uint64_t compose(uint32_t key, uint32_t pos) { return ((uint64_t)(~key) << 32) | pos; }

// Bitonic sort of buf[0 .. P) ascending, P a power of two, in shared memory: every thread takes
// whole compare-exchange pairs (i, i + j) of each step. Ends synchronised.
__device__ __forceinline__ void sort_smem(uint64_t* buf, int P) {
  const int tid = threadIdx.x;
  for (int k = 2; k <= P; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int q = tid; q < (P >> 1); q += kThreads) {
        const int i = ((q & ~(j - 1)) << 1) | (q & (j - 1)), ixj = i | j;
        const uint64_t a = buf[i], bv = buf[ixj];
        const bool up = (i & k) == 0;
        if ((a > bv) == up) {
          buf[i] = bv;
          buf[ixj] = a;
        }
      }
      __syncthreads();
    }
  }
}

// The same network with P = 1024 E (E = 2 or 4: K up to 4096): thread t holds elements E t .. E t + E - 1 in registers.
// Steps whose partner is in the same thread (j < E) or the same warp (j < 32 E, a shuffle with
// lane t ^ (j / E)) stay in registers; only the steps between warps go through shared memory.
// The pair (i, i + j) of a step keeps the smaller word at i when (i & k) == 0, else the larger.
// Ends with buf sorted and synchronised.
template <int E>
__device__ __forceinline__ void sort_regs(uint64_t* buf, int P) {
  const int tid = threadIdx.x;
  uint64_t v[E];
#pragma unroll
  for (int e = 0; e < E; ++e) v[e] = buf[E * tid + e];
  for (int k = 2; k <= P; k <<= 1) {
    int j = k >> 1;
    if (j >= 32 * E) {
      __syncthreads();  // every thread's reads of the previous layout are done
#pragma unroll
      for (int e = 0; e < E; ++e) buf[E * tid + e] = v[e];
      __syncthreads();
      for (; j >= 32 * E; j >>= 1) {
        for (int q = tid; q < (P >> 1); q += kThreads) {
          const int i = ((q & ~(j - 1)) << 1) | (q & (j - 1)), ixj = i | j;
          const uint64_t a = buf[i], bv = buf[ixj];
          const bool up = (i & k) == 0;
          if ((a > bv) == up) {
            buf[i] = bv;
            buf[ixj] = a;
          }
        }
        __syncthreads();
      }
#pragma unroll
      for (int e = 0; e < E; ++e) v[e] = buf[E * tid + e];
    }
    // the direction bit (i & k) is the same for every slot of a thread from k = E on
    const bool up_t = ((E * tid) & k) == 0;
#pragma unroll
    for (int lm = 16; lm >= 1; lm >>= 1) {  // j = lm * E: partner lane tid ^ lm, same slot
      if (lm * E <= (k >> 1)) {
        const bool take_max = ((tid & lm) == 0) != up_t;  // keep the larger word
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const uint64_t x = v[e];
          const uint32_t plo = __shfl_xor_sync(0xffffffffu, (uint32_t)x, lm);
          const uint32_t phi = __shfl_xor_sync(0xffffffffu, (uint32_t)(x >> 32), lm);
          const uint64_t y = ((uint64_t)phi << 32) | plo;
          v[e] = ((x < y) != take_max) ? x : y;
        }
      }
    }
#pragma unroll
    for (int jj = E / 2; jj >= 1; jj >>= 1) {  // partner in the same thread
      if (jj <= (k >> 1)) {
#pragma unroll
        for (int e = 0; e < E; ++e) {
          if ((e & jj) == 0) {
            const uint64_t a = v[e], bv = v[e | jj];
            const bool up = ((E * tid + e) & k) == 0;
            if ((a > bv) == up) {
              v[e] = bv;
              v[e | jj] = a;
            }
          }
        }
      }
    }
  }
  __syncthreads();
#pragma unroll
  for (int e = 0; e < E; ++e) buf[E * tid + e] = v[e];
  __syncthreads();
}

// MINB: CTAs per SM the registers are budgeted for (2 when the shared memory lets two rows run
// on an SM at once, which hides more of each row's synchronisation).
template <int MINB>
__global__ void __launch_bounds__(kThreads, MINB)
    topk_kernel(const float* __restrict__ scores, int64_t S, int64_t stride, const int32_t* __restrict__ lengths, int K,
                int P, int64_t kcap, int32_t* __restrict__ out, int64_t out_stride) {
  extern __shared__ uint64_t buf[];  // P entries (P = next power of two >= K), 32 warp histograms, candidates, kcap keys
  int* whist = reinterpret_cast<int*>(buf + P);  // [32 warps][256 digits]
  uint2* cand = reinterpret_cast<uint2*>(whist + 32 * 256);  // [kCandCap] (key, position)
  uint32_t* keys = reinterpret_cast<uint32_t*>(cand + kCandCap);
  __shared__ int hist[256];
  __shared__ int warp_sums[33];
  __shared__ int s_cnt_t[32];
  __shared__ uint32_t s_prefix;
  __shared__ int s_need, s_cand;
  const int tid = threadIdx.x;
  const int64_t t = blockIdx.x;
  const float* row = scores + t * stride;
  int64_t n = S;
  if (lengths) {
    const int64_t l = lengths[t];
    n = l < 0 ? 0 : (l > S ? S : l);
  }
  int sel;  // positions selected
  // the row's keys: from the shared copy when the row fits, else from global memory
  const bool cached = n > K && n <= kcap;
  if (cached) {
    if ((reinterpret_cast<uintptr_t>(row) & 15u) == 0) {  // 16-byte loads, four keys at a time
      const int64_t n4 = n >> 2;
      const float4* r4 = reinterpret_cast<const float4*>(row);
      uint4* k4 = reinterpret_cast<uint4*>(keys);
#pragma unroll 4
      for (int64_t i = tid; i < n4; i += kThreads) {
        const float4 f = __ldg(r4 + i);
        k4[i] = make_uint4(order_key(f.x), order_key(f.y), order_key(f.z), order_key(f.w));
      }
      for (int64_t i = 4 * n4 + tid; i < n; i += kThreads) keys[i] = order_key(row[i]);
    } else {
#pragma unroll 8
      for (int64_t i = tid; i < n; i += kThreads) keys[i] = order_key(row[i]);
    }
    __syncthreads();
  }
  auto key_at = [&](int64_t i) -> uint32_t { return cached ? keys[i] : order_key(row[i]); };
  if (n <= K) {
    sel = (int)n;
    for (int i = tid; i < sel; i += kThreads) buf[i] = compose(order_key(row[i]), (uint32_t)i);
  } else {
    // ---- radix select of the K-th largest key
    const int lane = tid & 31, warp = tid >> 5;
    const uint32_t lt_mask = (1u << lane) - 1u;
    uint32_t prefix = 0u, mask = 0u;
    int need = K;  // how many of the keys matching the prefix still have to be taken from the top
    // One-SM rows (long rows): after two passes over the row, one more pass sets aside the keys
    // that already rank above the 16-bit prefix of u* (into the list, any order) and the keys
    // that match it (candidates, when at most kCandCap); passes 2 and 3 and the final collection
    // then read only the candidates. na16 / nc16: this warp's keys above / at the prefix, read
    // off its histograms (positions warp * 32 + lane + 1024 k).
    int na16 = 0, nc16 = 0;
    bool filtered = false;
    int ncand = 0, abv16 = 0;  // candidates, and the keys above the 16-bit prefix (written first)
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      int* wh = whist + 256 * warp;
      if (!filtered) {
        for (int i = lane; i < 256; i += 32) wh[i] = 0;
        __syncwarp();
#pragma unroll 4
        for (int64_t i = tid; i < n; i += kThreads) {
          const uint32_t u = key_at(i);
          if ((u & mask) == prefix) atomicAdd(&wh[(u >> shift) & 255u], 1);
        }
      } else {
        for (int i = tid; i < 256; i += kThreads) hist[i] = 0;
        __syncthreads();
        for (int j = tid; j < ncand; j += kThreads) {
          const uint32_t u = cand[j].x;
          if ((u & mask) == prefix) atomicAdd(&hist[(u >> shift) & 255u], 1);
        }
      }
      __syncthreads();
      if (!filtered && tid < 256) {
        int c = 0;
#pragma unroll 8
        for (int w = 0; w < 32; ++w) c += whist[256 * w + tid];
        hist[tid] = c;
      }
      __syncthreads();
      if (warp == 0) {
        // lane l holds digits 255 - 8 l .. 248 - 8 l, top first; the chosen digit d is the first
        // from the top at which the running count reaches `need`
        int cnt[8], tot = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          cnt[j] = hist[255 - 8 * lane - j];
          tot += cnt[j];
        }
        int incl = tot;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int x = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += x;
        }
        int above = incl - tot;
        if (above < need && need <= incl) {
          int d = 255 - 8 * lane;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (above + cnt[j] >= need) break;
            above += cnt[j];
            --d;
          }
          s_prefix = prefix | ((uint32_t)d << shift);
          s_need = need - above;
          s_cand = hist[d];  // keys matching the new prefix
        }
      }
      __syncthreads();
      prefix = s_prefix;
      need = s_need;
      if constexpr (MINB == 1) {
        if (pass <= 1) {
          const uint32_t dsel = (prefix >> shift) & 255u;
          int a = 0;
#pragma unroll
          for (int j = 0; j < 8; ++j) a += (uint32_t)(8 * lane + j) > dsel ? wh[8 * lane + j] : 0;
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
          na16 += a;
          if (pass == 1) nc16 = wh[dsel];
        }
      }
      mask |= 255u << shift;
      __syncthreads();
      if constexpr (MINB == 1) {
        if (pass == 1 && s_cand <= kCandCap) {
          // the pass that sets the keys aside: per-warp offsets by a scan of na16 / nc16
          if (lane == 0) {
            warp_sums[warp] = na16;
            s_cnt_t[warp] = nc16;
          }
          __syncthreads();
          if (warp == 0) {
            const int a = warp_sums[lane], b2 = s_cnt_t[lane];
            int ia = a, ib = b2;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
              const int xa = __shfl_up_sync(0xffffffffu, ia, o), xb = __shfl_up_sync(0xffffffffu, ib, o);
              if (lane >= o) {
                ia += xa;
                ib += xb;
              }
            }
            warp_sums[lane] = ia - a;
            s_cnt_t[lane] = ib - b2;
          }
          __syncthreads();
          int oa = warp_sums[warp], oc = s_cnt_t[warp];
          for (int64_t c0 = 32 * warp; c0 < n; c0 += kThreads) {
            const int64_t i = c0 + lane;
            const uint32_t u = i < n ? key_at(i) : 0u;
            const bool ab = i < n && (u & mask) > prefix, cd = i < n && (u & mask) == prefix;
            const uint32_t ba = __ballot_sync(0xffffffffu, ab), bc = __ballot_sync(0xffffffffu, cd);
            if (ab) buf[oa + __popc(ba & lt_mask)] = compose(u, (uint32_t)i);
            if (cd) cand[oc + __popc(bc & lt_mask)] = make_uint2(u, (uint32_t)i);
            oa += __popc(ba);
            oc += __popc(bc);
          }
          ncand = s_cand;
          abv16 = K - need;
          filtered = true;
          __syncthreads();
        }
      }
    }
    const uint32_t ustar = prefix;  // the K-th largest key; `need` ties at ustar complete the K
    const int base = K - need;      // the ties follow the keys above u*
    bool ties_left = true;          // the position-ordered tie pass below still has to run
    if (filtered) {
      // the candidates above u* after the keys set aside, and the ties too when every one of
      // them is taken (warp-aggregated slots; the sort orders them)
      const bool all_ties = s_cand == need;
      if (tid == 0) {
        s_cnt_t[0] = 0;
        s_cnt_t[1] = 0;
      }
      __syncthreads();
      for (int j0 = 0; j0 < ncand; j0 += kThreads) {
        const int j = j0 + tid;
        const uint2 c = j < ncand ? cand[j] : make_uint2(0u, 0u);
        const bool ab = j < ncand && c.x > ustar, ti = all_ties && j < ncand && c.x == ustar;
        const uint32_t ba = __ballot_sync(0xffffffffu, ab), bt = __ballot_sync(0xffffffffu, ti);
        int wa = 0, wt = 0;
        if (lane == 0) {
          if (ba) wa = atomicAdd(&s_cnt_t[0], __popc(ba));
          if (bt) wt = atomicAdd(&s_cnt_t[1], __popc(bt));
        }
        wa = __shfl_sync(0xffffffffu, wa, 0);
        wt = __shfl_sync(0xffffffffu, wt, 0);
        if (ab) buf[abv16 + wa + __popc(ba & lt_mask)] = compose(c.x, c.y);
        if (ti) buf[base + wt + __popc(bt & lt_mask)] = compose(c.x, c.y);
      }
      ties_left = !all_ties;
      __syncthreads();
    }
    // ---- the keys above u* (K - need of them) and the first `need` ties at u* in position
    // order. Warp w takes the contiguous positions [w cs, (w + 1) cs): a first pass counts its
    // keys above and at u*, a scan over the warps gives each warp its offsets, and a second pass
    // writes them (ballot ranks: position order within the warp, and warps in position order).
    if (ties_left) {
      const bool take_above = !filtered;  // (set aside and collected above otherwise)
      const int64_t cs = ((n + 32 * 32 - 1) / (32 * 32)) * 32;  // a multiple of 32 positions per warp
      const int64_t w0 = (int64_t)warp * cs, w1 = w0 + cs < n ? w0 + cs : n;
      int na = 0, nt = 0;
      for (int64_t c0 = w0; c0 < w1; c0 += 32) {
        const int64_t i = c0 + lane;
        const uint32_t u = i < w1 ? key_at(i) : 0u;
        na += __popc(__ballot_sync(0xffffffffu, take_above && i < w1 && u > ustar));
        nt += __popc(__ballot_sync(0xffffffffu, i < w1 && u == ustar));
      }
      if (lane == 0) {
        warp_sums[warp] = na;
        s_cnt_t[warp] = nt;
      }
      __syncthreads();
      if (warp == 0) {
        const int a = warp_sums[lane], b = s_cnt_t[lane];
        int ia = a, ib = b;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int xa = __shfl_up_sync(0xffffffffu, ia, o), xb = __shfl_up_sync(0xffffffffu, ib, o);
          if (lane >= o) {
            ia += xa;
            ib += xb;
          }
        }
        warp_sums[lane] = ia - a;  // exclusive offsets
        s_cnt_t[lane] = ib - b;
      }
      __syncthreads();
      int oa = warp_sums[warp], ot = s_cnt_t[warp];
      for (int64_t c0 = w0; c0 < w1 && ((take_above && oa < base) || ot < need); c0 += 32) {
        const int64_t i = c0 + lane;
        const uint32_t u = i < w1 ? key_at(i) : 0u;
        const bool ab = take_above && i < w1 && u > ustar, ti = i < w1 && u == ustar;
        const uint32_t ba = __ballot_sync(0xffffffffu, ab), bt = __ballot_sync(0xffffffffu, ti);
        if (ab) buf[oa + __popc(ba & lt_mask)] = compose(u, (uint32_t)i);
        if (ti) {
          const int r = ot + __popc(bt & lt_mask);
          if (r < need) buf[base + r] = compose(ustar, (uint32_t)i);
        }
        oa += __popc(ba);
        ot += __popc(bt);
      }
    }
    sel = K;
  }
  // ---- bitonic sort of buf[0 .. P) (pad past `sel` with the largest word)
  for (int i = sel + tid; i < P; i += kThreads) buf[i] = ~0ull;
  __syncthreads();
  switch (P) {
    case 2048: sort_regs<2>(buf, P); break;
    case 4096: sort_regs<4>(buf, P); break;
    default: sort_smem(buf, P); break;
  }
  int32_t* orow = out + t * out_stride;
  for (int i = tid; i < K; i += kThreads) orow[i] = i < sel ? (int32_t)(uint32_t)(buf[i] & 0xFFFFFFFFull) : -1;
}

}  // namespace topk
}  // namespace dsa

using namespace dsa;

extern "C" dsa_status_t dsa_topk_select(const float* scores, int64_t T, int64_t S, int64_t score_stride_t,
                                        const int32_t* lengths, int K, int32_t* indices, int64_t idx_stride_t,
                                        void* stream) {
  if (T < 0 || S < 0 || K < 1 || K > topk::kMaxK) return DSA_ERR_INVALID_ARGUMENT;
  if (S > 0x7FFFFFFFLL) return DSA_ERR_UNSUPPORTED;
  if (T == 0) return DSA_OK;
  if (!indices || idx_stride_t < K || (S > 0 && (!scores || score_stride_t < S))) return DSA_ERR_INVALID_ARGUMENT;
  if (!aligned(indices, 4) || (scores && !aligned(scores, 4)) || (lengths && !aligned(lengths, 4)))
    return DSA_ERR_INVALID_ARGUMENT;
  DeviceInfo dev;
  dsa_status_t st = current_device(&dev);
  if (st != DSA_OK) return st;
  {  // one-time set-up per device: the kernel's dynamic shared-memory limit
    static std::mutex mu;
    static bool done[64] = {};
    if (dev.device < 0 || dev.device >= 64) return DSA_ERR_NO_DEVICE;
    std::lock_guard<std::mutex> lock(mu);
    if (!done[dev.device]) {
      cudaError_t e = cudaFuncSetAttribute(topk::topk_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, topk::kSmemMax);
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(topk::topk_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, topk::kSmemMax);
      if (e != cudaSuccess) return cuda_fail(e);
      done[dev.device] = true;
    }
  }
  int P = 1;
  while (P < K) P <<= 1;
  // keys cached per row: as many as fit beside the sort buffer, and no more than the row has
  // (rows longer than that read global memory in every pass)
  const int64_t room =
      ((int64_t)topk::kSmemMax - (int64_t)P * (int64_t)sizeof(uint64_t) - 32 * 256 * 4 - topk::kCandCap * 8) / 4;
  const int64_t kcap = S < room ? S : room;
  const size_t smem = (size_t)P * sizeof(uint64_t) + 32 * 256 * 4 + topk::kCandCap * 8 + (size_t)kcap * 4;
  const float* sp = S > 0 ? scores : nullptr;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (smem <= (size_t)(110 * 1024))  // two CTAs fit the SM's shared memory
    topk::topk_kernel<2><<<(unsigned)T, topk::kThreads, smem, cs>>>(sp, S, score_stride_t, lengths, K, P, kcap, indices,
                                                                     idx_stride_t);
  else
    topk::topk_kernel<1><<<(unsigned)T, topk::kThreads, smem, cs>>>(sp, S, score_stride_t, lengths, K, P, kcap, indices,
                                                                     idx_stride_t);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? DSA_OK : cuda_fail(e);
}
