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
// floats. A four-pass radix select (8 bits per pass, most significant first, a shared-memory
// histogram per pass) finds the K-th largest key u*; the keys above u* are collected in any order
// (shared atomic counter) and the ties at u* in position order (a block-wide scan over the row in
// position order), so the choice among equal scores is the lowest positions. The K selected
// (key, position) pairs are then sorted by a bitonic network in shared memory on 64-bit words
// (~key << 32 | position) and written out. Every decision is on integer keys: the result is the
// same on every run.
#include <cuda_runtime.h>

#include <mutex>

#include "dsa_host.h"

namespace dsa {
namespace topk {

constexpr int kThreads = 1024;
constexpr int kMaxK = 16384;
constexpr int kPerThread = 4;  // contiguous positions per thread in the ordered tie scan

// Unsigned key with the order of the float values (-0.0 maps as +0.0).
__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t b = __float_as_uint(f);
  if (b == 0x80000000u) b = 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
// Ascending order of the composite = descending key, then ascending position.
__device__ __forceinline__ uint64_t compose(uint32_t key, uint32_t pos) { return ((uint64_t)(~key) << 32) | pos; }

// Exclusive scan of one value per thread over the block; returns the prefix and the total.
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_sums, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int x = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += x;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int w = warp_sums[lane];  // kThreads / 32 == 32 warps
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int x = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += x;
    }
    warp_sums[lane] = wi - w;  // exclusive prefix of each warp
    if (lane == 31) warp_sums[32] = wi;
  }
  __syncthreads();
  const int r = warp_sums[warp] + incl - v;
  total = warp_sums[32];
  __syncthreads();  // warp_sums is reused by the next call
  return r;
}

__global__ void __launch_bounds__(kThreads, 1)
    topk_kernel(const float* __restrict__ scores, int64_t S, int64_t stride, const int32_t* __restrict__ lengths, int K,
                int P, int32_t* __restrict__ out, int64_t out_stride) {
  extern __shared__ uint64_t buf[];  // P entries (P = next power of two >= K)
  __shared__ int hist[256];
  __shared__ int warp_sums[33];
  __shared__ uint32_t s_prefix;
  __shared__ int s_need, s_count;
  const int tid = threadIdx.x;
  const int64_t t = blockIdx.x;
  const float* row = scores + t * stride;
  int64_t n = S;
  if (lengths) {
    const int64_t l = lengths[t];
    n = l < 0 ? 0 : (l > S ? S : l);
  }
  int sel;  // positions selected
  if (n <= K) {
    sel = (int)n;
    for (int i = tid; i < sel; i += kThreads) buf[i] = compose(order_key(row[i]), (uint32_t)i);
  } else {
    // ---- radix select of the K-th largest key
    uint32_t prefix = 0u, mask = 0u;
    int need = K;  // how many of the keys matching the prefix still have to be taken from the top
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      for (int i = tid; i < 256; i += kThreads) hist[i] = 0;
      __syncthreads();
      for (int64_t i = tid; i < n; i += kThreads) {
        const uint32_t u = order_key(row[i]);
        if ((u & mask) == prefix) atomicAdd(&hist[(u >> shift) & 255u], 1);
      }
      __syncthreads();
      if (tid == 0) {
        int above = 0, d = 255;
        for (; d > 0; --d) {
          if (above + hist[d] >= need) break;
          above += hist[d];
        }
        s_prefix = prefix | ((uint32_t)d << shift);
        s_need = need - above;
      }
      __syncthreads();
      prefix = s_prefix;
      need = s_need;
      mask |= 255u << shift;
      __syncthreads();
    }
    const uint32_t ustar = prefix;  // the K-th largest key; `need` ties at ustar complete the K
    // ---- keys above u*: K - need of them, any order (the sort below orders them)
    if (tid == 0) s_count = 0;
    __syncthreads();
    for (int64_t i = tid; i < n; i += kThreads) {
      const uint32_t u = order_key(row[i]);
      if (u > ustar) buf[atomicAdd(&s_count, 1)] = compose(u, (uint32_t)i);
    }
    __syncthreads();
    const int base = K - need;
    // ---- ties at u*: the `need` lowest positions, by a scan over the row in position order
    int taken = 0;
    for (int64_t c0 = 0; c0 < n && taken < need; c0 += (int64_t)kThreads * kPerThread) {
      const int64_t i0 = c0 + (int64_t)tid * kPerThread;
      int mine = 0;
#pragma unroll
      for (int k = 0; k < kPerThread; ++k)
        if (i0 + k < n && order_key(row[i0 + k]) == ustar) ++mine;
      int total;
      int r = taken + block_exclusive_scan(mine, warp_sums, total);
#pragma unroll
      for (int k = 0; k < kPerThread; ++k) {
        if (i0 + k < n && order_key(row[i0 + k]) == ustar) {
          if (r < need) buf[base + r] = compose(ustar, (uint32_t)(i0 + k));
          ++r;
        }
      }
      taken += total;
    }
    sel = K;
  }
  // ---- bitonic sort of buf[0 .. P) (pad past `sel` with the largest word)
  for (int i = sel + tid; i < P; i += kThreads) buf[i] = ~0ull;
  __syncthreads();
  for (int k = 2; k <= P; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = tid; i < P; i += kThreads) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const uint64_t a = buf[i], bv = buf[ixj];
          const bool up = (i & k) == 0;
          if ((a > bv) == up) {
            buf[i] = bv;
            buf[ixj] = a;
          }
        }
      }
      __syncthreads();
    }
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
      const cudaError_t e = cudaFuncSetAttribute(topk::topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)((size_t)topk::kMaxK * sizeof(uint64_t)));
      if (e != cudaSuccess) return cuda_fail(e);
      done[dev.device] = true;
    }
  }
  int P = 1;
  while (P < K) P <<= 1;
  const size_t smem = (size_t)P * sizeof(uint64_t);
  topk::topk_kernel<<<(unsigned)T, topk::kThreads, smem, static_cast<cudaStream_t>(stream)>>>(
      S > 0 ? scores : nullptr, S, score_stride_t, lengths, K, P, indices, idx_stride_t);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? DSA_OK : cuda_fail(e);
}
