// dsa_proj.cu - FP8 block-scaled projection GEMM for the dense MLA projections around the
// attention (q_b_proj, o_proj), on sm_103a.
//
// What is computed (sglang PR #31955 "Opt-in prefill-only FP8 dense projection GEMM for MLA
// q_b/o_proj", Motivation and Modifications): the weight is repacked into e4m3 with one UE8M0
// (power-of-two) scale per 128x128 block, the activations into e4m3 with one UE8M0 scale per
// token and 128-column group ("a8w8 blockscale"), and Y = X W^T runs on the 8-bit operands.
//  * Quantisation (dsa_quant_fp8_blockscale): per block, e = the smallest integer with
//    448 * 2^e >= amax (an all-zero block takes e = 0), found on the bits of amax: for
//    amax = m * 2^E (m in [1, 2)), e = E - 8 when m <= 1.75 and E - 7 otherwise, clamped to
//    [-127, 127]; code = e4m3 round-to-nearest-even of x * 2^-e (exact scaling, |x * 2^-e| <= 448,
//    so the saturating hardware conversion never saturates).
//  * The scales go straight into the layout of the tensor core's 32-element block scales: a
//    128-column block's exponent byte is four identical 32-element scales. Scale tiles cover 128
//    rows x 4 scale columns (512 bytes, row r at (r % 32) * 16 + ((r % 128) / 32) * 4), ordered
//    row tile major, then column tile.
//  * The product (dsa_proj_gemm) is a plain library GEMM: cuBLASLt with e4m3 operands, those
//    32-element UE8M0 block scales, fp32 accumulation and bf16 output.
#include <cublasLt.h>
#include <cuda_runtime.h>

#include <map>
#include <mutex>
#include <tuple>

#include "dsa_host.h"
#include "dsa_ptx.cuh"

namespace dsa {
namespace proj {

// byte offset of (row r, 32-element scale column c) in the block-scale layout of a matrix with
// `cols` columns (a multiple of 128)
__host__ __device__ __forceinline__ int64_t sf_offset(int64_t r, int64_t c, int64_t cols) {
  const int64_t col_tiles = cols / 128;
  return ((r / 128) * col_tiles + c / 4) * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4 + (c % 4);
}

// UE8M0 exponent of a block whose largest magnitude has the fp32 bits `abits` (sign clear)
__device__ __forceinline__ int block_exponent(uint32_t abits) {
  if (abits == 0u) return 0;
  const int E = (int)(abits >> 23) - 127;
  if (E < -119) return -127;  // subnormal or tiny amax: e would fall below -127
  const int e = E - 8 + ((abits & 0x7FFFFFu) > 0x600000u ? 1 : 0);
  return e > 127 ? 127 : e;
}

__device__ __forceinline__ float pow2f(int e) { return __uint_as_float((uint32_t)(e + 127) << 23); }

// Activation rows: one half warp per (row, 128-column block), lane l of it columns 8l .. 8l + 7
// (16-byte loads); the block maximum by four xor shuffles inside the half warp.
__global__ void __launch_bounds__(256) quant_rows_kernel(const uint16_t* __restrict__ x, int64_t rows, int64_t cols,
                                                         int64_t stride, uint8_t* __restrict__ codes,
                                                         uint8_t* __restrict__ scales) {
  const int hl = threadIdx.x & 15;
  const int64_t w = (int64_t)blockIdx.x * 16 + (threadIdx.x >> 4);  // block index
  const int64_t nb = cols / 128;
  const bool live = w < rows * nb;
  const int64_t r = live ? w / nb : 0, j = live ? w - r * nb : 0;
  const uint4 v = live ? *reinterpret_cast<const uint4*>(x + r * stride + 128 * j + 8 * hl) : make_uint4(0u, 0u, 0u, 0u);
  const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
  uint32_t a = 0u;
#pragma unroll
  for (int i = 0; i < 4; ++i) a = max(a, max((w4[i] << 16) & 0x7FFFFFFFu, w4[i] & 0x7FFF0000u));
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) a = max(a, __shfl_xor_sync(0xffffffffu, a, o));  // within the half warp
  if (!live) return;
  const int e = block_exponent(a);
  const float inv = pow2f(-e);
  uint32_t o2[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint16_t lo = f32x2_to_e4m3x2(__uint_as_float(w4[2 * h] << 16) * inv, __uint_as_float(w4[2 * h] & 0xFFFF0000u) * inv);
    const uint16_t hi = f32x2_to_e4m3x2(__uint_as_float(w4[2 * h + 1] << 16) * inv,
                                        __uint_as_float(w4[2 * h + 1] & 0xFFFF0000u) * inv);
    o2[h] = (uint32_t)lo | ((uint32_t)hi << 16);
  }
  *reinterpret_cast<uint2*>(codes + r * cols + 128 * j + 8 * hl) = make_uint2(o2[0], o2[1]);
  if (hl == 0)
    *reinterpret_cast<uint32_t*>(scales + sf_offset(r, 4 * j, cols)) = 0x01010101u * (uint32_t)(e + 127);
}

// Weight blocks: one CTA of 256 threads per 128 x 128 block; thread t takes row t / 2, columns
// 64 (t % 2) .. + 63 of the block.
__global__ void __launch_bounds__(256) quant_blocks_kernel(const uint16_t* __restrict__ x, int64_t rows, int64_t cols,
                                                           int64_t stride, uint8_t* __restrict__ codes,
                                                           uint8_t* __restrict__ scales) {
  __shared__ uint32_t wmax[8];
  const int t = threadIdx.x, lane = t & 31;
  const int64_t bi = blockIdx.y, bj = blockIdx.x;
  const int64_t r = bi * 128 + (t >> 1);
  const int64_t c0 = bj * 128 + 64 * (t & 1);
  const bool live = r < rows;
  uint4 v[8];
#pragma unroll
  for (int k = 0; k < 8; ++k)
    v[k] = live ? *reinterpret_cast<const uint4*>(x + r * stride + c0 + 8 * k) : make_uint4(0u, 0u, 0u, 0u);
  uint32_t a = 0u;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint32_t w4[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) a = max(a, max((w4[i] << 16) & 0x7FFFFFFFu, w4[i] & 0x7FFF0000u));
  }
  a = __reduce_max_sync(0xffffffffu, a);
  if (lane == 0) wmax[t >> 5] = a;
  __syncthreads();
  a = 0u;
#pragma unroll
  for (int k = 0; k < 8; ++k) a = max(a, wmax[k]);
  const int e = block_exponent(a);
  const float inv = pow2f(-e);
  if (live) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint32_t w4[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
      uint32_t o[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint16_t lo = f32x2_to_e4m3x2(__uint_as_float(w4[2 * h] << 16) * inv, __uint_as_float(w4[2 * h] & 0xFFFF0000u) * inv);
        const uint16_t hi = f32x2_to_e4m3x2(__uint_as_float(w4[2 * h + 1] << 16) * inv,
                                            __uint_as_float(w4[2 * h + 1] & 0xFFFF0000u) * inv);
        o[h] = (uint32_t)lo | ((uint32_t)hi << 16);
      }
      *reinterpret_cast<uint2*>(codes + r * cols + c0 + 8 * k) = make_uint2(o[0], o[1]);
    }
  }
  // the block's 128 rows x 4 scale columns are one 512-byte tile, all the same byte (rows past
  // the matrix included: the GEMM reads whole tiles)
  if (t < 128) reinterpret_cast<uint32_t*>(scales + (bi * (cols / 128) + bj) * 512)[t] = 0x01010101u * (uint32_t)(e + 127);
}

// ---------------------------------------------------------------------------- cuBLASLt --
struct Lt {
  cublasLtHandle_t h = nullptr;
  std::map<std::tuple<int64_t, int64_t, int64_t, int64_t, size_t>, cublasLtMatmulAlgo_t> algos;
};

}  // namespace proj
}  // namespace dsa

using namespace dsa;

extern "C" int64_t dsa_blockscale_bytes(int64_t rows, int64_t cols) {
  if (rows <= 0 || cols <= 0 || cols % 128) return -1;
  return ((rows + 127) / 128) * (cols / 128) * 512;
}

extern "C" dsa_status_t dsa_quant_fp8_blockscale(const void* x, int64_t rows, int64_t cols, int64_t row_stride,
                                                 int block_rows, void* codes, void* scales, void* stream) {
  if (rows < 0 || cols <= 0 || cols % 128 || (block_rows != 1 && block_rows != 128)) return DSA_ERR_INVALID_ARGUMENT;
  if (rows == 0) return DSA_OK;
  if (!x || !codes || !scales || row_stride < cols || row_stride % 8) return DSA_ERR_INVALID_ARGUMENT;
  if (!aligned(x, 16) || !aligned(codes, 16) || !aligned(scales, 16)) return DSA_ERR_INVALID_ARGUMENT;
  DeviceInfo dev;
  dsa_status_t st = current_device(&dev);
  if (st != DSA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // rows past the matrix in the last scale tile read as scale 1
  cudaError_t e = cudaMemsetAsync(scales, 127, (size_t)dsa_blockscale_bytes(rows, cols), s);
  if (e != cudaSuccess) return cuda_fail(e);
  const uint16_t* xp = static_cast<const uint16_t*>(x);
  if (block_rows == 1) {
    const int64_t blocks = rows * (cols / 128);
    proj::quant_rows_kernel<<<(unsigned)((blocks + 15) / 16), 256, 0, s>>>(xp, rows, cols, row_stride,
                                                                        static_cast<uint8_t*>(codes),
                                                                        static_cast<uint8_t*>(scales));
  } else {
    const dim3 grid((unsigned)(cols / 128), (unsigned)((rows + 127) / 128));
    proj::quant_blocks_kernel<<<grid, 256, 0, s>>>(xp, rows, cols, row_stride, static_cast<uint8_t*>(codes),
                                                   static_cast<uint8_t*>(scales));
  }
  e = cudaGetLastError();
  return e == cudaSuccess ? DSA_OK : cuda_fail(e);
}

extern "C" dsa_status_t dsa_proj_gemm(const void* x_codes, const void* x_scales, const void* w_codes,
                                      const void* w_scales, int64_t M, int64_t N, int64_t K, void* y, int64_t y_stride,
                                      void* workspace, size_t workspace_bytes, void* stream) {
  if (M < 0 || N <= 0 || K <= 0 || N % 128 || K % 128) return DSA_ERR_INVALID_ARGUMENT;
  if (M == 0) return DSA_OK;
  if (!x_codes || !x_scales || !w_codes || !w_scales || !y || y_stride < N || y_stride % 8)
    return DSA_ERR_INVALID_ARGUMENT;
  if (!aligned(x_codes, 16) || !aligned(w_codes, 16) || !aligned(x_scales, 16) || !aligned(w_scales, 16) ||
      !aligned(y, 16) || (workspace_bytes && (!workspace || !aligned(workspace, 256))))
    return DSA_ERR_INVALID_ARGUMENT;
  if (M > 0x7FFFFFFFLL || N > 0x7FFFFFFFLL || K > 0x7FFFFFFFLL) return DSA_ERR_UNSUPPORTED;
  DeviceInfo dev;
  dsa_status_t st = current_device(&dev);
  if (st != DSA_OK) return st;

  static std::mutex mu;
  static proj::Lt lt[64];
  if (dev.device < 0 || dev.device >= 64) return DSA_ERR_NO_DEVICE;
  std::lock_guard<std::mutex> lock(mu);
  proj::Lt& L = lt[dev.device];
  if (!L.h && cublasLtCreate(&L.h) != CUBLAS_STATUS_SUCCESS) return DSA_ERR_CUDA;

  // column-major view: D[N x M] = W^T-view (A, K x N stored, transposed) times X-view (B, K x M)
  cublasLtMatmulDesc_t op = nullptr;
  cublasLtMatrixLayout_t la = nullptr, lb = nullptr, ld = nullptr;
  cublasLtMatmulPreference_t pref = nullptr;
  dsa_status_t ret = DSA_ERR_CUDA;
  do {
    if (cublasLtMatmulDescCreate(&op, CUBLAS_COMPUTE_32F, CUDA_R_32F) != CUBLAS_STATUS_SUCCESS) break;
    const cublasOperation_t ta = CUBLAS_OP_T, tb = CUBLAS_OP_N;
    const cublasLtMatmulMatrixScale_t mode = CUBLASLT_MATMUL_MATRIX_SCALE_VEC32_UE8M0;
    const void* sa = w_scales;
    const void* sb = x_scales;
    if (cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_TRANSA, &ta, sizeof(ta)) ||
        cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_TRANSB, &tb, sizeof(tb)) ||
        cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_A_SCALE_MODE, &mode, sizeof(mode)) ||
        cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_B_SCALE_MODE, &mode, sizeof(mode)) ||
        cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_A_SCALE_POINTER, &sa, sizeof(sa)) ||
        cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_B_SCALE_POINTER, &sb, sizeof(sb)))
      break;
    if (cublasLtMatrixLayoutCreate(&la, CUDA_R_8F_E4M3, (uint64_t)K, (uint64_t)N, K) ||
        cublasLtMatrixLayoutCreate(&lb, CUDA_R_8F_E4M3, (uint64_t)K, (uint64_t)M, K) ||
        cublasLtMatrixLayoutCreate(&ld, CUDA_R_16BF, (uint64_t)N, (uint64_t)M, y_stride))
      break;
    const auto key = std::make_tuple(M, N, K, y_stride, workspace_bytes);
    auto it = L.algos.find(key);
    if (it == L.algos.end()) {
      if (cublasLtMatmulPreferenceCreate(&pref) ||
          cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_MAX_WORKSPACE_BYTES, &workspace_bytes,
                                               sizeof(workspace_bytes)))
        break;
      cublasLtMatmulHeuristicResult_t res{};
      int n = 0;
      if (cublasLtMatmulAlgoGetHeuristic(L.h, op, la, lb, ld, ld, pref, 1, &res, &n) != CUBLAS_STATUS_SUCCESS || n < 1) {
        ret = DSA_ERR_UNSUPPORTED;
        break;
      }
      it = L.algos.emplace(key, res.algo).first;
    }
    const float alpha = 1.0f, beta = 0.0f;
    if (cublasLtMatmul(L.h, op, &alpha, w_codes, la, x_codes, lb, &beta, y, ld, y, ld, &it->second, workspace,
                       workspace_bytes, static_cast<cudaStream_t>(stream)) != CUBLAS_STATUS_SUCCESS)
      break;
    ret = DSA_OK;
  } while (false);
  if (pref) cublasLtMatmulPreferenceDestroy(pref);
  if (ld) cublasLtMatrixLayoutDestroy(ld);
  if (lb) cublasLtMatrixLayoutDestroy(lb);
  if (la) cublasLtMatrixLayoutDestroy(la);
  if (op) cublasLtMatmulDescDestroy(op);
  return ret;
}
