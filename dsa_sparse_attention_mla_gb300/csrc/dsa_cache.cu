// dsa_cache.cu - packed scaled-FP8 latent cache: quant_k_cache (pack rows) and the
// gather/dequant helper, plus the small host entry points shared by the library
// (status strings, row sizes, device checks).
//
// Row layout (sglang PR #38547 "Enable zero-RoPE TileLang DSA on gfx950", Contract table,
// "scaled FP8 cache row"): [d_nope e4m3 codes][d_nope/128 fp32 scales][d_rope bf16 RoPE],
// 264 bytes for 256+0 and 656 bytes for 512+64. quant_k_cache / dequant_k_cache follow the
// Scope list of the same page: the NoPE width sets the number of 128-element scale tiles and
// the RoPE tensor may be empty; direct and paged (block table) gathers.
//
// Both kernels are HBM-bound streams: one warp per row, 8-byte loads and 4/16-byte stores,
// grids sized from the row count. The pack is bit-exact by construction: amax over the
// tile, scale = amax / 448 with IEEE division, codes by IEEE division and the hardware RNE
// satfinite e4m3 conversion.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "dsa_host.h"
#include "dsa_ptx.cuh"

namespace dsa {

static thread_local int g_last_cuda_error = 0;

dsa_status_t cuda_fail(cudaError_t e) {
  g_last_cuda_error = static_cast<int>(e);
  return DSA_ERR_CUDA;
}

dsa_status_t current_device(DeviceInfo* out) {
  static std::mutex mu;
  static DeviceInfo cache[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= 64) return DSA_ERR_NO_DEVICE;
  std::lock_guard<std::mutex> lock(mu);
  DeviceInfo& d = cache[dev];
  if (d.device != dev) {
    DeviceInfo n;
    n.device = dev;
    if ((e = cudaDeviceGetAttribute(&n.sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&n.cc_major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&n.cc_minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
      return cuda_fail(e);
    int optin = 0;
    if ((e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess)
      return cuda_fail(e);
    n.smem_optin = static_cast<size_t>(optin);
    d = n;
  }
  if (d.cc_major != 10 || d.cc_minor != 3) return DSA_ERR_NO_DEVICE;
  *out = d;
  return DSA_OK;
}

// ----------------------------------------------------------------------------- pack kernel --
// Packs one 128-element tile held by a warp, lane l owning elements 4 l .. 4 l + 3 (x):
// amax over the tile, scale = amax / 448, codes = e4m3_rne_satfinite(x / scale) (IEEE divisions;
// an all-zero tile stores scale 0 and codes 0). Writes lane l's four codes to codes + 4 l and the
// scale (lane 0) to *scale_out.
__device__ __forceinline__ void pack_tile(const float (&x)[4], int lane, uint8_t* codes_out, float* scale_out) {
  float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  uint32_t codes = 0;
  float scale = 0.0f;
  if (amax > 0.0f) {
    scale = __fdiv_rn(amax, 448.0f);
    const uint16_t c01 = f32x2_to_e4m3x2(__fdiv_rn(x[0], scale), __fdiv_rn(x[1], scale));
    const uint16_t c23 = f32x2_to_e4m3x2(__fdiv_rn(x[2], scale), __fdiv_rn(x[3], scale));
    codes = (uint32_t)c01 | ((uint32_t)c23 << 16);
  }
  *reinterpret_cast<uint32_t*>(codes_out + 4 * lane) = codes;
  if (lane == 0) *scale_out = scale;
}

// One warp per row. For tile j, lane l owns elements [128 j + 4 l, 128 j + 4 l + 4).
template <int D_NOPE, int D_ROPE>
__global__ void __launch_bounds__(256) quant_k_cache_kernel(const uint16_t* __restrict__ k_nope, int64_t nope_stride,
                                                            const uint16_t* __restrict__ k_rope, int64_t rope_stride,
                                                            int64_t n, const int64_t* __restrict__ out_loc,
                                                            uint8_t* __restrict__ cache, int64_t num_slots,
                                                            int32_t* error_word) {
  constexpr int TILES = D_NOPE / 128;
  constexpr int64_t RB = D_NOPE + 4 * TILES + 2 * D_ROPE;
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= n) return;
  const int64_t slot = out_loc ? out_loc[row] : row;
  if (slot < 0 || slot >= num_slots) {
    if (lane == 0 && error_word) atomicOr(error_word, DSA_DEVERR_SLOT_OUT_OF_RANGE);
    return;
  }
  uint8_t* dst = cache + slot * RB;
  const uint16_t* src = k_nope + row * nope_stride;
#pragma unroll
  for (int j = 0; j < TILES; ++j) {
    const uint2 raw = *reinterpret_cast<const uint2*>(src + 128 * j + 4 * lane);
    float x[4];
    x[0] = __uint_as_float(raw.x << 16);
    x[1] = __uint_as_float(raw.x & 0xFFFF0000u);
    x[2] = __uint_as_float(raw.y << 16);
    x[3] = __uint_as_float(raw.y & 0xFFFF0000u);
    pack_tile(x, lane, dst + 128 * j, reinterpret_cast<float*>(dst + D_NOPE + 4 * j));
  }
  if constexpr (D_ROPE > 0) {
    // D_ROPE bf16 = 2*D_ROPE bytes copied as 4-byte words (the RoPE part starts 8-byte aligned)
    const uint32_t* rs = reinterpret_cast<const uint32_t*>(k_rope + row * rope_stride);
    uint32_t* rd = reinterpret_cast<uint32_t*>(dst + D_NOPE + 4 * TILES);
    for (int w = lane; w < D_ROPE / 2; w += 32) rd[w] = rs[w];
  }
}

// ------------------------------------------------------------------ gather / dequant kernel --
__device__ __forceinline__ int64_t translate_slot(int64_t idx, int64_t req, int64_t num_slots,
                                                  const int32_t* __restrict__ bt, int64_t bt_stride, int page_size,
                                                  int max_pages) {
  // -1: masked (idx < 0); -2: addresses no slot
  if (idx < 0) return -1;
  if (!bt) return idx < num_slots ? idx : -2;
  if (idx >= (int64_t)max_pages * page_size) return -2;
  const int64_t page = bt[req * bt_stride + idx / page_size];
  if (page < 0) return -2;
  const int64_t slot = page * page_size + idx % page_size;
  return slot < num_slots ? slot : -2;
}

// One warp per output row. FP8 rows: lane l converts codes [8 l, 8 l + 8) of each 256-wide part.
template <int KIND, int D_NOPE, int D_ROPE>
__global__ void __launch_bounds__(256) gather_dequant_kernel(const uint8_t* __restrict__ cache, int64_t num_slots,
                                                             const int32_t* __restrict__ indices, int64_t n,
                                                             const int32_t* __restrict__ bt, int64_t bt_stride,
                                                             int page_size, int max_pages,
                                                             const int32_t* __restrict__ req_of_index,
                                                             uint16_t* __restrict__ out, int32_t* error_word) {
  constexpr int D = D_NOPE + D_ROPE;
  constexpr int TILES = D_NOPE / 128;
  const int lane = threadIdx.x & 31;
  const int64_t i = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (i >= n) return;
  const int64_t req = req_of_index ? req_of_index[i] : 0;
  const int64_t slot = translate_slot(indices[i], req, num_slots, bt, bt_stride, page_size, max_pages);
  uint16_t* o = out + i * D;
  if (slot < 0) {
    if (slot == -2 && lane == 0 && error_word) atomicOr(error_word, DSA_DEVERR_INDEX_OUT_OF_RANGE);
    for (int w = lane; w < D / 8; w += 32) reinterpret_cast<uint4*>(o)[w] = make_uint4(0, 0, 0, 0);
    return;
  }
  if constexpr (KIND == DSA_CACHE_BF16) {
    const uint4* s = reinterpret_cast<const uint4*>(cache + slot * (int64_t)(2 * D));
    for (int w = lane; w < D / 8; w += 32) reinterpret_cast<uint4*>(o)[w] = s[w];
  } else {
    constexpr int64_t RB = D_NOPE + 4 * TILES + 2 * D_ROPE;
    const uint8_t* r = cache + slot * RB;
#pragma unroll
    for (int part = 0; part < D_NOPE / 256; ++part) {
      const int d0 = 256 * part + 8 * lane;
      const uint2 c = *reinterpret_cast<const uint2*>(r + d0);
      const float sc = *reinterpret_cast<const float*>(r + D_NOPE + 4 * (d0 / 128));
      uint32_t w[4];
      const uint32_t cw[2] = {c.x, c.y};
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const float2 a = f16x2_to_f32x2(e4m3x2_to_f16x2((uint16_t)(cw[k] & 0xFFFFu)));
        const float2 b = f16x2_to_f32x2(e4m3x2_to_f16x2((uint16_t)(cw[k] >> 16)));
        w[2 * k] = f32x2_to_bf16x2(__fmul_rn(a.x, sc), __fmul_rn(a.y, sc));
        w[2 * k + 1] = f32x2_to_bf16x2(__fmul_rn(b.x, sc), __fmul_rn(b.y, sc));
      }
      *reinterpret_cast<uint4*>(o + d0) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    if constexpr (D_ROPE > 0) {
      const uint32_t* rs = reinterpret_cast<const uint32_t*>(r + D_NOPE + 4 * TILES);
      uint32_t* rd = reinterpret_cast<uint32_t*>(o + D_NOPE);
      for (int w = lane; w < D_ROPE / 2; w += 32) rd[w] = rs[w];
    }
  }
}

// ----------------------------------------------------------------- gather / requant kernel --
// One warp per kRqRows rows: gather packed row indices[i] (direct or paged, as gather_dequant),
// widen each tile to bf16_rne(fp32(e4m3(code)) * scale) exactly as gather_dequant does, and pack
// those values again (pack_tile) into row out_loc[i] (or i) of `out`; RoPE bits are copied. A
// masked index, or one that addresses no slot, packs the zero row. The rows' index and page
// lookups run on separate lanes at once, and the warp loads all its rows before converting any,
// so that the dependent lookups and the row loads of many rows overlap.
// rows per warp (16 for 264-byte rows measured slower: the registers cost occupancy)
template <int D_NOPE>
constexpr int rq_rows() { return 8; }
template <int D_NOPE, int D_ROPE>
__global__ void __launch_bounds__(256) gather_requant_kernel(const uint8_t* __restrict__ cache, int64_t num_slots,
                                                             const int32_t* __restrict__ indices, int64_t n,
                                                             const int32_t* __restrict__ bt, int64_t bt_stride,
                                                             int page_size, int max_pages,
                                                             const int32_t* __restrict__ req_of_index,
                                                             const int64_t* __restrict__ out_loc, uint8_t* __restrict__ out,
                                                             int64_t out_slots, int32_t* error_word) {
  constexpr int TILES = D_NOPE / 128;
  constexpr int64_t RB = D_NOPE + 4 * TILES + 2 * D_ROPE;
  constexpr int RW = D_ROPE / 2;  // RoPE words (<= 32: one per lane)
  constexpr int kRqRows = rq_rows<D_NOPE>();
  const int lane = threadIdx.x & 31;
  const int64_t i0 = ((int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * kRqRows;
  if (i0 >= n) return;
  // lane r < kRqRows resolves row i0 + r (destination, request, source slot) for the warp
  int64_t my_d = -1, my_slot = -1;
  if (lane < kRqRows && i0 + lane < n) {
    const int64_t i = i0 + lane;
    const int64_t d = out_loc ? out_loc[i] : i;
    if (d < 0 || d >= out_slots) {
      if (error_word) atomicOr(error_word, DSA_DEVERR_SLOT_OUT_OF_RANGE);
    } else {
      my_d = d;
      const int64_t req = req_of_index ? req_of_index[i] : 0;
      my_slot = translate_slot(indices[i], req, num_slots, bt, bt_stride, page_size, max_pages);
      if (my_slot == -2 && error_word) atomicOr(error_word, DSA_DEVERR_INDEX_OUT_OF_RANGE);
    }
  }
  uint32_t c[kRqRows][TILES];
  float sc[kRqRows][TILES];
  uint32_t rw[kRqRows];
  int64_t dslot[kRqRows];
#pragma unroll
  for (int r = 0; r < kRqRows; ++r) {
    dslot[r] = __shfl_sync(0xffffffffu, my_d, r);
    const int64_t slot = __shfl_sync(0xffffffffu, my_slot, r);
    rw[r] = 0u;
#pragma unroll
    for (int j = 0; j < TILES; ++j) {
      c[r][j] = 0u;
      sc[r][j] = 0.0f;
    }
    if (dslot[r] < 0 || slot < 0) continue;
    const uint8_t* row = cache + slot * RB;
#pragma unroll
    for (int j = 0; j < TILES; ++j) {
      c[r][j] = *reinterpret_cast<const uint32_t*>(row + 128 * j + 4 * lane);
      sc[r][j] = *reinterpret_cast<const float*>(row + D_NOPE + 4 * j);
    }
    if (RW > 0 && lane < RW) rw[r] = reinterpret_cast<const uint32_t*>(row + D_NOPE + 4 * TILES)[lane];
  }
#pragma unroll
  for (int r = 0; r < kRqRows; ++r) {
    if (dslot[r] < 0) continue;  // (warp-uniform)
    uint8_t* dst = out + dslot[r] * RB;
#pragma unroll
    for (int j = 0; j < TILES; ++j) {
      // A tile as the pack writes it (a positive scale, largest code magnitude 448 = 0x7E) comes
      // back with the same codes and the scale fp32(bf16_rne(448 * scale) / 448): its widened
      // maximum is bf16_rne(448 * scale), and widening then dividing by the new scale moves every
      // value by at most about 2^-7.9 relative, less than half the e4m3 spacing (2^-4.9 relative
      // for normal codes, 2^-10 absolute for subnormal ones). Any other tile takes the general
      // widen-and-pack path.
      const uint32_t mag = c[r][j] & 0x7F7F7F7Fu;  // code magnitudes, one per byte
      uint32_t cmax = max(max(mag & 0xFFu, (mag >> 8) & 0xFFu), max((mag >> 16) & 0xFFu, mag >> 24));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) cmax = max(cmax, __shfl_xor_sync(0xffffffffu, cmax, o));
      const float s0 = sc[r][j];
      // (the scale bounds keep 448 * scale and its bf16 rounding finite, and every non-zero
      // product code * scale a normal number, where the error bound above holds)
      if (cmax == 0x7Eu && s0 >= 0x1p-117f && s0 <= 7.0e35f) {
        *reinterpret_cast<uint32_t*>(dst + 128 * j + 4 * lane) = c[r][j];
        if (lane == 0) {
          const uint32_t m = __float_as_uint(__fmul_rn(448.0f, s0));
          const float amax = __uint_as_float(((m + 0x7FFFu + ((m >> 16) & 1u)) >> 16) << 16);  // bf16_rne
          *reinterpret_cast<float*>(dst + D_NOPE + 4 * j) = __fdiv_rn(amax, 448.0f);
        }
        continue;
      }
      const float2 a = f16x2_to_f32x2(e4m3x2_to_f16x2((uint16_t)(c[r][j] & 0xFFFFu)));
      const float2 b = f16x2_to_f32x2(e4m3x2_to_f16x2((uint16_t)(c[r][j] >> 16)));
      const uint32_t w0 = f32x2_to_bf16x2(__fmul_rn(a.x, s0), __fmul_rn(a.y, s0));
      const uint32_t w1 = f32x2_to_bf16x2(__fmul_rn(b.x, s0), __fmul_rn(b.y, s0));
      const float x[4] = {__uint_as_float(w0 << 16), __uint_as_float(w0 & 0xFFFF0000u), __uint_as_float(w1 << 16),
                          __uint_as_float(w1 & 0xFFFF0000u)};
      pack_tile(x, lane, dst + 128 * j, reinterpret_cast<float*>(dst + D_NOPE + 4 * j));
    }
    if (RW > 0 && lane < RW) reinterpret_cast<uint32_t*>(dst + D_NOPE + 4 * TILES)[lane] = rw[r];
  }
}

}  // namespace dsa

using namespace dsa;

extern "C" {

const char* dsa_status_string(dsa_status_t s) {
  switch (s) {
    case DSA_OK: return "DSA_OK";
    case DSA_ERR_INVALID_ARGUMENT: return "DSA_ERR_INVALID_ARGUMENT";
    case DSA_ERR_UNSUPPORTED: return "DSA_ERR_UNSUPPORTED";
    case DSA_ERR_WORKSPACE_TOO_SMALL: return "DSA_ERR_WORKSPACE_TOO_SMALL";
    case DSA_ERR_CUDA: return "DSA_ERR_CUDA";
    case DSA_ERR_NO_DEVICE: return "DSA_ERR_NO_DEVICE";
  }
  return "DSA_ERR_UNKNOWN";
}

int dsa_last_cuda_error(void) { return g_last_cuda_error; }

int64_t dsa_packed_row_bytes(int d_nope, int d_rope) {
  if (d_nope <= 0 || d_nope % 128 != 0 || d_rope < 0) return -1;
  return (int64_t)d_nope + 4 * (int64_t)(d_nope / 128) + 2 * (int64_t)d_rope;
}

int64_t dsa_cache_row_bytes(dsa_cache_kind_t kind, int d_nope, int d_rope) {
  if (kind == DSA_CACHE_BF16) return (d_nope <= 0 || d_rope < 0) ? -1 : 2 * (int64_t)(d_nope + d_rope);
  if (kind == DSA_CACHE_FP8_SCALED) return dsa_packed_row_bytes(d_nope, d_rope);
  return -1;
}

dsa_status_t dsa_quant_k_cache(const void* k_nope, int64_t k_nope_row_stride, const void* k_rope,
                               int64_t k_rope_row_stride, int64_t n, int d_nope, int d_rope, const int64_t* out_loc,
                               void* cache, int64_t num_slots, int32_t* error_word, void* stream) {
  if (n < 0 || num_slots < 0) return DSA_ERR_INVALID_ARGUMENT;
  if (!((d_nope == 256 && d_rope == 0) || (d_nope == 512 && d_rope == 64)))
    return (d_nope > 0 && d_nope % 128 == 0 && d_rope >= 0) ? DSA_ERR_UNSUPPORTED : DSA_ERR_INVALID_ARGUMENT;
  if (n == 0) return DSA_OK;
  if (!k_nope || !cache || (d_rope > 0 && !k_rope) || (d_rope == 0 && k_rope)) return DSA_ERR_INVALID_ARGUMENT;
  if (k_nope_row_stride < d_nope || (k_nope_row_stride & 3) || !aligned(k_nope, 8)) return DSA_ERR_INVALID_ARGUMENT;
  if (d_rope > 0 && (k_rope_row_stride < d_rope || (k_rope_row_stride & 1) || !aligned(k_rope, 4)))
    return DSA_ERR_INVALID_ARGUMENT;
  if (!aligned(cache, 8)) return DSA_ERR_INVALID_ARGUMENT;
  if (!out_loc && n > num_slots) return DSA_ERR_INVALID_ARGUMENT;
  DeviceInfo dev;
  dsa_status_t st = current_device(&dev);
  if (st != DSA_OK) return st;
  const dim3 block(256);
  const dim3 grid((unsigned)((n + 7) / 8));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (d_nope == 256)
    quant_k_cache_kernel<256, 0><<<grid, block, 0, s>>>((const uint16_t*)k_nope, k_nope_row_stride, nullptr, 0, n,
                                                        out_loc, (uint8_t*)cache, num_slots, error_word);
  else
    quant_k_cache_kernel<512, 64><<<grid, block, 0, s>>>((const uint16_t*)k_nope, k_nope_row_stride,
                                                         (const uint16_t*)k_rope, k_rope_row_stride, n, out_loc,
                                                         (uint8_t*)cache, num_slots, error_word);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? DSA_OK : cuda_fail(e);
}

dsa_status_t dsa_gather_dequant(const void* cache, dsa_cache_kind_t kind, int64_t num_slots, int d_nope, int d_rope,
                                const int32_t* indices, int64_t n, const int32_t* block_table, int64_t bt_stride,
                                int page_size, int max_pages, const int32_t* req_of_index, void* out,
                                int32_t* error_word, void* stream) {
  if (n < 0 || num_slots < 0) return DSA_ERR_INVALID_ARGUMENT;
  if (kind != DSA_CACHE_BF16 && kind != DSA_CACHE_FP8_SCALED) return DSA_ERR_INVALID_ARGUMENT;
  if (!((d_nope == 256 && d_rope == 0) || (d_nope == 512 && d_rope == 64))) return DSA_ERR_UNSUPPORTED;
  if (n == 0) return DSA_OK;
  if (!cache || !indices || !out) return DSA_ERR_INVALID_ARGUMENT;
  if (!aligned(out, 16) || !aligned(cache, 16)) return DSA_ERR_INVALID_ARGUMENT;
  if (block_table && (page_size <= 0 || max_pages <= 0 || bt_stride < max_pages)) return DSA_ERR_INVALID_ARGUMENT;
  DeviceInfo dev;
  dsa_status_t st = current_device(&dev);
  if (st != DSA_OK) return st;
  const dim3 block(256);
  const dim3 grid((unsigned)((n + 7) / 8));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const uint8_t* c = static_cast<const uint8_t*>(cache);
  uint16_t* o = static_cast<uint16_t*>(out);
#define DSA_GD(K, DN, DR)                                                                                     \
  gather_dequant_kernel<K, DN, DR><<<grid, block, 0, s>>>(c, num_slots, indices, n, block_table, bt_stride, \
                                                          page_size, max_pages, req_of_index, o, error_word)
  if (kind == DSA_CACHE_BF16) {
    if (d_nope == 256) DSA_GD(DSA_CACHE_BF16, 256, 0); else DSA_GD(DSA_CACHE_BF16, 512, 64);
  } else {
    if (d_nope == 256) DSA_GD(DSA_CACHE_FP8_SCALED, 256, 0); else DSA_GD(DSA_CACHE_FP8_SCALED, 512, 64);
  }
#undef DSA_GD
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? DSA_OK : cuda_fail(e);
}

dsa_status_t dsa_gather_requant(const void* cache, int64_t num_slots, int d_nope, int d_rope, const int32_t* indices,
                                int64_t n, const int32_t* block_table, int64_t bt_stride, int page_size, int max_pages,
                                const int32_t* req_of_index, const int64_t* out_loc, void* out, int64_t out_slots,
                                int32_t* error_word, void* stream) {
  if (n < 0 || num_slots < 0 || out_slots < 0) return DSA_ERR_INVALID_ARGUMENT;
  if (!((d_nope == 256 && d_rope == 0) || (d_nope == 512 && d_rope == 64)))
    return (d_nope > 0 && d_nope % 128 == 0 && d_rope >= 0) ? DSA_ERR_UNSUPPORTED : DSA_ERR_INVALID_ARGUMENT;
  if (n == 0) return DSA_OK;
  if (!cache || !indices || !out) return DSA_ERR_INVALID_ARGUMENT;
  if (!aligned(cache, 8) || !aligned(out, 8)) return DSA_ERR_INVALID_ARGUMENT;
  if (!out_loc && n > out_slots) return DSA_ERR_INVALID_ARGUMENT;
  if (block_table && (page_size <= 0 || max_pages <= 0 || bt_stride < max_pages)) return DSA_ERR_INVALID_ARGUMENT;
  DeviceInfo dev;
  dsa_status_t st = current_device(&dev);
  if (st != DSA_OK) return st;
  const dim3 block(256);
  const int64_t rows_per_block = 8 * (d_nope == 256 ? rq_rows<256>() : rq_rows<512>());
  const dim3 grid((unsigned)((n + rows_per_block - 1) / rows_per_block));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const uint8_t* c = static_cast<const uint8_t*>(cache);
  uint8_t* o = static_cast<uint8_t*>(out);
  if (d_nope == 256)
    gather_requant_kernel<256, 0><<<grid, block, 0, s>>>(c, num_slots, indices, n, block_table, bt_stride, page_size,
                                                         max_pages, req_of_index, out_loc, o, out_slots, error_word);
  else
    gather_requant_kernel<512, 64><<<grid, block, 0, s>>>(c, num_slots, indices, n, block_table, bt_stride, page_size,
                                                          max_pages, req_of_index, out_loc, o, out_slots, error_word);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? DSA_OK : cuda_fail(e);
}

}  // extern "C"
