/*
 * dsa_oracle.c - plain CPU oracle for DSA sparse MLA attention over a latent KV cache.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path links, loads or calls this file:
 * only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline / reference arms use it.
 * It shares no code, header, table or constant generator with the CUDA library.
 *
 * What it computes (sglang PR #38547 "Enable zero-RoPE TileLang DSA on gfx950"):
 *   - the packed scaled-FP8 cache row (Contract table, "scaled FP8 cache row"):
 *       [d_nope e4m3 codes][d_nope/128 fp32 scales, little endian][d_rope bf16 values]
 *     = 264 bytes for 256+0, 656 bytes for 512+64;
 *   - quant_k_cache / dequant_k_cache (Scope list) and the paged gather of rows
 *     (Contract table, "paged dequant/gather");
 *   - the sparse attention that the pages' tests use as their reference, written out step by
 *     step (Direct GLM geometry coverage list): per query token, gather the top-k latent rows
 *     named by its index list, mask entries < 0, score every head against every gathered row,
 *     softmax, and take the weighted sum of the same latent rows (the first d_v elements) as
 *     values.
 *
 * Readings where the pages are silent (each is also listed in the design notes):
 *   - scale = amax / 448 in fp32 (one IEEE division); codes = e4m3_rne_satfinite(x / scale),
 *     one IEEE fp32 division per element; an all-zero tile stores scale 0 and codes 0.
 *   - negative zero and negative values that round to zero keep their sign (code 0x80).
 *   - any index < 0 is masked; an index outside the addressable range is masked as well and
 *     counted as a caller error.
 *   - a token with no valid entry produces a zero output row and lse = -inf.
 *   - the dequantised value used by attention is the exact product e4m3(code) * scale (exact in
 *     double); the gather/dequant helper output is bf16_rne(fp32(e4m3(code) * scale)).
 *
 * Arithmetic: attention is fp64 throughout (scores, max, exp, sums, weighted values).
 * Build: gcc -O2 -fopenmp -ffp-contract=off (no fast-math; float ops must be plain IEEE).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------- e4m3 (OCP FP8 E4M3FN) --
 * Format: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits. No infinities. The code
 * S.1111.111 is NaN; the largest finite magnitude is 1.75 * 2^8 = 448 (S.1111.110). Exponent
 * field 0 encodes subnormals m * 2^-9.                                                       */

double oracle_e4m3_value(uint8_t code) {
  int s = code >> 7, e = (code >> 3) & 15, m = code & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m, -9);              /* subnormal: (m/8) * 2^(1-7) */
  else
    v = ldexp((double)(8 + m), e - 10);    /* normal: (1 + m/8) * 2^(e-7) */
  return s ? -v : v;
}

/* Round a finite float to the nearest e4m3 value, ties to the even mantissa, saturating
 * magnitudes at or above 448 to 448 (satfinite). The sign is kept for zero results.        */
uint8_t oracle_e4m3_encode(float x) {
  uint8_t sign = signbit(x) ? 0x80 : 0x00;
  double a = fabs((double)x), q, n, r, val;
  int ex, E;
  if (isnan(x)) return (uint8_t)(sign | 0x7F);
  if (a >= 448.0) return (uint8_t)(sign | 0x7E);
  if (a == 0.0) return sign;
  /* spacing of e4m3 values around a: 2^(E-3) for a in [2^E, 2^(E+1)), E >= -6;
     below 2^-6 the subnormal spacing 2^-9 continues down to zero. */
  frexp(a, &ex);
  E = ex - 1;
  if (E < -6) E = -6;
  q = ldexp(1.0, E - 3);
  n = a / q;                 /* exact: division by a power of two */
  r = nearbyint(n);          /* default rounding mode: nearest, ties to even */
  val = r * q;               /* the rounded magnitude (an e4m3 value) */
  if (val == 0.0) return sign;
  if (val < ldexp(1.0, -6)) return (uint8_t)(sign | (int)(val / ldexp(1.0, -9)));
  frexp(val, &ex);
  {
    int e = (ex - 1) + 7;                                       /* biased exponent */
    int m = (int)(val / ldexp(1.0, (ex - 1) - 3)) - 8;          /* 3-bit mantissa */
    return (uint8_t)(sign | (e << 3) | m);
  }
}

/* ------------------------------------------------------------------------ bf16 <-> float -- */
static float bf16_bits_to_float(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* Round a float to bf16, nearest with ties to even (finite inputs; NaN stays NaN). */
uint16_t oracle_float_to_bf16(float f) {
  uint32_t u, kept, rest;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x0040);
  kept = u >> 16;
  rest = u & 0xFFFFu;
  if (rest > 0x8000u || (rest == 0x8000u && (kept & 1u))) kept += 1u;
  return (uint16_t)kept;
}

/* --------------------------------------------------------------------- packed row layout -- */
int64_t oracle_packed_row_bytes(int d_nope, int d_rope) {
  return (int64_t)d_nope + 4 * (int64_t)(d_nope / 128) + 2 * (int64_t)d_rope;
}

static float read_f32_le(const uint8_t* p) {
  uint32_t u = (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
  float f;
  memcpy(&f, &u, 4);
  return f;
}

static void write_f32_le(uint8_t* p, float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  p[0] = (uint8_t)u; p[1] = (uint8_t)(u >> 8); p[2] = (uint8_t)(u >> 16); p[3] = (uint8_t)(u >> 24);
}

/* quant_k_cache: pack n latent rows into the scaled-FP8 layout.
 *   k_nope: bf16 bits, row i at k_nope + i*nope_stride (d_nope values)
 *   k_rope: bf16 bits, row i at k_rope + i*rope_stride (d_rope values), may be NULL iff d_rope == 0
 *   out_loc: destination slot of row i, or NULL for slot i
 * Returns the number of rows whose slot was outside [0, num_slots) (those rows are skipped). */
int64_t oracle_quant_k_cache(const uint16_t* k_nope, int64_t nope_stride, const uint16_t* k_rope,
                             int64_t rope_stride, int64_t n, int d_nope, int d_rope,
                             const int64_t* out_loc, uint8_t* cache, int64_t num_slots, int n_threads) {
  const int64_t rb = oracle_packed_row_bytes(d_nope, d_rope);
  const int tiles = d_nope / 128;
  int64_t bad = 0;
#ifdef _OPENMP
  if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel for schedule(static) reduction(+ : bad)
#endif
  for (int64_t i = 0; i < n; ++i) {
    int64_t slot = out_loc ? out_loc[i] : i;
    uint8_t* row;
    if (slot < 0 || slot >= num_slots) { bad += 1; continue; }
    row = cache + slot * rb;
    for (int j = 0; j < tiles; ++j) {
      const uint16_t* x = k_nope + i * nope_stride + 128 * j;
      float amax = 0.0f, scale;
      for (int k = 0; k < 128; ++k) {
        float v = fabsf(bf16_bits_to_float(x[k]));
        if (v > amax) amax = v;
      }
      scale = amax / 448.0f;
      for (int k = 0; k < 128; ++k)
        row[128 * j + k] = (amax == 0.0f) ? 0x00 : oracle_e4m3_encode(bf16_bits_to_float(x[k]) / scale);
      write_f32_le(row + d_nope + 4 * j, amax == 0.0f ? 0.0f : scale);
    }
    for (int k = 0; k < d_rope; ++k) {
      uint16_t b = k_rope[i * rope_stride + k];
      row[d_nope + 4 * tiles + 2 * k] = (uint8_t)(b & 0xFF);
      row[d_nope + 4 * tiles + 2 * k + 1] = (uint8_t)(b >> 8);
    }
  }
  return bad;
}

/* ----------------------------------------------------------------- slot translation (paged) --
 * Direct mode (block_table == NULL): the index is the slot.
 * Paged mode: the index is a logical position p of request r; its slot is
 *   block_table[r * bt_stride + p / page_size] * page_size + p % page_size.
 * Returns -1 for a masked entry (index < 0) and -2 for an entry outside the addressable range. */
static int64_t translate(int64_t idx, int64_t req, int64_t num_slots, const int32_t* block_table,
                         int64_t bt_stride, int page_size, int max_pages) {
  int64_t page, slot;
  if (idx < 0) return -1;
  if (!block_table) return idx < num_slots ? idx : -2;
  if (idx >= (int64_t)max_pages * page_size) return -2;
  page = block_table[req * bt_stride + idx / page_size];
  if (page < 0) return -2;
  slot = page * page_size + idx % page_size;
  return slot < num_slots ? slot : -2;
}

/* Exact dequantisation of one cache row into double: FP8 codes times their tile scale
 * (exact in double), then the RoPE bf16 values; a BF16 cache row is widened as is. */
static void dequant_row_exact(const uint8_t* cache, int kind, int64_t slot, int d_nope, int d_rope,
                              double* out) {
  if (kind == 0) {
    const uint16_t* r = (const uint16_t*)(cache) + slot * (int64_t)(d_nope + d_rope);
    for (int d = 0; d < d_nope + d_rope; ++d) out[d] = (double)bf16_bits_to_float(r[d]);
  } else {
    const int64_t rb = oracle_packed_row_bytes(d_nope, d_rope);
    const uint8_t* r = cache + slot * rb;
    const int tiles = d_nope / 128;
    for (int d = 0; d < d_nope; ++d)
      out[d] = oracle_e4m3_value(r[d]) * (double)read_f32_le(r + d_nope + 4 * (d / 128));
    for (int k = 0; k < d_rope; ++k) {
      const uint8_t* p = r + d_nope + 4 * tiles + 2 * k;
      out[d_nope + k] = (double)bf16_bits_to_float((uint16_t)(p[0] | (p[1] << 8)));
    }
  }
}

/* dequant_k_cache gather: out[i] = bf16 row for index i (zero row when masked).
 *   FP8 rows: bf16_rne(float(e4m3(code)) * scale) with one fp32 multiply; RoPE bits copied.
 *   BF16 rows: copied.
 * Returns the number of indices outside the addressable range (their rows are zero). */
int64_t oracle_gather_dequant(const uint8_t* cache, int kind, int64_t num_slots, int d_nope, int d_rope,
                              const int32_t* indices, int64_t n, const int32_t* block_table,
                              int64_t bt_stride, int page_size, int max_pages,
                              const int32_t* req_of_index, uint16_t* out) {
  const int D = d_nope + d_rope;
  const int64_t rb = oracle_packed_row_bytes(d_nope, d_rope);
  int64_t bad = 0;
  for (int64_t i = 0; i < n; ++i) {
    int64_t req = req_of_index ? req_of_index[i] : 0;
    int64_t slot = translate(indices[i], req, num_slots, block_table, bt_stride, page_size, max_pages);
    uint16_t* o = out + i * D;
    if (slot < 0) {
      if (slot == -2) bad += 1;
      memset(o, 0, sizeof(uint16_t) * D);
      continue;
    }
    if (kind == 0) {
      memcpy(o, (const uint16_t*)cache + slot * D, sizeof(uint16_t) * D);
    } else {
      const uint8_t* r = cache + slot * rb;
      for (int d = 0; d < d_nope; ++d) {
        float v = (float)oracle_e4m3_value(r[d]);
        float s = read_f32_le(r + d_nope + 4 * (d / 128));
        float prod = v * s;
        o[d] = oracle_float_to_bf16(prod);
      }
      for (int k = 0; k < d_rope; ++k) {
        const uint8_t* p = r + d_nope + 4 * (d_nope / 128) + 2 * k;
        o[d_nope + k] = (uint16_t)(p[0] | (p[1] << 8));
      }
    }
  }
  return bad;
}

/* ------------------------------------------------------------------------ sparse attention --
 * For each requested token t (tokens[k], or k itself when tokens == NULL) and head h:
 *   valid entries j: idx[t, j] >= 0 and addressable; row k_j = exact dequantised latent row
 *   s_j  = sm_scale * sum_d q[t,h,d] * k_j[d]            (d over d_nope + d_rope)
 *   m    = max_j s_j,  p_j = exp(s_j - m),  l = sum_j p_j
 *   out[t,h,:] = sum_j p_j * k_j[0:d_v] / l,   lse[t,h] = m + log(l)
 * Duplicate indices are separate terms. No valid entry: out = 0, lse = -inf.
 * q is bf16 bits; element (t,h,d) at q + t*q_stride_t + h*q_stride_h + d.
 * out is [n_tokens, H, d_v] double, lse is [n_tokens, H] double (may be NULL).
 * Returns the number of entries outside the addressable range (they are masked). */
int64_t oracle_sparse_attn(const uint16_t* q, int64_t q_stride_t, int64_t q_stride_h, int H,
                           const uint8_t* cache, int kind, int64_t num_slots, int d_nope, int d_rope,
                           int d_v, const int32_t* indices, int64_t idx_stride_t, int topk,
                           const int32_t* block_table, int64_t bt_stride, int page_size, int max_pages,
                           const int32_t* req_of_token, double sm_scale, const int64_t* tokens,
                           int64_t n_tokens, double* out, double* lse, int n_threads) {
  const int D = d_nope + d_rope;
  int64_t bad = 0;
#ifdef _OPENMP
  if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : bad)
#endif
  for (int64_t k = 0; k < n_tokens; ++k) {
    const int64_t t = tokens ? tokens[k] : k;
    const int64_t req = req_of_token ? req_of_token[t] : 0;
    double* rows = (double*)malloc(sizeof(double) * (size_t)topk * (size_t)D);
    double* qd = (double*)malloc(sizeof(double) * (size_t)D);
    double* s = (double*)malloc(sizeof(double) * (size_t)topk);
    int n = 0;
    /* explicit gather + mask */
    for (int j = 0; j < topk; ++j) {
      int64_t slot = translate(indices[t * idx_stride_t + j], req, num_slots, block_table, bt_stride,
                               page_size, max_pages);
      if (slot == -2) bad += 1;
      if (slot < 0) continue;
      dequant_row_exact(cache, kind, slot, d_nope, d_rope, rows + (int64_t)n * D);
      n += 1;
    }
    for (int h = 0; h < H; ++h) {
      double* o = out + (k * H + h) * (int64_t)d_v;
      double m = -INFINITY, l = 0.0;
      for (int d = 0; d < D; ++d) qd[d] = (double)bf16_bits_to_float(q[t * q_stride_t + h * q_stride_h + d]);
      for (int d = 0; d < d_v; ++d) o[d] = 0.0;
      if (n == 0) {
        if (lse) lse[k * H + h] = -INFINITY;
        continue;
      }
      /* score */
      for (int j = 0; j < n; ++j) {
        const double* r = rows + (int64_t)j * D;
        double acc = 0.0;
        for (int d = 0; d < D; ++d) acc += qd[d] * r[d];
        s[j] = sm_scale * acc;
        if (s[j] > m) m = s[j];
      }
      /* softmax and value */
      for (int j = 0; j < n; ++j) {
        const double p = exp(s[j] - m);
        const double* r = rows + (int64_t)j * D;
        l += p;
        for (int d = 0; d < d_v; ++d) o[d] += p * r[d];
      }
      for (int d = 0; d < d_v; ++d) o[d] /= l;
      if (lse) lse[k * H + h] = m + log(l);
    }
    free(rows);
    free(qd);
    free(s);
  }
  return bad;
}

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
