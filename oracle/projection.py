"""CPU oracle for the FP8 block-scaled projection GEMM (test infrastructure only).

The dense MLA projections around the attention (q_b_proj, o_proj) run, for prefill, as FP8
GEMMs on e4m3 operands with power-of-two block scales (sglang PR #31955 "Opt-in prefill-only FP8
dense projection GEMM for MLA q_b/o_proj", Motivation and Modifications: the bf16 weight is
repacked into e4m3 with one UE8M0 scale per 128x128 block; the activations are quantised the
same way per token and 128-column group, "a8w8 blockscale").

Definitions, written from those formats (the page gives no formula):
  * A block is block_rows x 128 elements of a matrix (128 x 128 for weights, 1 x 128 for
    activations). Its scale is s = 2^e, e the smallest integer with 448 * 2^e >= amax (amax the
    largest |x| of the block; e clamped to [-127, 127]; an all-zero block takes e = 0), stored
    as the UE8M0 byte e + 127.
  * Each element's code is e4m3 round-to-nearest-even of x / s (exact: s is a power of two, and
    |x / s| <= 448, the largest e4m3 value, so nothing saturates). Negative zero keeps its sign.
  * The product Y[m, n] = sum_k (code_x[m,k] * s_x[m, k/128]) * (code_w[n,k] * s_w[n/128, k/128]),
    computed here in fp64 on the exact dequantised values, then rounded to bf16 (RNE).

Only ``tests/`` and ``bench.py``'s CPU leg import this module.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def bf16_to_f64(bits) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def f64_to_bf16(x) -> np.ndarray:
    """Round-to-nearest-even of float64 values to bf16 bit patterns, directly from the fp64
    value (one rounding)."""
    x = np.asarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    flat, of = x.ravel(), out.ravel()
    for i, v in enumerate(flat):
        of[i] = _bf16_rne(float(v))
    return out


def _bf16_rne(v: float) -> int:
    import math

    if math.isnan(v):
        return 0x7FC0
    sign = 0x8000 if math.copysign(1.0, v) < 0 else 0
    a = abs(v)
    if a == 0.0:
        return sign
    if math.isinf(a):
        return sign | 0x7F80
    m, e = math.frexp(a)  # a = m * 2^e, m in [0.5, 1)
    E = e - 1              # a = (2m) * 2^E, 2m in [1, 2)
    if E < -126:           # subnormal range: quantum 2^-133
        q = 2.0 ** -133
    else:
        q = 2.0 ** (E - 7)
    n = a / q              # exact in fp64 for bf16-range inputs of fp64 precision
    r = round(n)           # Python round: half to even
    val = r * q
    if val >= 2.0 ** 128:  # overflow rounds to infinity
        return sign | 0x7F80
    # encode val
    if val == 0.0:
        return sign
    m2, e2 = math.frexp(val)
    E2 = e2 - 1
    if E2 < -126:
        return sign | int(round(val / 2.0 ** -133))
    mant = int(round((val / 2.0 ** E2 - 1.0) * 128))
    return sign | ((E2 + 127) << 7) | mant


def e4m3_decode(codes) -> np.ndarray:
    """float64 values of e4m3 codes (0x7F / 0xFF, NaN, are never produced here)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    ex = (c >> 3) & 0xF
    man = c & 0x7
    val = np.where(ex == 0, man * 2.0 ** -9, (1.0 + man / 8.0) * np.power(2.0, ex - 7))
    return sign * val


def e4m3_encode(v) -> np.ndarray:
    """e4m3 round-to-nearest-even codes of float64 values with |v| <= 448 (the sign of zero kept)."""
    v = np.asarray(v, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint8)
    flat, of = v.ravel(), out.ravel()
    for i, x in enumerate(flat):
        of[i] = _e4m3_rne(float(x))
    return out


def _e4m3_rne(x: float) -> int:
    import math

    sign = 0x80 if math.copysign(1.0, x) < 0 else 0
    a = abs(x)
    if a > E4M3_MAX:
        raise ValueError("outside the e4m3 range")
    if a == 0.0:
        return sign
    m, e = math.frexp(a)
    E = max(e - 1, -6)          # normal exponents -6 .. 8; below -6 the subnormal quantum 2^-9
    q = 2.0 ** (E - 3)
    n = round(a / q)            # half to even
    if n == 0:
        return sign
    val = n * q
    m2, e2 = math.frexp(val)
    E2 = e2 - 1
    if E2 < -6:
        return sign | int(n)    # subnormal: mantissa = val / 2^-9
    return sign | ((E2 + 7) << 3) | (int(round(val / 2.0 ** (E2 - 3))) - 8)


def block_exponent(amax: float) -> int:
    """Smallest e in [-127, 127] with 448 * 2^e >= amax (0 for amax == 0)."""
    import math

    if amax == 0.0:
        return 0
    m, ex = math.frexp(amax / E4M3_MAX)
    e = ex if m != 0.5 else ex - 1  # amax/448 = m 2^ex; a power of two m = 1/2 needs ex - 1
    # correct for the rounding of amax / 448 in fp64 by exact comparisons
    while e > -127 and E4M3_MAX * 2.0 ** (e - 1) >= amax:
        e -= 1
    while E4M3_MAX * 2.0 ** e < amax:
        e += 1
    return max(-127, min(127, e))


def quant_blockscale(x_bits, block_rows: int):
    """e4m3 codes uint8 [R, C] and scale exponents int [ceil(R / block_rows), C / 128] of a bf16
    matrix (C a multiple of 128)."""
    x = bf16_to_f64(x_bits)
    R, C = x.shape
    if C % 128:
        raise ValueError("columns must be a multiple of 128")
    nbr = (R + block_rows - 1) // block_rows
    exps = np.zeros((nbr, C // 128), dtype=np.int64)
    codes = np.zeros((R, C), dtype=np.uint8)
    for bi in range(nbr):
        r0, r1 = bi * block_rows, min(R, (bi + 1) * block_rows)
        for bj in range(C // 128):
            blk = x[r0:r1, 128 * bj:128 * (bj + 1)]
            e = block_exponent(float(np.abs(blk).max()))
            exps[bi, bj] = e
            codes[r0:r1, 128 * bj:128 * (bj + 1)] = e4m3_encode(blk / 2.0 ** e)
    return codes, exps


def dequant(codes, exps, block_rows: int) -> np.ndarray:
    """float64 values code * 2^e of a block-scaled matrix."""
    v = e4m3_decode(codes)
    s = np.power(2.0, np.repeat(np.repeat(exps, block_rows, axis=0)[: v.shape[0]], 128, axis=1).astype(np.float64))
    return v * s


def proj_gemm(x_codes, x_exps, w_codes, w_exps) -> np.ndarray:
    """bf16 bits [M, N] of Y = X W^T over the exact dequantised operands (fp64 products and sums),
    X [M, K] with 1 x 128 blocks, W [N, K] with 128 x 128 blocks."""
    x = dequant(x_codes, x_exps, 1)
    w = dequant(w_codes, w_exps, 128)
    return f64_to_bf16(x @ w.T)
