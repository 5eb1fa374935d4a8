"""Pins of the FP8 block-scaled projection oracle (oracle/projection.py) against the e4m3 and
bf16 formats and closed forms: every e4m3 code round-trips, every midpoint between neighbouring
codes rounds to the even one, the block exponent is the smallest power of two that keeps the
block within 448, quantisation errors stay within half a code spacing, and the product equals
brute-force sums (exactly, where every term and sum is representable)."""
import numpy as np
import pytest

from oracle import projection as P


def _finite_codes():
    return np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)


def test_every_e4m3_code_round_trips():
    c = _finite_codes()
    v = P.e4m3_decode(c)
    assert np.array_equal(P.e4m3_encode(v), c)
    assert P.e4m3_decode(np.array([0x7E], np.uint8))[0] == 448.0
    assert P.e4m3_decode(np.array([0x01], np.uint8))[0] == 2.0 ** -9
    assert P.e4m3_decode(np.array([0x08], np.uint8))[0] == 2.0 ** -6


def test_midpoints_round_to_even_and_neighbours_to_nearest():
    pos = np.arange(0, 0x7E, dtype=np.uint8)  # 0x00 .. 0x7D and their successors
    lo, hi = P.e4m3_decode(pos), P.e4m3_decode(pos + 1)
    mid = (lo + hi) / 2
    even = np.where(pos % 2 == 0, pos, pos + 1).astype(np.uint8)
    assert np.array_equal(P.e4m3_encode(mid), even)
    assert np.array_equal(P.e4m3_encode(-mid), even | 0x80)
    gap = hi - lo
    assert np.array_equal(P.e4m3_encode(mid - gap / 64), pos)
    assert np.array_equal(P.e4m3_encode(mid + gap / 64), (pos + 1).astype(np.uint8))
    assert P.e4m3_encode(np.array([-0.0]))[0] == 0x80


def test_bf16_rounding_matches_the_format():
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 0x7F80, size=4000).astype(np.uint16)  # finite positive bf16
    v = P.bf16_to_f64(bits)
    assert np.array_equal(P.f64_to_bf16(v), bits)
    nxt = P.bf16_to_f64(bits + 1)
    mid = (v + nxt) / 2
    assert np.array_equal(P.f64_to_bf16(mid), np.where(bits % 2 == 0, bits, bits + 1).astype(np.uint16))


@pytest.mark.parametrize("k", [-30, -8, 0, 5, 100])
def test_block_exponent_closed_forms(k):
    assert P.block_exponent(448.0 * 2.0 ** k) == k
    assert P.block_exponent(448.0 * 2.0 ** k * (1 + 2.0 ** -20)) == k + 1
    assert P.block_exponent(448.0 * 2.0 ** k * 0.5000001) == k
    assert P.block_exponent(448.0 * 2.0 ** k * 0.5) == k - 1


def test_block_exponent_edges():
    assert P.block_exponent(0.0) == 0
    assert P.block_exponent(1.0) == -8          # 448 * 2^-8 = 1.75 >= 1 > 0.875
    assert P.block_exponent(1.75) == -8
    assert P.block_exponent(1.7500001) == -7
    assert P.block_exponent(1e-45) == -127      # clamped


@pytest.mark.parametrize("block_rows", [1, 128])
def test_quantisation_error_and_block_maximum(block_rows):
    rng = np.random.default_rng(block_rows)
    R, C = 130, 256
    x = rng.standard_normal((R, C)) * np.exp2(rng.integers(-20, 20, size=(R, 1)))
    bits = P.f64_to_bf16(x)
    xv = P.bf16_to_f64(bits)
    codes, exps = P.quant_blockscale(bits, block_rows)
    deq = P.dequant(codes, exps, block_rows)
    nbr = exps.shape[0]
    for bi in range(nbr):
        r0, r1 = bi * block_rows, min(R, (bi + 1) * block_rows)
        for bj in range(C // 128):
            blk = xv[r0:r1, 128 * bj:128 * (bj + 1)]
            s = 2.0 ** exps[bi, bj]
            v = blk / s
            assert np.abs(v).max() <= 448.0 and np.abs(v).max() > 224.0  # the smallest scale that fits
            # error at most half the e4m3 spacing of each value (2^-4 relative, 2^-10 absolute below 2^-6)
            d = np.abs(deq[r0:r1, 128 * bj:128 * (bj + 1)] / s - v)
            assert (d <= np.maximum(np.abs(v) * 2.0 ** -4, 2.0 ** -10) + 1e-300).all()


def test_zero_block_and_signed_zero():
    bits = np.zeros((1, 128), dtype=np.uint16)
    bits[0, 3] = 0x8000  # -0.0
    codes, exps = P.quant_blockscale(bits, 1)
    assert exps[0, 0] == 0 and codes[0, 3] == 0x80 and (np.delete(codes[0], 3) == 0).all()


def test_gemm_against_brute_force_sums():
    rng = np.random.default_rng(3)
    M, N, K = 5, 128, 256
    xb = P.f64_to_bf16(rng.standard_normal((M, K)))
    wb = P.f64_to_bf16(rng.standard_normal((N, K)) * 0.1)
    xc, xe = P.quant_blockscale(xb, 1)
    wc, we = P.quant_blockscale(wb, 128)
    y = P.proj_gemm(xc, xe, wc, we)
    for m in range(M):
        for n in (0, 7, 127):
            s = 0.0
            for k in range(K):
                xv = P.e4m3_decode(xc[m:m + 1, k])[0] * 2.0 ** xe[m, k // 128]
                wv = P.e4m3_decode(wc[n:n + 1, k])[0] * 2.0 ** we[n // 128, k // 128]
                s += xv * wv
            assert y[m, n] == P.f64_to_bf16(np.array([s]))[0]


def test_gemm_exact_on_small_integers():
    """Integer inputs of magnitude <= 15 are exact e4m3 values after a power-of-two scale, and
    every sum stays an integer below 2^8 in bf16's exact range: the product is exact."""
    rng = np.random.default_rng(4)
    M, N, K = 3, 128, 128
    xi = rng.integers(-3, 4, size=(M, K)).astype(np.float64)
    wi = np.zeros((N, K))
    wi[np.arange(N), rng.integers(0, K, size=N)] = rng.integers(-3, 4, size=N)
    xc, xe = P.quant_blockscale(P.f64_to_bf16(xi), 1)
    wc, we = P.quant_blockscale(P.f64_to_bf16(wi), 128)
    y = P.bf16_to_f64(P.proj_gemm(xc, xe, wc, we))
    assert np.array_equal(y, xi @ wi.T)
