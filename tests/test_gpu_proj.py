"""GPU FP8 block-scaled projection (dsa_quant_fp8_blockscale, dsa_proj_gemm) against the oracle:
codes and scales bit for bit, the scales checked in the documented block-scale layout, and the
product within the rounding of an fp32-accumulated, bf16-rounded result."""
import numpy as np
import pytest
import torch

import dsa_sparse_attention_mla_gb300 as dsa
from oracle import projection as P

pytestmark = pytest.mark.gpu


def _bf16(bits, device):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def _matrix(rng, R, C, spread=20):
    """bf16 bits with row (and block) magnitudes 2^-spread .. 2^spread, an all-zero block, -0.0."""
    x = rng.standard_normal((R, C)) * np.exp2(rng.integers(-spread, spread + 1, size=(R, 1)))
    if C >= 256:
        x[:, 128:256] *= np.exp2(rng.integers(-spread, spread + 1))
    if R > 2:
        x[1, :128] = 0.0
        x[2, 5] = -0.0
    return P.f64_to_bf16(x)


def _layout_bytes(exps, R, C, block_rows):
    """The scale tensor the header documents: 512-byte tiles of 128 rows x 4 scale columns,
    row-tile major; row r, 32-element scale column c at (r % 32) * 16 + ((r % 128) / 32) * 4 + c % 4;
    each 128-column block four equal scales; rows past R read 127."""
    nrt, nct = (R + 127) // 128, C // 128
    out = np.full(nrt * nct * 512, 127, dtype=np.uint8)
    for r in range(nrt * 128):
        for j in range(nct):
            if block_rows == 1:
                if r >= R:
                    continue
                e = exps[r, j]
            else:
                e = exps[r // 128, j]
            base = ((r // 128) * nct + j) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4
            out[base:base + 4] = e + 127
    return out


@pytest.mark.parametrize("block_rows", [1, 128])
@pytest.mark.parametrize("R,C", [(1, 128), (37, 384), (130, 256), (256, 128)])
def test_quant_bit_exact(gpu, block_rows, R, C):
    rng = np.random.default_rng(R * 7 + C + block_rows)
    bits = _matrix(rng, R, C)
    codes, scales = dsa.dsa_quant_fp8_blockscale(_bf16(bits, gpu), block_rows)
    torch.cuda.synchronize()
    rc, re = P.quant_blockscale(bits, block_rows)
    assert np.array_equal(codes.cpu().numpy(), rc)
    assert np.array_equal(scales.cpu().numpy(), _layout_bytes(re, R, C, block_rows))


def test_quant_strided_rows_and_tiny_huge_blocks(gpu):
    rng = np.random.default_rng(9)
    R, C = 40, 256
    x = rng.standard_normal((R, C))
    x[0] *= 2.0 ** -130   # subnormal-range block: exponent clamps at -127
    x[1] *= 2.0 ** 120    # near the bf16 top
    bits = P.f64_to_bf16(x)
    wide = np.zeros((R, C + 64), dtype=np.uint16)
    wide[:, :C] = bits
    xt = _bf16(wide, gpu)[:, :C]
    codes, scales = dsa.dsa_quant_fp8_blockscale(xt, 1)
    torch.cuda.synchronize()
    rc, re = P.quant_blockscale(bits, 1)
    assert re[0, 0] == -127
    assert np.array_equal(codes.cpu().numpy(), rc)
    assert np.array_equal(scales.cpu().numpy(), _layout_bytes(re, R, C, 1))


def _gemm_case(gpu, M, N, K, seed):
    rng = np.random.default_rng(seed)
    xb = _matrix(rng, M, K, spread=6)
    wb = P.f64_to_bf16(rng.standard_normal((N, K)) * np.exp2(rng.integers(-4, 5, size=(N // 128, 1)).repeat(128, 0)))
    xc, xs = dsa.dsa_quant_fp8_blockscale(_bf16(xb, gpu), 1)
    wc, ws = dsa.dsa_quant_fp8_blockscale(_bf16(wb, gpu), 128)
    y = dsa.dsa_proj_gemm(xc, xs, wc, ws)
    torch.cuda.synchronize()
    rxc, rxe = P.quant_blockscale(xb, 1)
    rwc, rwe = P.quant_blockscale(wb, 128)
    ref_bits = P.proj_gemm(rxc, rxe, rwc, rwe)
    got = y.float().cpu().numpy()
    ref = P.bf16_to_f64(ref_bits)
    # fp32 accumulation in some order, then one bf16 rounding: within two bf16 steps of the
    # exactly rounded value, plus the accumulation error bound K * 2^-24 * sum |x w|
    mag = np.abs(P.dequant(rxc, rxe, 1)) @ np.abs(P.dequant(rwc, rwe, 128)).T
    tol = 2.0 ** -7 * np.abs(ref) + K * 2.0 ** -24 * mag + 1e-30
    bad = np.abs(got - ref) > tol
    assert not bad.any(), (np.argwhere(bad)[:5], got[bad][:5], ref[bad][:5])
    return got, ref


@pytest.mark.parametrize("M,N,K", [(1, 128, 128), (37, 256, 384), (256, 384, 512), (300, 128, 1024)])
def test_gemm_against_oracle(gpu, M, N, K):
    _gemm_case(gpu, M, N, K, seed=M + N + K)


def test_gemm_exact_on_small_integers(gpu):
    """Small integer operands are exact after their power-of-two scales and every sum is an
    integer below 2^8: the bf16 result is the exact product."""
    rng = np.random.default_rng(12)
    M, N, K = 64, 256, 256
    xi = rng.integers(-3, 4, size=(M, K)).astype(np.float64)
    wi = np.zeros((N, K))
    for n in range(N):
        wi[n, rng.choice(K, size=4, replace=False)] = rng.integers(-3, 4, size=4)
    xc, xs = dsa.dsa_quant_fp8_blockscale(_bf16(P.f64_to_bf16(xi), gpu), 1)
    wc, ws = dsa.dsa_quant_fp8_blockscale(_bf16(P.f64_to_bf16(wi), gpu), 128)
    y = dsa.dsa_proj_gemm(xc, xs, wc, ws)
    torch.cuda.synchronize()
    assert np.array_equal(y.float().cpu().numpy(), xi @ wi.T)
