"""Pins of the oracle's e4m3 codec against things other than itself.

The encoder/decoder follow the OCP E4M3FN definition (bias 7, 3 mantissa bits, no infinities,
NaN = S.1111.111, max 448). They are checked here against (a) code values printed in the
format definition (tests/golden/e4m3_codes.txt), (b) torch's float8_e4m3fn casts (a library
routine), and (c) a brute-force nearest-value search written independently in this file.
"""
import math
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e4m3_codes.txt")


def _golden():
    rows = []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        code, val = line.split()
        rows.append((int(code, 16), float("nan") if val == "NaN" else float(val)))
    return rows


def test_decode_golden_codes(oracle):
    for code, val in _golden():
        got = oracle.e4m3_value(code)
        if math.isnan(val):
            assert math.isnan(got), hex(code)
        else:
            assert got == val and math.copysign(1.0, got) == math.copysign(1.0, val), hex(code)


def test_decode_all_codes_match_torch(oracle):
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_value(int(c)) for c in codes])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def _finite_table():
    """All finite e4m3 values with their codes (brute-force reference, from the bit fields)."""
    out = []
    for c in range(256):
        s, e, m = c >> 7, (c >> 3) & 15, c & 7
        if e == 15 and m == 7:
            continue
        v = (m / 8.0) * 2.0 ** -6 if e == 0 else (1 + m / 8.0) * 2.0 ** (e - 7)
        out.append((-v if s else v, c))
    return out


_TABLE = _finite_table()


def _brute_force_encode(x: float) -> int:
    """Nearest finite e4m3 value; ties to the code with even mantissa; |x| >= 448 saturates."""
    neg = math.copysign(1.0, x) < 0
    a = abs(x)
    if a >= 448.0:
        return 0xFE if neg else 0x7E
    best = None
    for v, c in _TABLE:
        if v < 0 or (v == 0 and c != 0):
            continue
        d = abs(v - a)
        if best is None or d < best[0] or (d == best[0] and (c & 1) == 0):
            best = (d, c)
    code = best[1]
    return code | 0x80 if neg else code


def test_encode_matches_brute_force(oracle):
    rng = np.random.default_rng(0)
    xs = list(rng.standard_normal(2000).astype(np.float32) * np.float32(60))
    xs += list((rng.standard_normal(500) * 0.01).astype(np.float32))      # subnormal region
    # exact midpoints between neighbouring positive values (ties) and their neighbours
    pos = sorted(v for v, c in _TABLE if v >= 0 and c < 0x80)
    for a, b in zip(pos[:-1], pos[1:]):
        mid = np.float32((a + b) / 2)
        xs += [mid, np.nextafter(mid, np.float32(0)), np.nextafter(mid, np.float32(1000)), -mid]
    xs += [np.float32(0.0), np.float32(-0.0), np.float32(448.0), np.float32(-448.0), np.float32(447.99),
           np.float32(460.0), np.float32(1e30), np.float32(-1e30), np.float32(1e-30), np.float32(-1e-30)]
    for x in xs:
        assert oracle.e4m3_encode(float(x)) == _brute_force_encode(float(x)), float(x)


def test_encode_matches_torch_cast(oracle):
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.uniform(-448, 448, 20000), rng.standard_normal(20000),
                        rng.standard_normal(5000) * 1e-3]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.e4m3_encode_array(x)
    assert np.array_equal(got, ref)


def test_encode_saturates_and_keeps_zero_sign(oracle):
    assert oracle.e4m3_encode(1000.0) == 0x7E
    assert oracle.e4m3_encode(-1000.0) == 0xFE
    assert oracle.e4m3_encode(float("inf")) == 0x7E
    assert oracle.e4m3_encode(-float("inf")) == 0xFE
    assert oracle.e4m3_encode(-0.0) == 0x80
    assert oracle.e4m3_encode(-1e-9) == 0x80
    assert oracle.e4m3_encode(1e-9) == 0x00
    # 2^-10 is the tie between 0 and 2^-9: ties to even -> 0; just above -> 0x01
    assert oracle.e4m3_encode(2.0 ** -10) == 0x00
    assert oracle.e4m3_encode(float(np.nextafter(np.float32(2.0 ** -10), np.float32(1)))) == 0x01


def test_encode_decode_roundtrip_all_finite_codes(oracle):
    for v, c in _TABLE:
        assert oracle.e4m3_encode(v) == c, hex(c)


def test_bf16_rounding_matches_torch(oracle):
    rng = np.random.default_rng(2)
    x = np.concatenate([rng.standard_normal(4000) * 10, rng.standard_normal(1000) * 1e-38]).astype(np.float32)
    # exact ties at the bf16 boundary: low 16 bits = 0x8000 with both parities of the kept part
    ties = (np.arange(1000, dtype=np.uint32) * 0x10000 + 0x3F800000 + 0x8000).view(np.float32)
    x = np.concatenate([x, ties])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.float_to_bf16(float(v)) for v in x], dtype=np.uint16)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("d_nope,d_rope", [(256, 0), (512, 64)])
def test_packed_row_bytes_golden(oracle, d_nope, d_rope):
    path = os.path.join(os.path.dirname(__file__), "golden", "packed_rows.txt")
    rows = [list(map(int, l.split())) for l in open(path) if l.strip() and not l.startswith("#")]
    (row,) = [r for r in rows if r[0] == d_nope and r[1] == d_rope]
    assert oracle.packed_row_bytes(d_nope, d_rope) == row[2] == row[3] + row[4] + row[5]
    assert row[3] == d_nope and row[4] == 4 * (d_nope // 128) and row[5] == 2 * d_rope
