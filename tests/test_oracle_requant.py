"""Pins of the gather/requant oracle (pack of the gathered, bf16-widened rows), from the
arithmetic of the format rather than from the oracle itself:
- every non-zero tile of a packed row holds a +-448 code (the tile maximum divided by
  amax/448 rounds to 448), so its widened maximum is bf16_rne(448 * scale) and the new scale is
  exactly fp32(bf16_rne(448 * scale) / 448);
- widening and rescaling move a value by at most about 2^-8 relative, less than half the e4m3
  spacing at any exponent (2^-4 relative for normal codes, 2^-10 absolute for subnormal ones),
  so every code rounds back to itself; zero tiles stay zero;
- hence requant is idempotent, and RoPE bits pass through."""
import numpy as np
import pytest

import oracle
from dsa_sparse_attention_mla_gb300 import workloads as W


def _bf16_rne(f32):
    u = np.asarray(f32, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return r.astype(np.uint32).view(np.float32)


def _rows(d_nope, d_rope, n=3000, seed=9):
    rng = np.random.default_rng(seed)
    src = W.normal_bf16_bits(seed, 5, 0, n * (d_nope + d_rope)).reshape(n, d_nope + d_rope)
    f = (src.astype(np.uint32) << 16).view(np.float32)
    f = f * (np.float32(2.0) ** rng.integers(-24, 24, size=(n, 1)).astype(np.float32))  # wide magnitudes
    f[::97, :128] = 0.0                           # some all-zero tiles
    f[1::53, : d_nope] *= np.float32(2.0 ** -12)  # tiles whose small values land on subnormal codes
    return (f.view(np.uint32) >> 16).astype(np.uint16)


@pytest.mark.parametrize("d_nope,d_rope", [(256, 0), (512, 64)])
def test_requant_keeps_codes_and_rope_and_rescales_in_closed_form(d_nope, d_rope):
    src = _rows(d_nope, d_rope)
    n = src.shape[0]
    cache = oracle.quant_k_cache(src[:, :d_nope], src[:, d_nope:] if d_rope else None)
    out, bad = oracle.gather_requant(cache, d_nope, d_rope, np.arange(n, dtype=np.int32))
    assert bad == 0
    np.testing.assert_array_equal(out[:, :d_nope], cache[:, :d_nope])
    tiles = d_nope // 128
    sc = cache[:, d_nope:d_nope + 4 * tiles].copy().view(np.float32)
    sc2 = out[:, d_nope:d_nope + 4 * tiles].copy().view(np.float32)
    np.testing.assert_array_equal(sc2, (_bf16_rne(np.float32(448) * sc) / np.float32(448)).astype(np.float32))
    assert (sc2[sc == 0] == 0).all()
    np.testing.assert_array_equal(out[:, d_nope + 4 * tiles:], cache[:, d_nope + 4 * tiles:])


@pytest.mark.parametrize("d_nope,d_rope", [(256, 0), (512, 64)])
def test_requant_is_idempotent(d_nope, d_rope):
    src = _rows(d_nope, d_rope, n=1000, seed=11)
    cache = oracle.quant_k_cache(src[:, :d_nope], src[:, d_nope:] if d_rope else None)
    idx = np.arange(cache.shape[0], dtype=np.int32)
    once, _ = oracle.gather_requant(cache, d_nope, d_rope, idx)
    twice, _ = oracle.gather_requant(once, d_nope, d_rope, idx)
    np.testing.assert_array_equal(twice, once)


def test_requant_masked_out_of_range_paged_and_scatter():
    d_nope, d_rope = 512, 64
    src = _rows(d_nope, d_rope, n=256, seed=13)
    cache = oracle.quant_k_cache(src[:, :d_nope], src[:, d_nope:])
    rb = cache.shape[1]
    # masked (-1, -5) and out-of-range (300) entries pack the zero row; the latter are counted
    idx = np.array([3, -1, 300, 7, -5, 255], dtype=np.int32)
    out, bad = oracle.gather_requant(cache, d_nope, d_rope, idx)
    assert bad == 1
    assert not out[[1, 2, 4]].any()
    direct, _ = oracle.gather_requant(cache, d_nope, d_rope, np.array([3, 7, 255], dtype=np.int32))
    np.testing.assert_array_equal(out[[0, 3, 5]], direct)
    # paged: logical position p of request r is slot bt[r, p // 16] * 16 + p % 16
    bt = np.array([[15, 0, 3], [2, 9, 1]], dtype=np.int32)
    pos = np.array([0, 17, 40, 5], dtype=np.int32)
    req = np.array([0, 0, 1, 1], dtype=np.int32)
    paged, bad = oracle.gather_requant(cache, d_nope, d_rope, pos, block_table=bt, page_size=16, req_of_index=req)
    assert bad == 0
    slots = bt[req, pos // 16] * 16 + pos % 16
    np.testing.assert_array_equal(paged, oracle.gather_requant(cache, d_nope, d_rope, slots.astype(np.int32))[0])
    # out_loc scatters result i to row out_loc[i]; untouched rows stay as they were
    loc = np.array([5, 0, 2], dtype=np.int64)
    base = np.full((6, rb), 0xAB, dtype=np.uint8)
    scat, _ = oracle.gather_requant(cache, d_nope, d_rope, np.array([3, 7, 255], dtype=np.int32), out_loc=loc,
                                    out=base.copy())
    np.testing.assert_array_equal(scat[loc], direct)
    np.testing.assert_array_equal(scat[[1, 3, 4]], base[[1, 3, 4]])
