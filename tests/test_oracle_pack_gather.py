"""Pins of the oracle's quant_k_cache (pack) and gather/dequant against closed forms, library
routines (torch float8/bf16 casts) and brute force.

Row layout (sglang PR #38547, Contract table "scaled FP8 cache row"): codes, then one fp32
scale per 128-element tile (little endian), then the RoPE tail as raw bf16.
"""
import numpy as np
import pytest
import torch

from dsa_sparse_attention_mla_gb300 import workloads as W


def _bf16_bits(x):
    return torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _bits_to_f32(b):
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).float().numpy()


def _scales(row, d_nope):
    return np.frombuffer(row[d_nope: d_nope + 4 * (d_nope // 128)].tobytes(), dtype="<f4")


def test_single_nonzero_element_tile(oracle):
    x = np.zeros((2, 256), dtype=np.float32)
    x[0, 5] = 3.25
    x[0, 200] = -0.0078125
    x[1, 130] = -7.5
    cache = oracle.quant_k_cache(_bf16_bits(x))
    assert cache.shape == (2, 264)
    s0 = _scales(cache[0], 256)
    assert s0[0] == np.float32(3.25) / np.float32(448)
    assert s0[1] == np.float32(0.0078125) / np.float32(448)
    assert cache[0, 5] == 0x7E and cache[0, 200] == 0xFE
    assert np.count_nonzero(cache[0, :256]) == 2
    s1 = _scales(cache[1], 256)
    assert s1[0] == 0.0 and s1[1] == np.float32(7.5) / np.float32(448)
    assert cache[1, 130] == 0xFE and np.count_nonzero(cache[1, :256]) == 1


def test_constant_and_zero_tiles(oracle):
    x = np.zeros((3, 256), dtype=np.float32)
    x[0, :128] = 1.5
    x[1, 128:] = -2.0
    cache = oracle.quant_k_cache(_bf16_bits(x))
    assert (cache[0, :128] == 0x7E).all() and (cache[0, 128:256] == 0).all()
    assert (cache[1, 128:256] == 0xFE).all()
    assert (_scales(cache[2], 256) == 0).all() and (cache[2, :256] == 0).all()


@pytest.mark.parametrize("d_nope,d_rope", [(256, 0), (512, 64)])
def test_codes_match_torch_cast_and_layout(oracle, d_nope, d_rope):
    rows = W.NormalRows(7, 1, 300, d_nope + d_rope).bits()
    rows[3, :] = 0
    rows[4, 10] = 0x8000                     # -0.0 in a row
    nope, rope = rows[:, :d_nope], rows[:, d_nope:]
    cache = oracle.quant_k_cache(nope, rope if d_rope else None)
    rb = d_nope + 4 * (d_nope // 128) + 2 * d_rope
    assert cache.shape == (300, rb)
    x = _bits_to_f32(nope).reshape(300, d_nope // 128, 128)
    amax = np.abs(x).max(axis=2)
    scale = (torch.from_numpy(amax) / torch.tensor(448.0, dtype=torch.float32)).numpy()
    got_scale = np.stack([_scales(cache[i], d_nope) for i in range(300)])
    assert np.array_equal(got_scale.view(np.uint32), np.where(amax == 0, 0, scale).astype(np.float32).view(np.uint32))
    q = torch.from_numpy(x) / torch.from_numpy(np.where(amax == 0, 1, scale))[:, :, None]
    ref_codes = q.to(torch.float8_e4m3fn).view(torch.uint8).numpy().reshape(300, d_nope)
    ref_codes[amax.repeat(128, axis=1).reshape(300, d_nope) == 0] = 0
    assert np.array_equal(cache[:, :d_nope], ref_codes)
    if d_rope:
        tail = cache[:, d_nope + 4 * (d_nope // 128):].copy().view("<u2")
        assert np.array_equal(tail, rope)


def test_round_trip_error_bound(oracle):
    rows = W.NormalRows(3, 2, 500, 256).bits()
    cache = oracle.quant_k_cache(rows)
    x = _bits_to_f32(rows).astype(np.float64)
    codes = torch.from_numpy(cache[:, :256].copy()).view(torch.float8_e4m3fn).double().numpy()
    sc = np.stack([_scales(cache[i], 256) for i in range(500)]).astype(np.float64)
    xh = codes * np.repeat(sc, 128, axis=1)
    # e4m3 normals: half-ulp relative error 2^-4; subnormals: half-step 2^-10 in code units;
    # plus the fp32 rounding of x/scale (relative 2^-24 of the quotient)
    bound = 2.0 ** -4 * np.abs(x) + 2.0 ** -10 * np.repeat(sc, 128, axis=1) + 2.0 ** -20 * np.abs(x)
    assert (np.abs(xh - x) <= bound).all()


def test_pack_idempotent_on_dequantised_rows(oracle):
    rows = W.NormalRows(4, 3, 400, 256).bits()
    cache = oracle.quant_k_cache(rows)
    # dequantise in fp32 and round to bf16 (the gather/dequant helper), then pack again
    deq, bad = oracle.gather_dequant(cache, oracle.CACHE_FP8_SCALED, 256, 0, np.arange(400, dtype=np.int32))
    assert bad == 0
    cache2 = oracle.quant_k_cache(deq)
    same = (cache2[:, :256] == cache[:, :256]).mean()
    assert same > 0.999, same


def test_out_loc_scatter(oracle):
    rows = W.NormalRows(5, 4, 64, 256).bits()
    loc = np.random.default_rng(0).permutation(128)[:64].astype(np.int64)
    cache = oracle.quant_k_cache(rows, out_loc=loc, num_slots=128)
    direct = oracle.quant_k_cache(rows)
    assert np.array_equal(cache[loc], direct)
    untouched = np.setdiff1d(np.arange(128), loc)
    assert (cache[untouched] == 0).all()
    with pytest.raises(ValueError):
        oracle.quant_k_cache(rows, out_loc=np.full(64, 128, dtype=np.int64), num_slots=128)


def test_gather_dequant_fp8_matches_torch(oracle):
    rows = W.NormalRows(6, 5, 200, 576).bits()
    cache = oracle.quant_k_cache(rows[:, :512], rows[:, 512:])
    idx = np.array([5, -1, 199, 0, 5, 77, -7], dtype=np.int32)
    out, bad = oracle.gather_dequant(cache, oracle.CACHE_FP8_SCALED, 512, 64, idx)
    assert bad == 0 and out.shape == (7, 576)
    for i, j in enumerate(idx):
        if j < 0:
            assert (out[i] == 0).all()
            continue
        codes = torch.from_numpy(cache[j, :512].copy()).view(torch.float8_e4m3fn).float()
        sc = torch.from_numpy(_scales(cache[j], 512).copy()).repeat_interleave(128)
        ref = (codes * sc).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(out[i, :512], ref)
        assert np.array_equal(out[i, 512:], rows[j, 512:])


def test_gather_bf16_and_paged_translation(oracle):
    slots, ps = 512, 64
    kv = W.NormalRows(8, 6, slots, 256).bits()
    rng = np.random.default_rng(3)
    bt = rng.permutation(slots // ps).astype(np.int32).reshape(2, 4)     # 2 requests x 4 pages
    pos = rng.integers(0, 4 * ps, size=50).astype(np.int32)
    req = rng.integers(0, 2, size=50).astype(np.int32)
    pos[7] = -1
    out, bad = oracle.gather_dequant(kv, oracle.CACHE_BF16, 256, 0, pos, block_table=bt, page_size=ps,
                                     req_of_index=req)
    assert bad == 0
    for i in range(50):
        if pos[i] < 0:
            assert (out[i] == 0).all()
        else:
            slot = bt[req[i], pos[i] // ps] * ps + pos[i] % ps
            assert np.array_equal(out[i], kv[slot])
    # identity page table == direct mode
    ident = np.arange(slots // ps, dtype=np.int32)[None, :]
    idx = rng.integers(0, slots, size=40).astype(np.int32)
    a, _ = oracle.gather_dequant(kv, 0, 256, 0, idx, block_table=ident, page_size=ps)
    b, _ = oracle.gather_dequant(kv, 0, 256, 0, idx)
    assert np.array_equal(a, b)
    # repeated-page table: every logical page maps to physical page 3
    rep = np.full((1, 4), 3, dtype=np.int32)
    c, _ = oracle.gather_dequant(kv, 0, 256, 0, np.arange(4 * ps, dtype=np.int32), block_table=rep, page_size=ps)
    assert np.array_equal(c, np.tile(kv[3 * ps: 4 * ps], (4, 1)))
    # out-of-range entries are masked and counted
    _, bad = oracle.gather_dequant(kv, 0, 256, 0, np.array([0, slots, 10**6], dtype=np.int32))
    assert bad == 2
    _, bad = oracle.gather_dequant(kv, 0, 256, 0, np.array([4 * ps, 3], dtype=np.int32), block_table=bt,
                                   page_size=ps)
    assert bad == 1
