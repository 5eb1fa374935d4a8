"""GPU parity of the packed-cache kernels against the oracle: dsa_quant_k_cache must be
bit-exact (e4m3 RNE codes, fp32 amax/448 scales, RoPE bytes), and dsa_gather_dequant must
be bit-exact (bf16_rne(fp32(code) * scale)), in direct and paged modes, for the 264-byte
(256+0) and 656-byte (512+64) rows (sglang PR #38547, Contract table and Scope list)."""
import numpy as np
import pytest
import torch

import oracle
import dsa_sparse_attention_mla_gb300 as dsa
from dsa_sparse_attention_mla_gb300 import workloads as W

from _helpers import bf16_dev, bits_of

pytestmark = pytest.mark.gpu


def _special_rows(n, D, seed):
    rows = W.NormalRows(seed, 1, n, D).bits().copy()
    rows[0] = 0                                       # all-zero tiles -> scale 0
    rows[1, :] = 0x8000                               # all -0.0
    rows[2, 5] = 0x7F7F                               # a huge value in one tile
    rows[3, :128] = 0x3F80                            # constant tile
    x = torch.from_numpy(rows[4].view(np.int16)).view(torch.bfloat16).float() * 1e-30
    rows[4] = x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)   # tiny values (subnormal codes)
    return rows


@pytest.mark.parametrize("d_nope,d_rope", [(256, 0), (512, 64)])
def test_quant_bit_exact(gpu, d_nope, d_rope):
    n = 5000
    rows = _special_rows(n, d_nope + d_rope, 3)
    ref = oracle.quant_k_cache(rows[:, :d_nope], rows[:, d_nope:] if d_rope else None)
    kn = bf16_dev(rows[:, :d_nope], gpu)
    kr = bf16_dev(rows[:, d_nope:], gpu) if d_rope else None
    got = dsa.dsa_quant_k_cache(kn, kr).cpu().numpy()
    assert got.shape == ref.shape
    bad = np.argwhere(got != ref)
    assert bad.size == 0, f"{len(bad)} bytes differ, first at {bad[:5].tolist()}"


def test_quant_out_loc_strided_and_errors(gpu):
    n, slots = 700, 2048
    rows = W.NormalRows(5, 2, n, 300).bits()          # 300-wide source: rows strided, use [:, :256]
    loc = np.random.default_rng(0).permutation(slots)[:n].astype(np.int64)
    ref = oracle.quant_k_cache(rows[:, :256], out_loc=loc, num_slots=slots)
    src = bf16_dev(rows, gpu)[:, :256]
    cache = torch.zeros((slots, 264), dtype=torch.uint8, device=gpu)
    err = torch.zeros(1, dtype=torch.int32, device=gpu)
    dsa.dsa_quant_k_cache(src, out_loc=torch.from_numpy(loc).to(gpu), cache=cache, error_word=err)
    assert np.array_equal(cache.cpu().numpy(), ref)
    assert err.item() == 0
    bad_loc = torch.full((n,), slots, dtype=torch.int64, device=gpu)
    dsa.dsa_quant_k_cache(src, out_loc=bad_loc, cache=cache, error_word=err)
    assert err.item() & dsa.DEVERR_SLOT_OUT_OF_RANGE
    assert np.array_equal(cache.cpu().numpy(), ref)


def test_quant_every_e4m3_decision(gpu):
    """Rows whose quotients x/scale sweep every e4m3 rounding boundary: tiles of 128 values
    with amax fixed at 448 * 2^k so that x / scale hits exact midpoints and the bf16 values one
    bf16 step either side of each (the nearest inputs that do not tie), both signs."""
    def bf16_step(v, d):  # the bf16 value d steps of the bf16 grid away from v (v is on the grid)
        b = int(np.array([v], dtype=np.float32).view(np.uint32)[0]) >> 16
        return float(np.array([(b + d) << 16], dtype=np.uint32).view(np.float32)[0])

    vals = []
    pos = sorted(set(abs(oracle.e4m3_value(c)) for c in range(0x7F)))
    for a, b in zip(pos[:-1], pos[1:]):
        mid = (a + b) / 2
        assert bf16_step(mid, 0) == mid  # every e4m3 midpoint is a bf16 value
        below, above = bf16_step(mid, -1), bf16_step(mid, 1)
        assert a < below < mid < above < b
        vals += [mid, below, above, -mid, -below, -above, a, -b]
    vals = np.array(vals, dtype=np.float32)
    vals = vals[np.abs(vals) < 448]
    per = 127
    n = (len(vals) + per - 1) // per
    x = np.zeros((n, 256), dtype=np.float32)
    for i in range(n):
        chunk = vals[i * per: (i + 1) * per]
        x[i, : len(chunk)] = chunk
        x[i, 127] = 448.0                              # amax = 448 -> scale exactly 1
        x[i, 128:] = x[i, :128] * 2.0 ** -20           # same pattern, scale 2^-20
    bits = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    ref = oracle.quant_k_cache(bits)
    got = dsa.dsa_quant_k_cache(bf16_dev(bits, gpu)).cpu().numpy()
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("kind,d_nope,d_rope", [(1, 256, 0), (1, 512, 64), (0, 256, 0), (0, 512, 64)])
def test_gather_dequant_bit_exact(gpu, kind, d_nope, d_rope):
    slots = 3000
    D = d_nope + d_rope
    rows = _special_rows(slots, D, 7)
    cache = rows if kind == 0 else oracle.quant_k_cache(rows[:, :d_nope], rows[:, d_nope:] if d_rope else None)
    rng = np.random.default_rng(1)
    idx = rng.integers(-2, slots, size=4000).astype(np.int32)
    ref, bad = oracle.gather_dequant(cache, kind, d_nope, d_rope, idx)
    assert bad == 0
    dcache = bf16_dev(cache, gpu) if kind == 0 else torch.from_numpy(cache).to(gpu)
    got = dsa.dsa_gather_dequant(dcache, kind, d_nope, d_rope, torch.from_numpy(idx).to(gpu))
    assert np.array_equal(bits_of(got), ref)


def test_gather_dequant_paged_repeated_pages_and_errors(gpu):
    ps, pages = 64, 40
    slots = ps * pages
    rows = W.NormalRows(9, 3, slots, 256).bits()
    cache = oracle.quant_k_cache(rows)
    rng = np.random.default_rng(2)
    bt = rng.integers(0, pages, size=(3, 12)).astype(np.int32)       # repeated physical pages
    bt[1, :] = 7                                                      # every logical page -> page 7
    idx = rng.integers(-1, 12 * ps, size=3000).astype(np.int32)
    req = rng.integers(0, 3, size=3000).astype(np.int32)
    ref, bad = oracle.gather_dequant(cache, 1, 256, 0, idx, block_table=bt, page_size=ps, req_of_index=req)
    assert bad == 0
    dcache = torch.from_numpy(cache).to(gpu)
    got = dsa.dsa_gather_dequant(dcache, 1, 256, 0, torch.from_numpy(idx).to(gpu),
                                 block_table=torch.from_numpy(bt).to(gpu), page_size=ps,
                                 req_of_index=torch.from_numpy(req).to(gpu))
    assert np.array_equal(bits_of(got), ref)
    # out-of-range logical positions / slots: zero rows and the error bit
    err = torch.zeros(1, dtype=torch.int32, device=gpu)
    oob = torch.tensor([12 * ps, 3, 10 ** 6], dtype=torch.int32, device=gpu)
    got = dsa.dsa_gather_dequant(dcache, 1, 256, 0, oob, block_table=torch.from_numpy(bt).to(gpu), page_size=ps,
                                 error_word=err)
    assert err.item() & dsa.DEVERR_INDEX_OUT_OF_RANGE
    g = bits_of(got)
    assert (g[0] == 0).all() and (g[2] == 0).all() and (g[1] != 0).any()


def test_pack_then_gather_round_trip_on_gpu_matches_oracle(gpu):
    """GPU pack followed by GPU gather equals the oracle's pack + gather (256+0 and 512+64)."""
    for d_nope, d_rope in [(256, 0), (512, 64)]:
        rows = W.NormalRows(11, 4, 1000, d_nope + d_rope).bits()
        ref_cache = oracle.quant_k_cache(rows[:, :d_nope], rows[:, d_nope:] if d_rope else None)
        idx = np.arange(999, -1, -1, dtype=np.int32)
        ref, _ = oracle.gather_dequant(ref_cache, 1, d_nope, d_rope, idx)
        c = dsa.dsa_quant_k_cache(bf16_dev(rows[:, :d_nope], gpu), bf16_dev(rows[:, d_nope:], gpu) if d_rope else None)
        got = dsa.dsa_gather_dequant(c, 1, d_nope, d_rope, torch.from_numpy(idx).to(gpu))
        assert np.array_equal(bits_of(got), ref)


# ------------------------------------------------------------------------- gather / requant --
@pytest.mark.parametrize("d_nope,d_rope", [(256, 0), (512, 64)])
def test_gather_requant_bit_exact(gpu, d_nope, d_rope):
    """dsa_gather_requant == the oracle's pack of its gathered bf16 rows, byte for byte; masked
    entries pack the zero row (special rows: zero, -0, huge, constant and tiny tiles)."""
    n = 3000
    rows = _special_rows(n, d_nope + d_rope, seed=21)
    cache = oracle.quant_k_cache(rows[:, :d_nope], rows[:, d_nope:] if d_rope else None)
    rng = np.random.default_rng(4)
    idx = rng.integers(-2, n, size=4097).astype(np.int32)
    idx[:5] = [0, 1, 2, 3, 4]
    ref, bad = oracle.gather_requant(cache, d_nope, d_rope, idx)
    assert bad == 0
    got = dsa.dsa_gather_requant(torch.from_numpy(cache).to(gpu), d_nope, d_rope,
                                 torch.from_numpy(idx).to(gpu)).cpu().numpy()
    diff = np.argwhere(got != ref)
    assert diff.size == 0, (len(diff), diff[:4].tolist(), got[tuple(diff[0])], ref[tuple(diff[0])],
                            cache[idx[diff[0][0]], d_nope:d_nope + 4 * (d_nope // 128)].view(np.float32).tolist())


def test_gather_requant_paged_scatter_and_errors(gpu):
    d_nope, d_rope, ps, pages = 512, 64, 64, 30
    slots = ps * pages
    rows = W.NormalRows(23, 2, slots, d_nope + d_rope).bits()
    cache = oracle.quant_k_cache(rows[:, :d_nope], rows[:, d_nope:])
    rng = np.random.default_rng(6)
    bt = rng.integers(0, pages, size=(2, 10)).astype(np.int32)
    idx = rng.integers(-1, 10 * ps, size=900).astype(np.int32)
    idx[7] = 10 * ps + 3                                             # past the request's pages
    req = rng.integers(0, 2, size=900).astype(np.int32)
    out_slots = 1200
    loc = rng.permutation(out_slots)[:900].astype(np.int64)
    base = np.full((out_slots, cache.shape[1]), 0x5A, dtype=np.uint8)
    ref, bad = oracle.gather_requant(cache, d_nope, d_rope, idx, block_table=bt, page_size=ps, req_of_index=req,
                                     out_loc=loc, out=base.copy())
    assert bad == 1
    err = torch.zeros(1, dtype=torch.int32, device=gpu)
    out = torch.from_numpy(base.copy()).to(gpu)
    dsa.dsa_gather_requant(torch.from_numpy(cache).to(gpu), d_nope, d_rope, torch.from_numpy(idx).to(gpu),
                           block_table=torch.from_numpy(bt).to(gpu), page_size=ps,
                           req_of_index=torch.from_numpy(req).to(gpu), out_loc=torch.from_numpy(loc).to(gpu),
                           out=out, error_word=err)
    assert np.array_equal(out.cpu().numpy(), ref)
    assert err.item() & dsa.DEVERR_INDEX_OUT_OF_RANGE
    # a destination row outside the output is skipped and flagged
    err.zero_()
    bad_loc = torch.tensor([0, out_slots], dtype=torch.int64, device=gpu)
    dsa.dsa_gather_requant(torch.from_numpy(cache).to(gpu), d_nope, d_rope,
                           torch.tensor([1, 2], dtype=torch.int32, device=gpu), block_table=None,
                           out_loc=bad_loc, out=out, error_word=err)
    torch.cuda.synchronize()
    assert err.item() & dsa.DEVERR_SLOT_OUT_OF_RANGE


@pytest.mark.parametrize("d_nope,d_rope", [(256, 0), (512, 64)])
def test_gather_requant_non_canonical_rows_bit_exact(gpu, d_nope, d_rope):
    """Rows the pack would never write (arbitrary codes without a 448 maximum, zero, negative,
    huge and tiny scales) take the general widen-and-pack path: still the oracle's bytes."""
    rng = np.random.default_rng(8)
    n = 2000
    rb = dsa.dsa_packed_row_bytes(d_nope, d_rope)
    tiles = d_nope // 128
    cache = rng.integers(0, 256, size=(n, rb), dtype=np.uint8)
    codes = cache[:, :d_nope]
    codes[(codes & 0x7F) == 0x7F] = 0x11                          # no NaN codes (out of contract)
    codes[: n // 2] &= 0xBD                                       # half the rows: no 0x7E maximum
    # scales across the whole range where 448 * scale stays finite in bf16 (wider ones give
    # inf and NaN codes: outside the format), denormal ones included
    sc = np.exp2(rng.uniform(-140, 118.5, size=(n, tiles))).astype(np.float32)
    sc *= rng.choice(np.array([1, -1], dtype=np.float32), size=(n, tiles))
    sc[::7, 0] = 0.0
    cache[:, d_nope:d_nope + 4 * tiles] = sc.view(np.uint8).reshape(n, 4 * tiles)
    idx = rng.permutation(n).astype(np.int32)
    ref, bad = oracle.gather_requant(cache, d_nope, d_rope, idx)
    assert bad == 0
    got = dsa.dsa_gather_requant(torch.from_numpy(cache).to(gpu), d_nope, d_rope,
                                 torch.from_numpy(idx).to(gpu)).cpu().numpy()
    diff = np.argwhere(got != ref)
    assert diff.size == 0, (len(diff), diff[:4].tolist(), got[tuple(diff[0])], ref[tuple(diff[0])],
                            cache[idx[diff[0][0]], d_nope:d_nope + 4 * (d_nope // 128)].view(np.float32).tolist())
