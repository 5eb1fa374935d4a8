"""GPU parity of dsa_sparse_attn against the fp64 oracle (step-by-step gather, mask, score,
softmax and weighted sum), over the geometry coverage of sglang PR #38547 (Direct GLM geometry coverage list):
Q [tokens, 64, 256] with token counts 1, 8, 17; top-k widths 2048 and 2112; fully valid rows and
2051 valid entries padded with -1 to 2112; BF16 and packed-FP8 caches; direct and paged slots;
the 512+64 control; bit-identical repeated execution; and edge cases (masked tokens, a single
valid entry, duplicate and repeated-page entries, out-of-range indices)."""
import numpy as np
import pytest
import torch

import dsa_sparse_attention_mla_gb300 as dsa
from dsa_sparse_attention_mla_gb300 import workloads as W

from _helpers import (MAX_ABS, MAX_ABS_ORDER_ONE, bf16_dev, check_close, f32_of, oracle_cache, run_oracle,
                      run_oracle_on_dequantised, token_gates)

pytestmark = pytest.mark.gpu


def _dev_inputs(wl, cache, device):
    q = bf16_dev(wl.q_bits(), device)
    dcache = bf16_dev(cache, device) if wl.kind == 0 else torch.from_numpy(cache).to(device)
    idx = torch.from_numpy(wl.indices).to(device)
    bt = None if wl.block_table is None else torch.from_numpy(wl.block_table).to(device)
    req = None if wl.req_of_token is None else torch.from_numpy(wl.req_of_token).to(device)
    return q, dcache, idx, bt, req


def _gpu_attn(wl, cache, device, lse=False, err=None, **kw):
    q, dcache, idx, bt, req = _dev_inputs(wl, cache, device)
    lse_t = torch.empty((wl.T, wl.H), dtype=torch.float32, device=device) if lse else None
    out = dsa.dsa_sparse_attn(q, dcache, wl.kind, idx, wl.sm_scale, d_nope=wl.d_nope, d_rope=wl.d_rope, d_v=wl.d_v,
                              block_table=bt, page_size=wl.page_size, req_of_token=req, lse=lse_t, error_word=err, **kw)
    torch.cuda.synchronize()
    return out, lse_t


def _check_lse(got, ref, atol):
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(got), fin)
    np.testing.assert_allclose(got[fin], ref[fin], rtol=1e-5, atol=atol)


def _check(wl, device, tokens=None, lse=True, max_abs=MAX_ABS):
    """Output and LSE against the oracle.

    BF16 cache: the oracle sees exactly the kernel's inputs (fp32 accumulation is the only
    difference; LSE within 2e-4). FP8 cache: the kernel never rounds a dequantised value; it
    multiplies the exact e4m3 codes and applies each row's fp32 tile scales to its score
    accumulators and to the probabilities, so the reference is the oracle's exact dequantisation
    (code * scale in fp64), to the same tolerances as BF16. Where the scores are of order one
    (sm_scale <= 1/sqrt(D), the regime of the named workloads) the output is also checked
    against the oracle over the bf16-rounded rows of the gather/dequant helper, with the LSE
    bound that follows from that rounding: |ds| <= sm_scale * 2^-9 * sum_d |q_d k_d|, at most
    about 2e-2 for unit-variance rows of width 256."""
    cache = oracle_cache(wl)
    out, lse_t = _gpu_attn(wl, cache, device, lse=lse)
    got = f32_of(out) if tokens is None else f32_of(out)[tokens]
    g_lse = None if not lse else (f32_of(lse_t) if tokens is None else f32_of(lse_t)[tokens])
    ref, ref_lse, bad = run_oracle(wl, cache, tokens=tokens)
    assert bad == 0
    check_close(got, ref, wl.name + (" (exact dequantisation)" if wl.kind == 1 else ""), max_abs=max_abs)
    if lse:
        _check_lse(g_lse, ref_lse, 2e-4)
    if wl.kind == 1 and wl.sm_scale <= 1.0 / np.sqrt(wl.D) + 1e-12:
        ref_d, ref_lse_d, _ = run_oracle_on_dequantised(wl, cache, tokens=tokens)
        check_close(got, ref_d, wl.name + " (bf16-rounded dequantised rows)", max_abs=max_abs)
        if lse:
            _check_lse(g_lse, ref_lse_d, 2e-2)
    return out


# ------------------------------------------------------------------ the named small configs --
def test_config1_bf16_direct_T17_k2112(gpu):
    _check(W.config(1), gpu)


def test_config2_fp8_paged_T8_k2048(gpu):
    _check(W.config(2), gpu)


# ------------------------------------------------------------------------- coverage matrix --
@pytest.mark.parametrize("T", [1, 8, 17])
@pytest.mark.parametrize("topk,n_valid", [(2048, 2048), (2112, 2051), (2112, 2112)])
@pytest.mark.parametrize("kind", [0, 1])
def test_matrix_direct(gpu, T, topk, n_valid, kind):
    if kind == 0:
        wl = W.bf16_direct(T=T, slots=6000, topk=topk, n_valid=n_valid, seed=100 + T, sm_scale=1 / 16)
    else:
        wl = W.fp8_paged(T=T, requests=1, positions=6016, page_size=64, topk=topk, n_valid=n_valid, seed=200 + T,
                         sm_scale=1 / 16)
        # direct-slot variant of the same FP8 problem: translate positions to slots on the host
        idx = wl.indices.astype(np.int64)
        phys = wl.block_table[0, np.maximum(idx, 0) // 64].astype(np.int64) * 64 + np.maximum(idx, 0) % 64
        wl.indices = np.where(idx >= 0, phys, -1).astype(np.int32)
        wl.block_table, wl.page_size, wl.req_of_token = None, 0, None
    _check(wl, gpu)


@pytest.mark.parametrize("T", [1, 8, 17])
@pytest.mark.parametrize("topk,n_valid", [(2048, 2048), (2112, 2051)])
@pytest.mark.parametrize("kind", [0, 1])
def test_matrix_paged(gpu, T, topk, n_valid, kind):
    wl = W.fp8_paged(T=T, requests=3, positions=4096, page_size=64, topk=topk, n_valid=n_valid, seed=300 + T,
                     sm_scale=1 / 16, scatter_frac=0.5)
    if kind == 0:
        wl.kind = 0
    _check(wl, gpu)


@pytest.mark.parametrize("kind", [0, 1])
@pytest.mark.parametrize("T", [1, 8])
def test_control_512_64(gpu, kind, T):
    wl = W.fp8_direct(T=T, slots=5000, topk=2048, n_valid=2048, seed=400 + T)
    wl.kind = kind
    _check(wl, gpu)


@pytest.mark.parametrize("T,topk,n_valid", [(1, 4096, 4096), (1, 4224, 4100), (3, 4096, 3001)])
def test_control_512_64_many_parts(gpu, T, topk, n_valid):
    """Long lists over few tokens: each (token, head half) sequence spans up to seventeen CTAs,
    so the head CTA merges up to sixteen parts, streamed through its idle code stages."""
    wl = W.fp8_paged(T=T, requests=2, positions=8192, page_size=64, topk=topk, n_valid=n_valid, d_nope=512,
                     d_rope=64, d_v=512, seed=70 + T + topk % 7, sm_scale=1 / 24, scatter_frac=0.5)
    _check(wl, gpu)


def test_control_512_64_paged_padded(gpu):
    wl = W.fp8_paged(T=5, requests=2, positions=4096, page_size=64, topk=2112, n_valid=2051, d_nope=512, d_rope=64,
                     d_v=512, seed=45, sm_scale=1 / 24, scatter_frac=0.4)
    _check(wl, gpu)


def test_control_512_64_edge_cases(gpu):
    """The 512+64 FP8 control with: token 0 all entries masked, token 1 one valid entry, token 2
    every entry the same slot, token 3 a list shorter than a tile, token 4 entries scattered
    among -1 (and -7), token 5 an index past the cache (masked and flagged)."""
    wl = W.fp8_direct(T=6, slots=3000, topk=2112, n_valid=2000, seed=47, sm_scale=1 / 24)
    idx = wl.indices
    idx[0, :] = -1
    idx[1, :] = -1
    idx[1, 1500] = 77
    idx[2, :] = 555
    idx[3, 90:] = -1
    idx[4, ::3] = -7
    idx[5, 2001] = 3000
    cache = oracle_cache(wl)
    err = torch.zeros(1, dtype=torch.int32, device=gpu)
    out, lse_t = _gpu_attn(wl, cache, gpu, lse=True, err=err)
    assert err.item() & dsa.DEVERR_INDEX_OUT_OF_RANGE
    ref, ref_lse, bad = run_oracle(wl, cache)
    assert bad == 1
    check_close(f32_of(out), ref, "control edge cases (exact dequantisation)", max_abs=MAX_ABS_ORDER_ONE)
    _check_lse(f32_of(lse_t), ref_lse, 2e-4)


@pytest.mark.parametrize("sm_scale", [0.0, 0.5, -1 / 24])
def test_control_512_64_scales(gpu, sm_scale):
    """The control at scale 0 (the mean of the rows), at 0.5 (scores of order 10-40 on rows of
    width 576: the lazy maxima of the row sums and of the four output quarters grow and rescale)
    and at a negative scale."""
    wl = W.fp8_direct(T=4, slots=4000, topk=2048, n_valid=2048, seed=48, sm_scale=sm_scale)
    _check(wl, gpu, max_abs=MAX_ABS_ORDER_ONE if sm_scale > 0.1 else MAX_ABS)


# -------------------------------------------------------------------------------- edge cases --
def test_masked_single_duplicate_and_small_topk(gpu):
    """Token 0: all entries masked; token 1: one valid entry; token 2: every entry the same slot;
    token 3: top-k list shorter than a tile; token 4: entries scattered among -1 (and -7)."""
    wl = W.bf16_direct(T=5, slots=900, topk=300, n_valid=250, seed=7, sm_scale=1 / 16)
    idx = wl.indices
    idx[0, :] = -1
    idx[1, :] = -1
    idx[1, 123] = 77
    idx[2, :] = 555
    idx[3, 5:] = -1
    idx[4, ::3] = -7
    # tokens 1 and 2 return one row (outputs of order one)
    _check(wl, gpu, max_abs=MAX_ABS_ORDER_ONE)
    wl.kind = 1
    wl.kv_slot = None
    _check(wl, gpu, max_abs=MAX_ABS_ORDER_ONE)


def test_single_entry_equals_row_bf16(gpu):
    """One valid entry: the softmax weight is exactly 1, so the output is the bf16 row itself."""
    wl = W.bf16_direct(T=3, slots=500, topk=2112, n_valid=1, seed=8, sm_scale=1 / 16)
    cache = oracle_cache(wl)
    out, _ = _gpu_attn(wl, cache, gpu)
    o = out.cpu()
    for t in range(3):
        j = wl.indices[t][wl.indices[t] >= 0][0]
        row = torch.from_numpy(cache[j].view(np.int16)).view(torch.bfloat16)
        assert torch.equal(o[t], row[None].expand(64, -1))


def test_repeated_pages_and_duplicates_paged(gpu):
    wl = W.fp8_paged(T=6, requests=2, positions=2048, page_size=64, topk=2048, n_valid=2000, seed=9, sm_scale=1 / 16)
    wl.block_table[1, :] = wl.block_table[1, 3]          # request 1: every logical page -> one physical page
    wl.indices[0, 1000:1500] = wl.indices[0, :500]        # duplicates are separate terms
    # request 1's tokens see only 64 distinct rows: outputs of order one
    _check(wl, gpu, max_abs=np.where(wl.req_of_token == 1, MAX_ABS_ORDER_ONE, MAX_ABS))


def test_out_of_range_entries_masked_and_flagged(gpu):
    wl = W.bf16_direct(T=4, slots=1000, topk=512, n_valid=500, seed=10, sm_scale=1 / 16)
    wl.indices[1, 7] = 1000
    wl.indices[2, 0] = 10 ** 8
    cache = oracle_cache(wl)
    err = torch.zeros(1, dtype=torch.int32, device=gpu)
    out, _ = _gpu_attn(wl, cache, gpu, err=err)
    assert err.item() & dsa.DEVERR_INDEX_OUT_OF_RANGE
    ref, _, bad = run_oracle(wl, cache)
    assert bad == 2
    check_close(f32_of(out), ref, "oob")


def test_sm_scale_zero_is_mean(gpu):
    wl = W.bf16_direct(T=2, slots=3000, topk=2112, n_valid=2051, seed=11, sm_scale=0.0)
    _check(wl, gpu)


def test_large_scores_no_overflow(gpu):
    """Scale 1.0 on N(0,1) rows of width 256 gives scores of order 16-60: exercises the lazy
    rescale (running max growth above 2^8) and the max subtraction."""
    wl = W.bf16_direct(T=8, slots=4000, topk=2048, n_valid=2048, seed=12, sm_scale=1.0)
    _check(wl, gpu, max_abs=MAX_ABS_ORDER_ONE)
    wl = W.fp8_paged(T=8, requests=2, positions=2048, page_size=64, topk=2048, n_valid=2048, seed=13, sm_scale=0.5)
    _check(wl, gpu, max_abs=MAX_ABS_ORDER_ONE)


@pytest.mark.parametrize("kind", [0, 1])
def test_negative_sm_scale(gpu, kind):
    """A negative scale reverses the ranking of the keys (the softmax favours the keys least
    aligned with q); any finite scale is accepted, as the pages set no limit."""
    if kind == 0:
        wl = W.bf16_direct(T=6, slots=4000, topk=2112, n_valid=2051, seed=17, sm_scale=-1 / 16, scatter_frac=0.2)
    else:
        wl = W.fp8_paged(T=6, requests=2, positions=4096, page_size=64, topk=2112, n_valid=2051, seed=18,
                         sm_scale=-1 / 16, scatter_frac=0.2)
    _check(wl, gpu)


def test_many_tokens_stream_split(gpu):
    """T small relative to the SM count: every token is split across several CTAs and merged."""
    for T in (2, 3, 40):
        wl = W.bf16_direct(T=T, slots=5000, topk=2112, n_valid=2051, seed=20 + T, sm_scale=1 / 16, scatter_frac=0.3)
        _check(wl, gpu)


@pytest.mark.parametrize("kind", [0, 1])
@pytest.mark.parametrize("T,topk", [(1, 8192), (2, 4096), (37, 2048), (74, 2048), (150, 2048)])
def test_split_token_merge_part_counts(gpu, kind, T, topk):
    """Batches whose tokens span up to sixteen, eight, four, three and two CTAs: the head CTA's
    merge streams every part through its two shared-memory slot pairs (more than two parts
    reuse them) and adds them in a fixed order."""
    wl = W.fp8_paged(T=T, requests=2, positions=2 * topk, page_size=64, topk=topk, n_valid=topk - 48,
                     seed=60 + T, sm_scale=1 / 16, scatter_frac=0.3)
    if kind == 0:
        wl.kind = 0
    _check(wl, gpu)


def test_strided_q_and_out(gpu):
    wl = W.bf16_direct(T=5, slots=3000, topk=2048, n_valid=2048, seed=14, sm_scale=1 / 16)
    cache = oracle_cache(wl)
    q, dcache, idx, _, _ = _dev_inputs(wl, cache, gpu)
    qbig = torch.zeros((5, 64, 320), dtype=torch.bfloat16, device=gpu)
    qbig[:, :, :256] = q
    outbig = torch.full((5, 64, 264), 7.0, dtype=torch.bfloat16, device=gpu)
    dsa.dsa_sparse_attn(qbig[:, :, :256], dcache, 0, idx, wl.sm_scale, out=outbig[:, :, :256])
    torch.cuda.synchronize()
    ref, _, _ = run_oracle(wl, cache)
    check_close(f32_of(outbig[:, :, :256]), ref, "strided")
    assert (outbig[:, :, 256:] == 7.0).all()


def test_bit_identical_repeats(gpu):
    for wl in (W.config(1), W.config(2)):
        cache = oracle_cache(wl)
        q, dcache, idx, bt, req = _dev_inputs(wl, cache, gpu)
        outs = []
        for _ in range(10):
            o = dsa.dsa_sparse_attn(q, dcache, wl.kind, idx, wl.sm_scale, block_table=bt, page_size=wl.page_size,
                                    req_of_token=req)
            outs.append(o.clone())
        torch.cuda.synchronize()
        for o in outs[1:]:
            assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))


def _scaled_halves(bits, lo, hi):
    """bf16 bits with columns 0-127 multiplied by 2^lo and 128-255 by 2^hi (exact)."""
    f = (bits.astype(np.uint32) << 16).view(np.float32).copy()
    f[:, :128] *= 2.0 ** lo
    f[:, 128:] *= 2.0 ** hi
    return (f.view(np.uint32) >> 16).astype(np.uint16)


@pytest.mark.parametrize("e", [10, -10, 16, -16])
def test_fp8_tile_scales_applied_per_tile(gpu, e):
    """Rows whose two 128-column tiles differ in magnitude by 2^(2e), so that their tile scales
    do, with the query scaled inversely (scores stay of order one): the kernel applies each
    tile's fp32 scale to its own half of the score and of the output (at |e| = 16 one tile's
    scales are about 2^9, the other's about 2^-23). Each output half is compared after undoing
    its exact power-of-two factor, i.e. at the precision of the unscaled problem; the LSE is
    unaffected by the value scaling and is checked as is."""
    wl = W.fp8_paged(T=6, requests=1, positions=4096, page_size=64, topk=2112, n_valid=2051, seed=15, sm_scale=1 / 16)
    wl.kv = W.FixedRows(_scaled_halves(wl.kv.bits(), -e, e))
    wl.q = W.FixedRows(_scaled_halves(wl.q.bits(), e, -e))
    cache = oracle_cache(wl)
    out, lse_t = _gpu_attn(wl, cache, gpu, lse=True)
    ref, ref_lse, bad = run_oracle(wl, cache)
    assert bad == 0
    undo = np.concatenate([np.full(128, 2.0 ** e), np.full(128, 2.0 ** -e)])
    check_close(f32_of(out) * undo, ref * undo, "fp8 tile scales")
    _check_lse(f32_of(lse_t), ref_lse, 2e-4)


def test_fp8_large_scale_rows_among_ordinary_ones(gpu):
    """Every seventh row has its second tile replaced by its magnitude times 2^15 (tile scales
    above 2^7), the query's second half scaled by 2^-15: one loader warp holds rows with scales
    2^15 apart in the same tile half, and each row's scale must reach only that row. Those rows
    dominate the second half of the output; their values there are positive, so the output is
    a sum without cancellation and keeps the precision of its terms (signed values of that size
    would cancel to outputs far smaller than the terms, below what bf16 probabilities resolve).
    Output and LSE against the exact oracle."""
    wl = W.fp8_paged(T=5, requests=1, positions=4096, page_size=64, topk=2048, n_valid=2048, seed=16, sm_scale=1 / 16)
    kv = (wl.kv.bits().astype(np.uint32) << 16).view(np.float32).copy()
    kv[::7, 128:] = np.abs(kv[::7, 128:]) * 2.0 ** 15
    wl.kv = W.FixedRows((kv.view(np.uint32) >> 16).astype(np.uint16))
    q = (wl.q.bits().astype(np.uint32) << 16).view(np.float32).copy()
    q[:, 128:] *= 2.0 ** -15
    wl.q = W.FixedRows((q.view(np.uint32) >> 16).astype(np.uint16))
    cache = oracle_cache(wl)
    scales = cache[:, 256:264].copy().view(np.float32)
    big = np.zeros(wl.num_slots, dtype=bool)
    big[::7] = True
    assert scales[wl.kv_slot[big], 1].min() >= 128.0 and scales[wl.kv_slot[~big], 1].max() < 128.0
    out, lse_t = _gpu_attn(wl, cache, gpu, lse=True)
    ref, ref_lse, bad = run_oracle(wl, cache)
    assert bad == 0
    # the second output half holds values of order 2^15: compare it scaled back by that exact
    # power of two, where the outputs are of order one
    undo = np.concatenate([np.ones(128), np.full(128, 2.0 ** -15)])
    check_close(f32_of(out) * undo, ref * undo, "fp8 large-scale rows", max_abs=MAX_ABS_ORDER_ONE)
    _check_lse(f32_of(lse_t), ref_lse, 2e-4)


def test_balanced_split_causal_prefill(gpu):
    """Long causal lists (T=3072, top-k 2048): every CTA holds hundreds of (token, 128-entry)
    units, so the CTA ranges come from the work-balanced split by valid entries, and the first
    2048 tokens' lists are mostly padding. Sampled tokens (including split ones) against the
    oracle; repeated calls are bit-identical (the split depends only on the index lists)."""
    wl = W.prefill_causal(T=3072, topk=2048, window=128, seed=31, name="prefill_causal_T3072")
    rng = np.random.default_rng(5)
    tokens = np.unique(np.concatenate([np.arange(0, wl.T, 97), rng.integers(0, wl.T, 16),
                                       [0, 1, 127, 128, 2047, 2048, wl.T - 1]]))
    out = _check(wl, gpu, tokens=tokens, max_abs=token_gates(wl.indices, tokens))
    cache = oracle_cache(wl)
    again, _ = _gpu_attn(wl, cache, gpu)
    assert torch.equal(again.view(torch.int16), out.view(torch.int16))


def test_balanced_split_with_every_entry_masked(gpu):
    """Many tokens whose lists are all padding: the work-balanced split sees only the per-token
    weights (no valid entry anywhere). Every output is zero and every lse -inf."""
    T, topk = 2048, 2048
    wl = W.bf16_direct(T=T, slots=512, topk=topk, n_valid=1, seed=90, sm_scale=1 / 16)
    wl.indices[:] = -1
    out, lse_t = _gpu_attn(wl, oracle_cache(wl), gpu, lse=True)
    assert (f32_of(out) == 0).all()
    assert np.isneginf(f32_of(lse_t)).all()
