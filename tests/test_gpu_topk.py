"""GPU top-k selection (dsa_topk_select) against the oracle's stable sort, element for element:
random scores at the decode and prefill widths (top-k 2048 and 2112), causal row lengths, heavy
ties (the lowest positions must win), signed zeros and infinities, rows shorter than K, and the
lists fed end to end into dsa_sparse_attn against the oracle attention over the oracle's lists."""
import numpy as np
import pytest
import torch

import dsa_sparse_attention_mla_gb300 as dsa
from dsa_sparse_attention_mla_gb300 import workloads as W
from oracle.selection import topk_select

from _helpers import bf16_dev, check_close, f32_of, oracle_cache, run_oracle

pytestmark = pytest.mark.gpu


def _gpu(scores, K, lengths=None, device="cuda:0"):
    s = torch.from_numpy(np.ascontiguousarray(scores)).to(device)
    ln = None if lengths is None else torch.from_numpy(np.asarray(lengths, dtype=np.int32)).to(device)
    out = dsa.dsa_topk_select(s, K, lengths=ln)
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("K", [2048, 2112])
def test_random_scores_causal_lengths(gpu, K):
    rng = np.random.default_rng(K)
    T, S = 48, 32768
    scores = rng.standard_normal((T, S)).astype(np.float32)
    lengths = rng.integers(0, S + 1, size=T)
    lengths[:4] = [0, 1, K - 1, K]           # empty, single, short of K, exactly K
    lengths[4:6] = [K + 1, S]
    got = _gpu(scores, K, lengths, gpu)
    ref = topk_select(scores, K, lengths)
    assert np.array_equal(got, ref)


def test_heavy_ties_take_the_lowest_positions(gpu):
    rng = np.random.default_rng(5)
    T, S, K = 24, 8192, 2048
    scores = (rng.integers(0, 16, size=(T, S)) * 0.25).astype(np.float32)   # 16 distinct values
    scores[0] = 1.0                                                          # a row of one value
    got = _gpu(scores, K, None, gpu)
    assert np.array_equal(got, topk_select(scores, K))


@pytest.mark.parametrize("distinct", [8, 64, 1000])
def test_heavy_ties_long_rows(gpu, distinct):
    """Rows of 32768 positions (the one-row-per-SM kernel, which sets the keys matching the top
    16 bits of the K-th largest aside after two radix passes): with 8 distinct values those keys
    overflow the set-aside list and the row takes the full passes; with 64 and 1000 they fit, and
    the ties at the K-th largest value outnumber the places left, so the lowest positions must
    be taken in order."""
    rng = np.random.default_rng(100 + distinct)
    T, S = 12, 32768
    for K in (2048, 2112):
        scores = (rng.integers(0, distinct, size=(T, S)) * 0.125).astype(np.float32)
        lengths = rng.integers(K + 1, S + 1, size=T)
        lengths[0] = S
        got = _gpu(scores, K, lengths, gpu)
        assert np.array_equal(got, topk_select(scores, K, lengths))


def test_signed_zeros_infinities_and_short_rows(gpu):
    rng = np.random.default_rng(6)
    pool = np.array([-np.inf, -2.0, -0.0, 0.0, 3.0, np.inf], dtype=np.float32)
    for S, K in [(100, 64), (100, 2112), (5000, 2048), (1, 1), (3000, 16384)]:
        scores = pool[rng.integers(0, len(pool), size=(7, S))]
        lengths = rng.integers(-2, S + 3, size=7)
        got = _gpu(scores, K, lengths, gpu)
        assert np.array_equal(got, topk_select(scores, K, lengths)), (S, K)


def test_prefill_shape_and_repeats(gpu):
    """T = 512 rows with the causal lengths of a prefill (row t sees t + 1 positions); two calls
    agree bit for bit."""
    rng = np.random.default_rng(7)
    T, S, K = 512, 4096, 2048
    scores = rng.standard_normal((T, S)).astype(np.float32)
    lengths = np.arange(1, T + 1) * (S // T)
    a = _gpu(scores, K, lengths, gpu)
    b = _gpu(scores, K, lengths, gpu)
    assert np.array_equal(a, b)
    assert np.array_equal(a, topk_select(scores, K, lengths))


def test_selected_lists_feed_the_attention(gpu):
    """Scores over each request's positions -> dsa_topk_select -> dsa_sparse_attn on the packed
    paged cache; the oracle attention runs on the oracle's own lists (which the GPU lists equal)."""
    wl = W.fp8_paged(T=8, requests=2, positions=4096, page_size=64, topk=2112, n_valid=2051, seed=81, sm_scale=1 / 16)
    rng = np.random.default_rng(8)
    scores = rng.standard_normal((wl.T, 4096)).astype(np.float32)
    lengths = rng.integers(1500, 4097, size=wl.T)
    ref_idx = topk_select(scores, 2112, lengths)
    got_idx = _gpu(scores, 2112, lengths, gpu)
    assert np.array_equal(got_idx, ref_idx)
    wl.indices = ref_idx
    cache = oracle_cache(wl)
    q = bf16_dev(wl.q_bits(), gpu)
    out = dsa.dsa_sparse_attn(q, torch.from_numpy(cache).to(gpu), wl.kind, torch.from_numpy(got_idx).to(gpu),
                              wl.sm_scale, block_table=torch.from_numpy(wl.block_table).to(gpu),
                              page_size=wl.page_size, req_of_token=torch.from_numpy(wl.req_of_token).to(gpu))
    torch.cuda.synchronize()
    ref, _, bad = run_oracle(wl, cache)
    assert bad == 0
    check_close(f32_of(out), ref, "top-k lists into the attention")
