"""Pins of the oracle's sparse attention (step-by-step gather, mask, score, softmax, weighted sum) against
dense attention from a library routine, closed forms and invariances.

The attention the pages check (sglang PR #38547, Direct GLM geometry coverage list): per token
gather the top-k latent rows, mask -1 entries, score 64 heads against the rows, softmax, and sum
the same rows (first d_v elements) weighted by the probabilities.
"""
import numpy as np
import pytest
import torch

from dsa_sparse_attention_mla_gb300 import workloads as W


def _f64(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).double()


def _dequant_torch(cache, d_nope, d_rope):
    """Exact fp64 dequantisation with torch's float8 decode (independent of the oracle)."""
    n = cache.shape[0]
    codes = torch.from_numpy(cache[:, :d_nope].copy()).view(torch.float8_e4m3fn).double()
    t = d_nope // 128
    sc = torch.from_numpy(cache[:, d_nope: d_nope + 4 * t].copy().view("<f4").astype(np.float64))
    k = codes * sc.repeat_interleave(128, dim=1)
    if d_rope:
        rope = cache[:, d_nope + 4 * t:].copy().view("<u2")
        k = torch.cat([k, _f64(rope)], dim=1)
    return k.reshape(n, d_nope + d_rope)


def _dense(q_bits, k, d_v, scale):
    q = _f64(q_bits)                                    # [T, H, D]
    kk = k[None, None].expand(q.shape[0], 1, *k.shape)  # [T, 1, S, D]
    v = kk[..., :d_v]
    out = torch.nn.functional.scaled_dot_product_attention(q[:, :, None], kk.expand(-1, q.shape[1], -1, -1),
                                                           v.expand(-1, q.shape[1], -1, -1), scale=scale)
    s = torch.einsum("thd,sd->ths", q, k) * scale
    return out[:, :, 0].numpy(), torch.logsumexp(s, dim=-1).numpy()


@pytest.mark.parametrize("kind,d_nope,d_rope,d_v", [(0, 256, 0, 256), (1, 256, 0, 256), (1, 512, 64, 512)])
def test_dense_equivalence(oracle, kind, d_nope, d_rope, d_v):
    slots, T, H = 192, 3, 64
    D = d_nope + d_rope
    kv = W.NormalRows(11, 1, slots, D).bits()
    q = W.NormalRows(11, 2, T * H, D).bits().reshape(T, H, D)
    if kind == 0:
        cache = kv
        k = _f64(kv)
    else:
        cache = oracle.quant_k_cache(kv[:, :d_nope], kv[:, d_nope:] if d_rope else None)
        k = _dequant_torch(cache, d_nope, d_rope)
    rng = np.random.default_rng(0)
    idx = np.stack([rng.permutation(slots) for _ in range(T)]).astype(np.int32)
    scale = 1.0 / np.sqrt(D)
    out, lse, bad = oracle.sparse_attn(q, cache, kind, d_nope, d_rope, d_v, idx, scale)
    ref, ref_lse = _dense(q, k, d_v, scale)
    assert bad == 0
    np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-12, atol=1e-12)


def test_single_entry_gives_the_row(oracle):
    kv = W.NormalRows(12, 1, 64, 256).bits()
    q = W.NormalRows(12, 2, 2 * 64, 256).bits().reshape(2, 64, 256)
    idx = np.full((2, 16), -1, dtype=np.int32)
    idx[0, 9] = 17
    idx[1, 0] = 63
    out, lse, _ = oracle.sparse_attn(q, kv, 0, 256, 0, 256, idx, 1 / 16)
    assert np.array_equal(out[0], np.broadcast_to(_f64(kv[17]).numpy(), (64, 256)))
    assert np.array_equal(out[1], np.broadcast_to(_f64(kv[63]).numpy(), (64, 256)))
    s = (_f64(q[0]) @ _f64(kv[17])).numpy() / 16
    np.testing.assert_allclose(lse[0], s, rtol=1e-14, atol=1e-14)


def test_zero_scale_gives_mean_of_rows(oracle):
    kv = W.NormalRows(13, 1, 300, 256).bits()
    q = W.NormalRows(13, 2, 64, 256).bits().reshape(1, 64, 256)
    rng = np.random.default_rng(1)
    sel = rng.choice(300, 50, replace=False)
    idx = np.full((1, 80), -1, dtype=np.int32)
    idx[0, rng.choice(80, 50, replace=False)] = sel
    out, lse, _ = oracle.sparse_attn(q, kv, 0, 256, 0, 256, idx, 0.0)
    mean = _f64(kv[sel]).mean(0).numpy()
    np.testing.assert_allclose(out[0], np.broadcast_to(mean, (64, 256)), rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(lse, np.log(50.0), rtol=1e-14)


def test_invariances(oracle):
    """Permuting the list, inserting -1 entries, and duplicating the whole list leave the output
    unchanged (exact arithmetic; fp64 rounding differences only)."""
    slots = 1000
    kv = W.NormalRows(14, 1, slots, 256).bits()
    q = W.NormalRows(14, 2, 4 * 64, 256).bits().reshape(4, 64, 256)
    rng = np.random.default_rng(2)
    base = np.stack([rng.choice(slots, 300, replace=False) for _ in range(4)]).astype(np.int32)
    perm = np.stack([r[rng.permutation(300)] for r in base])
    padded = np.full((4, 420), -1, dtype=np.int32)
    for t in range(4):
        padded[t, np.sort(rng.choice(420, 300, replace=False))] = base[t]
    dup = np.concatenate([base, base[:, ::-1]], axis=1)
    ref, ref_lse, _ = oracle.sparse_attn(q, kv, 0, 256, 0, 256, base, 1 / 16)
    for other, dl in ((perm, 0.0), (padded, 0.0), (dup, np.log(2.0))):
        out, lse, _ = oracle.sparse_attn(q, kv, 0, 256, 0, 256, other, 1 / 16)
        np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(lse, ref_lse + dl, rtol=1e-12, atol=1e-12)


def test_planted_key_dominates(oracle):
    """A key aligned with the query and a large score takes (almost) all the weight: catches a
    missing max subtraction (overflow) and a wrong softmax axis."""
    slots = 400
    kv = W.NormalRows(15, 1, slots, 256).bits()
    q = W.NormalRows(15, 2, 64, 256).bits().reshape(1, 64, 256)
    kv = kv.copy()
    kv[123] = q[0, 5]                  # key 123 equals head 5's query
    idx = np.arange(slots, dtype=np.int32)[None]
    out, lse, _ = oracle.sparse_attn(q, kv, 0, 256, 0, 256, idx, 10.0)
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    np.testing.assert_allclose(out[0, 5], _f64(kv[123]).numpy(), rtol=0, atol=1e-12)
    assert not np.allclose(out[0, 6], _f64(kv[123]).numpy(), atol=1e-3)


def test_all_masked_and_out_of_range(oracle):
    kv = W.NormalRows(16, 1, 32, 256).bits()
    q = W.NormalRows(16, 2, 2 * 64, 256).bits().reshape(2, 64, 256)
    idx = np.array([[-1, -1, -5, -1], [3, 32, 99999, -1]], dtype=np.int32)
    out, lse, bad = oracle.sparse_attn(q, kv, 0, 256, 0, 256, idx, 1 / 16)
    assert bad == 2
    assert (out[0] == 0).all() and np.isneginf(lse[0]).all()
    assert np.array_equal(out[1], np.broadcast_to(_f64(kv[3]).numpy(), (64, 256)))


def test_paged_equals_direct_after_translation(oracle):
    wl = W.fp8_paged(T=5, requests=3, positions=1024, page_size=64, topk=300, n_valid=280, seed=4)
    kv = wl.kv.bits()
    cache = oracle.quant_k_cache(kv, out_loc=wl.kv_slot, num_slots=wl.num_slots)
    q = wl.q_bits()
    out_p, lse_p, bad = oracle.sparse_attn(q, cache, 1, 256, 0, 256, wl.indices, wl.sm_scale,
                                          block_table=wl.block_table, page_size=wl.page_size,
                                          req_of_token=wl.req_of_token)
    assert bad == 0
    # translate logical positions by hand and run in direct mode
    idx = wl.indices.astype(np.int64)
    r = wl.req_of_token[:, None]
    phys = wl.block_table[r, np.maximum(idx, 0) // 64] * 64 + np.maximum(idx, 0) % 64
    direct = np.where(idx >= 0, phys, -1).astype(np.int32)
    out_d, lse_d, _ = oracle.sparse_attn(q, cache, 1, 256, 0, 256, direct, wl.sm_scale)
    assert np.array_equal(out_p, out_d) and np.array_equal(lse_p, lse_d)
    # and the physical rows hold the latent of the logical positions (out_loc write path)
    direct_kv = oracle.quant_k_cache(kv)
    logical = np.where(idx >= 0, r * 1024 + np.maximum(idx, 0), -1).astype(np.int32)
    out_l, _, _ = oracle.sparse_attn(q, direct_kv, 1, 256, 0, 256, logical, wl.sm_scale)
    assert np.array_equal(out_l, out_p)


def test_token_subset_matches_full(oracle):
    wl = W.bf16_direct(T=9, slots=700, topk=260, n_valid=250, seed=5)
    q, kv = wl.q_bits(), wl.kv.bits()
    full, lse_full, _ = oracle.sparse_attn(q, kv, 0, 256, 0, 256, wl.indices, wl.sm_scale)
    sub, lse_sub, _ = oracle.sparse_attn(q, kv, 0, 256, 0, 256, wl.indices, wl.sm_scale, tokens=[8, 2, 5])
    assert np.array_equal(sub, full[[8, 2, 5]]) and np.array_equal(lse_sub, lse_full[[8, 2, 5]])
