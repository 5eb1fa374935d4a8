"""Parity at the benchmark's full sizes and in its launch configuration: the FP8 paged decode
(T=256, top-k 2112 over an 8.4M-slot packed cache), the BF16 causal prefill (T=8192, top-k 2048)
and the 512+64 control (T=1024). The GPU runs the whole batch exactly as bench.py does: inputs
generated on the device, the cache packed by dsa_quant_k_cache, one dsa_sparse_attn call. The
oracle recomputes sampled tokens from its own pack of the same seeded source rows (the
counter-based generator gives every row by index on the host), gathered through a compact
direct view of the slots those tokens name; no oracle input comes from the GPU."""
import numpy as np
import pytest
import torch

import bench
import oracle
import dsa_sparse_attention_mla_gb300 as dsa
from dsa_sparse_attention_mla_gb300 import workloads as W

from _helpers import check_close, f32_of, token_gates

pytestmark = pytest.mark.gpu


def _physical_slots(wl, tokens):
    """[n, topk] physical slot of every entry of the given tokens (-1 where masked)."""
    idx = wl.indices[tokens].astype(np.int64)
    valid = idx >= 0
    pos = np.where(valid, idx, 0)
    if wl.block_table is None:
        phys = pos
    else:
        req = wl.req_of_token[tokens].astype(np.int64)[:, None]
        phys = wl.block_table[req, pos // wl.page_size].astype(np.int64) * wl.page_size + pos % wl.page_size
    return np.where(valid, phys, -1)


def _oracle_tokens(wl, tokens):
    """fp64 oracle (out, lse, and for packed rows also over the bf16-rounded rows) of the given
    tokens, over a compact cache of only the slots they name."""
    phys = _physical_slots(wl, tokens)
    slots = np.unique(phys[phys >= 0])
    assert wl.kv_slot is None  # slot i holds source row i
    src = wl.kv.bits(slots)
    sub = np.where(phys >= 0, np.searchsorted(slots, np.maximum(phys, 0)), -1).astype(np.int32)
    H, D = wl.H, wl.D
    q_rows = (np.asarray(tokens, dtype=np.int64)[:, None] * H + np.arange(H)[None, :]).ravel()
    q = wl.q.bits(q_rows).reshape(len(tokens), H, D)
    if wl.kind == oracle.CACHE_BF16:
        cache = src
    else:
        rb = oracle.packed_row_bytes(wl.d_nope, wl.d_rope)
        cache = oracle.quant_k_cache(src[:, : wl.d_nope], src[:, wl.d_nope:] if wl.d_rope else None,
                                     cache=np.zeros((len(slots), rb), dtype=np.uint8), num_slots=len(slots))
    out, lse, bad = oracle.sparse_attn(q, cache, wl.kind, wl.d_nope, wl.d_rope, wl.d_v, sub, wl.sm_scale)
    assert bad == 0
    rounded = None
    if wl.kind == oracle.CACHE_FP8_SCALED:
        deq, bad = oracle.gather_dequant(cache, oracle.CACHE_FP8_SCALED, wl.d_nope, wl.d_rope,
                                         np.arange(len(slots), dtype=np.int32))
        assert bad == 0
        rounded = oracle.sparse_attn(q, deq, oracle.CACHE_BF16, wl.d_nope, wl.d_rope, wl.d_v, sub, wl.sm_scale)[:2]
    return out, lse, rounded


def _gpu_full(wl, device):
    q, cache, idx, bt, req = bench.build_device_inputs(wl, device)
    lse = torch.empty((wl.T, wl.H), dtype=torch.float32, device=device)
    out = dsa.dsa_sparse_attn(q, cache, wl.kind, idx, wl.sm_scale, d_nope=wl.d_nope, d_rope=wl.d_rope, d_v=wl.d_v,
                              block_table=bt, page_size=wl.page_size, req_of_token=req, lse=lse)
    torch.cuda.synchronize()
    del q, cache
    return out, lse


def _check_sampled(wl, tokens, device):
    out, lse = _gpu_full(wl, device)
    got, g_lse = f32_of(out)[tokens], f32_of(lse)[tokens]
    ref, ref_lse, rounded = _oracle_tokens(wl, tokens)
    gates = token_gates(wl.indices, tokens)
    check_close(got, ref, wl.name + f" ({len(tokens)} tokens)", max_abs=gates)
    np.testing.assert_allclose(g_lse, ref_lse, rtol=1e-5, atol=2e-4)
    if rounded is not None and wl.sm_scale <= 1.0 / np.sqrt(wl.D) + 1e-12:
        check_close(got, rounded[0], wl.name + " (bf16-rounded dequantised rows)", max_abs=gates)
        np.testing.assert_allclose(g_lse, rounded[1], rtol=1e-5, atol=2e-2)
    return out


def test_config3_fp8_paged_decode_full_size(gpu):
    """Every one of the 256 tokens (those with a -1 tail and those with scattered -1 entries)."""
    wl = W.config(3)
    assert (wl.indices[:, :-64] < 0).any(axis=1).sum() > 0
    _check_sampled(wl, np.arange(wl.T), gpu)


def test_config4_bf16_causal_prefill_full_size(gpu):
    """256 tokens: the short causal lists (t < 2048) and the boundary, split tokens and full
    windows, then random ones."""
    wl = W.config(4)
    rng = np.random.default_rng(4)
    fixed = np.array([0, 1, 2, 63, 64, 127, 128, 129, 1023, 1024, 2046, 2047, 2048, 2049, 4095, 4096, wl.T - 2, wl.T - 1])
    rest = rng.choice(np.setdiff1d(np.arange(wl.T), fixed), 256 - len(fixed), replace=False)
    _check_sampled(wl, np.unique(np.concatenate([fixed, rest])), gpu)


def test_config5_fp8_512_64_full_size(gpu):
    """256 of the 1024 tokens, the first and last included."""
    wl = W.config(5)
    rng = np.random.default_rng(5)
    rest = rng.choice(np.arange(1, wl.T - 1), 254, replace=False)
    _check_sampled(wl, np.unique(np.concatenate([[0, wl.T - 1], rest])), gpu)
