"""Shared helpers for the GPU parity tests: moving bit patterns between numpy and torch, building
caches with the oracle, and the tolerance gates.

Tolerances (attention): every element must satisfy |gpu - oracle| <= 2e-2 + 1e-2 * |oracle|
(the bound stated for this path: max-abs 2e-2 and max-rel 1e-2 against the fp64 oracle on the
same dequantised inputs), and in aggregate ||gpu - oracle||_F <= 1e-2 * ||oracle||_F, which a
kernel with a dropped term or a wrong row would fail even where outputs are near zero.
"""
import numpy as np
import torch

import oracle

ATOL, RTOL, FRO = 2e-2, 1e-2, 1e-2


def bf16_dev(bits, device):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def bits_of(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def f32_of(t):
    return t.detach().cpu().float().numpy()


def oracle_cache(wl, rows=None):
    """Host cache bytes for a workload, built by the oracle (uint8 rows for FP8, bf16 bits for BF16).

    ``rows``: only these kv rows are generated and written (the rest stay zero) - enough for an
    oracle run restricted to tokens whose entries name only those rows."""
    if wl.kind == oracle.CACHE_BF16:
        if rows is None:
            return wl.kv.bits()
        cache = np.zeros((wl.num_slots, wl.D), dtype=np.uint16)
        cache[rows] = wl.kv.bits(rows)
        return cache
    src = wl.kv.bits() if rows is None else wl.kv.bits(rows)
    if rows is None:
        loc = wl.kv_slot
    else:
        loc = (wl.kv_slot[rows] if wl.kv_slot is not None else np.asarray(rows, dtype=np.int64))
    rb = oracle.packed_row_bytes(wl.d_nope, wl.d_rope)
    cache = np.zeros((wl.num_slots, rb), dtype=np.uint8)
    return oracle.quant_k_cache(src[:, : wl.d_nope], src[:, wl.d_nope:] if wl.d_rope else None,
                                out_loc=None if loc is None else np.asarray(loc, dtype=np.int64), cache=cache,
                                num_slots=wl.num_slots)


def slots_of_tokens(wl, tokens):
    """Physical slots named by the valid entries of the given tokens."""
    idx = wl.indices[tokens].astype(np.int64)
    valid = idx >= 0
    if wl.block_table is None:
        s = idx[valid]
    else:
        r = wl.req_of_token[tokens][:, None].repeat(idx.shape[1], axis=1)[valid]
        pos = idx[valid]
        s = wl.block_table[r, pos // wl.page_size].astype(np.int64) * wl.page_size + pos % wl.page_size
    return np.unique(s)


def run_oracle(wl, cache, tokens=None, n_threads=0):
    return oracle.sparse_attn(wl.q_bits(), cache, wl.kind, wl.d_nope, wl.d_rope, wl.d_v, wl.indices, wl.sm_scale,
                              block_table=wl.block_table, page_size=wl.page_size, req_of_token=wl.req_of_token,
                              tokens=tokens, n_threads=n_threads)


def dequantised_rows(wl, cache, rows=None):
    """The bf16 rows the FP8 path computes on: the oracle's gather/dequant output
    bf16_rne(fp32(code) * scale) for every slot (or only ``rows``; other slots zero)."""
    if rows is None:
        rows = np.arange(wl.num_slots)
    rows = np.asarray(rows, dtype=np.int64)
    deq, bad = oracle.gather_dequant(cache, oracle.CACHE_FP8_SCALED, wl.d_nope, wl.d_rope, rows.astype(np.int32))
    assert bad == 0
    out = np.zeros((wl.num_slots, wl.D), dtype=np.uint16)
    out[rows] = deq
    return out


def run_oracle_on_dequantised(wl, cache, tokens=None, rows=None, n_threads=0):
    """fp64 oracle attention over the same dequantised (bf16) rows the FP8 kernel uses."""
    deq = dequantised_rows(wl, cache, rows)
    return oracle.sparse_attn(wl.q_bits(), deq, oracle.CACHE_BF16, wl.d_nope, wl.d_rope, wl.d_v, wl.indices,
                              wl.sm_scale, block_table=wl.block_table, page_size=wl.page_size,
                              req_of_token=wl.req_of_token, tokens=tokens, n_threads=n_threads)


def check_close(gpu, ref, what=""):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    assert np.isfinite(gpu).all(), f"{what}: non-finite output"
    err = np.abs(gpu - ref)
    bound = ATOL + RTOL * np.abs(ref)
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    assert (err <= bound).all(), f"{what}: max err {err.max():.3e} at {worst} (ref {ref[worst]:.4f}, gpu {gpu[worst]:.4f})"
    fro = np.linalg.norm(gpu - ref) / max(np.linalg.norm(ref), 1e-30)
    assert fro <= FRO, f"{what}: relative Frobenius error {fro:.3e}"
    return float(err.max()), float(fro)
