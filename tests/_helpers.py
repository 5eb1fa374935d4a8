"""Shared helpers for the GPU parity tests: moving bit patterns between numpy and torch, building
caches with the oracle, and the tolerance gates.

Tolerances (attention), every one enforced by check_close:
  - elementwise |gpu - oracle| <= 2e-2 + 1e-2 * |oracle| (the bound stated for this path:
    max-abs 2e-2 and max-rel 1e-2 against the fp64 oracle on the same dequantised inputs);
  - max |gpu - oracle| <= 5e-3 for outputs of the workloads' scale (averages of hundreds of
    unit-variance rows, a spread of about 0.04, where the observed error is about 1e-3): a wrong
    row or a dropped term moves an output by far more. Tests whose outputs are of order one
    (a single dominant key, large sm_scale) pass max_abs=2e-2, the literal bound, which their
    bf16 output rounding alone (2^-9 relative) can approach;
  - ||gpu - oracle||_F <= 1e-2 * ||oracle||_F, which a kernel with a dropped term or a wrong
    row fails even where outputs are near zero.
"""
import numpy as np
import torch

import oracle
from oracle.workload_inputs import oracle_cache, slots_of_tokens  # noqa: F401 (re-exported)

ATOL, RTOL, FRO, MAX_ABS = 2e-2, 1e-2, 1e-2, 5e-3
MAX_ABS_ORDER_ONE = 2e-2


def bf16_dev(bits, device):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def bits_of(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def f32_of(t):
    return t.detach().cpu().float().numpy()


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


def check_close(gpu, ref, what="", max_abs=MAX_ABS):
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
    emax = float(err.max()) if err.size else 0.0
    print(f"[check_close] {what}: max abs err {emax:.3e}, rel Frobenius {fro:.3e}, |ref| max {np.abs(ref).max() if ref.size else 0:.3e}")
    if max_abs is not None:
        # a scalar, or one gate per token (first axis)
        gate = np.asarray(max_abs, dtype=np.float64).reshape((-1,) + (1,) * (err.ndim - 1))
        over = err - gate
        arg = np.unravel_index(np.argmax(over), err.shape)
        assert over.max() <= 0, (f"{what}: abs err {err[arg]:.3e} > {np.broadcast_to(gate, err.shape)[arg]:.1e} at "
                                 f"{arg} (ref {ref[arg]:.4f})")
    return emax, float(fro)


def token_gates(indices, tokens=None, few=256):
    """Per-token max-abs gates: MAX_ABS for tokens with at least ``few`` valid entries (outputs
    are averages of many rows), MAX_ABS_ORDER_ONE for tokens with fewer (a causal prefix of a
    handful of keys gives outputs of order one)."""
    idx = indices if tokens is None else indices[tokens]
    n = (idx >= 0).sum(axis=1)
    return np.where(n >= few, MAX_ABS, MAX_ABS_ORDER_ONE)
