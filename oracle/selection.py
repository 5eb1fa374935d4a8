"""CPU oracle for top-k index selection (test infrastructure only).

The selection step that feeds the sparse attention: for each query token, the positions of its
top-k index-logits, padded with -1 (FreeToken PR #270 "glm5_next: support GLM-5.3-Flash",
Summary, the DSA key-pooling bullet: pooled keys are scored, and the best-scoring positions
are what the sparse kernels gather; sglang PR #38547 "Enable zero-RoPE TileLang DSA on gfx950",
Direct GLM geometry coverage list: top-k widths 2048 and 2112, rows padded with -1). The pages
give the scoring no formula, so the scores are an input here.

Definition (a plain stable sort, nothing blocked or fused): row t considers positions
0 .. n_t - 1 (n_t = lengths[t] clamped to [0, S], or S when no lengths are given); they are
ordered by descending score, equal scores by ascending position (-0.0 and +0.0 are equal); the
first min(K, n_t) positions are the row's result, followed by -1 up to width K. Scores are
finite or +-inf; NaN is outside the contract.

Only ``tests/`` imports this module.
"""
from __future__ import annotations

import numpy as np


def order_keys(scores) -> np.ndarray:
    """int64 keys with the order of the float32 values (a < b iff key(a) < key(b); -0 == +0)."""
    bits = np.ascontiguousarray(scores, dtype=np.float32).view(np.int32).astype(np.int64)
    bits = np.where(bits == -(1 << 31), 0, bits)  # -0.0 -> +0.0
    # non-negative floats order as their bit patterns; negative ones in reverse
    return np.where(bits >= 0, bits, -(bits & 0x7FFFFFFF))


def topk_select(scores, K: int, lengths=None) -> np.ndarray:
    """int32 [T, K]: per row, the positions of its K largest scores (ties: lower position
    first), in that order, then -1."""
    scores = np.asarray(scores, dtype=np.float32)
    if scores.ndim != 2:
        raise ValueError("scores must be [T, S]")
    T, S = scores.shape
    out = np.full((T, K), -1, dtype=np.int32)
    for t in range(T):
        n = S if lengths is None else int(min(max(int(lengths[t]), 0), S))
        if n == 0:
            continue
        keys = order_keys(scores[t, :n])
        pos = np.arange(n, dtype=np.int64)
        # lexsort: the last key is the primary one -> descending score, then ascending position
        order = np.lexsort((pos, -keys))
        take = min(K, n)
        out[t, :take] = order[:take].astype(np.int32)
    return out
