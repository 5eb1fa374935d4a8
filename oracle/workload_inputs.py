"""Host-side oracle inputs for the seeded workloads (test infrastructure only).

Builds, with the oracle's own pack, the cache bytes a workload's tokens read, so that the
parity tests and the benchmark's CPU baseline run the oracle on inputs that never come from
the CUDA path. Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference arms use it.
"""
from __future__ import annotations

import numpy as np

from . import CACHE_BF16, packed_row_bytes, quant_k_cache


def oracle_cache(wl, rows=None):
    """Host cache bytes for a workload, built by the oracle (uint8 rows for FP8, bf16 bits for BF16).

    ``rows``: only these kv rows are generated and written (the rest stay zero) - enough for an
    oracle run restricted to tokens whose entries name only those rows."""
    if wl.kind == CACHE_BF16:
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
    rb = packed_row_bytes(wl.d_nope, wl.d_rope)
    cache = np.zeros((wl.num_slots, rb), dtype=np.uint8)
    return quant_k_cache(src[:, : wl.d_nope], src[:, wl.d_nope:] if wl.d_rope else None,
                         out_loc=None if loc is None else np.asarray(loc, dtype=np.int64), cache=cache,
                         num_slots=wl.num_slots)


def slots_of_tokens(wl, tokens):
    """Physical slots named by the valid entries of the given tokens (page translation as the
    Contract table's paged gather defines it)."""
    idx = wl.indices[tokens].astype(np.int64)
    valid = idx >= 0
    if wl.block_table is None:
        s = idx[valid]
    else:
        r = wl.req_of_token[tokens][:, None].repeat(idx.shape[1], axis=1)[valid]
        pos = idx[valid]
        s = wl.block_table[r, pos // wl.page_size].astype(np.int64) * wl.page_size + pos % wl.page_size
    return np.unique(s)


def kv_rows_for(wl, slots):
    """kv row ids whose packed row lands in the given physical slots."""
    if wl.kv_slot is None:
        return slots
    inv = np.empty(wl.num_slots, dtype=np.int64)
    inv[wl.kv_slot] = np.arange(wl.num_slots)
    return inv[slots]


def cache_for_tokens(wl, tokens):
    """The oracle's cache with only the rows the given tokens read (the rest zero)."""
    return oracle_cache(wl, rows=kv_rows_for(wl, slots_of_tokens(wl, tokens)))
