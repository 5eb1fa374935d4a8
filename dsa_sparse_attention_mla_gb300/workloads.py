"""Seeded synthetic inputs for DSA sparse MLA attention.

This module only draws random numbers: it holds none of the method's arithmetic (no packing,
no dequantisation, no attention). Both the CUDA path (tests, bench) and the CPU oracle consume
the arrays it returns, so the two sides always see the same bytes.

Normal tensors use a counter-based generator so any row range can be regenerated anywhere:
element e of stream (seed, stream) takes 16 bits of ``hash32(key ^ (e // 2))`` (low half for
even e, high half for odd e) and maps them through a fixed table of standard-normal quantiles
``ndtri((u + 0.5) / 65536)`` held as float32, then rounds to bf16 (nearest-even). The numpy
and torch implementations below are integer-exact, so the CPU and the GPU produce identical
bits for the same elements. Index lists and page tables use ``numpy.random.default_rng``.

The five named workloads follow the synthetic shapes of the geometry coverage list of sglang
PR #38547 (Q [tokens, 64, 256], KV [slots, 1, 256], top-k 2048 / 2112, -1 padding, 264-byte and
656-byte packed rows, paged gathers).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np

MASK32 = 0xFFFFFFFF
_MIX = 0x45D9F3B  # multiplier of the integer mixing function (fits in 31 bits: exact in int64)

_TABLE_NP: Optional[np.ndarray] = None
_TABLE_T = {}


def _quantile_table_np() -> np.ndarray:
    global _TABLE_NP
    if _TABLE_NP is None:
        import torch

        u = torch.arange(65536, dtype=torch.float64)
        _TABLE_NP = torch.special.ndtri((u + 0.5) / 65536.0).to(torch.float32).numpy().copy()
    return _TABLE_NP


def _stream_key(seed: int, stream: int) -> int:
    x = (seed * 0x9E3779B1 + stream * 0x85EBCA77 + 0x27D4EB2F) & MASK32
    for _ in range(2):
        x = (((x >> 16) ^ x) * _MIX) & MASK32
    return ((x >> 16) ^ x) & MASK32


def _hash32_np(x: np.ndarray) -> np.ndarray:
    x = (((x >> np.uint64(16)) ^ x) * np.uint64(_MIX)) & np.uint64(MASK32)
    x = (((x >> np.uint64(16)) ^ x) * np.uint64(_MIX)) & np.uint64(MASK32)
    return (x >> np.uint64(16)) ^ x


def normal_bf16_at(seed: int, stream: int, elems) -> np.ndarray:
    """bf16 bit patterns (numpy uint16) of the given element numbers of a normal stream."""
    import torch

    e = np.asarray(elems, dtype=np.uint64)
    h = _hash32_np((e >> np.uint64(1)) ^ np.uint64(_stream_key(seed, stream)))
    u = np.where((e & np.uint64(1)) == 0, h & np.uint64(0xFFFF), h >> np.uint64(16)).astype(np.int64)
    vals = np.ascontiguousarray(_quantile_table_np()[u].reshape(-1))
    bits = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    return bits.reshape(e.shape)


def normal_bf16_bits(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Elements [start, start + count) of a normal stream as bf16 bit patterns (numpy uint16)."""
    return normal_bf16_at(seed, stream, np.arange(start, start + count, dtype=np.uint64))


def normal_bf16_torch(seed: int, stream: int, start: int, count: int, device, chunk: int = 1 << 26):
    """Same elements as :func:`normal_bf16_bits`, produced on ``device`` as a bf16 tensor."""
    import torch

    dev = torch.device(device)
    if dev not in _TABLE_T:
        _TABLE_T[dev] = torch.from_numpy(_quantile_table_np()).to(dev)
    table = _TABLE_T[dev]
    key = _stream_key(seed, stream)
    out = torch.empty(count, dtype=torch.bfloat16, device=dev)
    pos = 0
    while pos < count:
        n = min(chunk, count - pos)
        s = start + pos
        c0, c1 = s // 2, (s + n + 1) // 2
        x = torch.arange(c0, c1, dtype=torch.int64, device=dev) ^ key
        x = (((x >> 16) ^ x) * _MIX) & MASK32
        x = (((x >> 16) ^ x) * _MIX) & MASK32
        x = (x >> 16) ^ x
        u = torch.stack((x & 0xFFFF, x >> 16), dim=1).reshape(-1)
        u = u[s - 2 * c0: s - 2 * c0 + n]
        out[pos: pos + n] = table[u].to(torch.bfloat16)
        pos += n
    return out


@dataclass
class NormalRows:
    """A [rows, cols] bf16 matrix of the counter-based normal stream (seed, stream)."""

    seed: int
    stream: int
    rows: int
    cols: int

    def bits(self, row_ids=None) -> np.ndarray:
        """uint16 bf16 bits for the given rows (all rows when None)."""
        if row_ids is None:
            return normal_bf16_bits(self.seed, self.stream, 0, self.rows * self.cols).reshape(self.rows, self.cols)
        row_ids = np.asarray(row_ids, dtype=np.uint64).ravel()
        elems = row_ids[:, None] * np.uint64(self.cols) + np.arange(self.cols, dtype=np.uint64)[None, :]
        return normal_bf16_at(self.seed, self.stream, elems)

    def torch(self, device):
        return normal_bf16_torch(self.seed, self.stream, 0, self.rows * self.cols, device).view(self.rows, self.cols)


@dataclass
class FixedRows:
    """Explicit bf16 rows (uint16 bits [rows, cols]) with the interface of NormalRows."""

    data: np.ndarray

    @property
    def rows(self) -> int:
        return int(self.data.shape[0])

    @property
    def cols(self) -> int:
        return int(self.data.shape[1])

    def bits(self, row_ids=None) -> np.ndarray:
        if row_ids is None:
            return self.data
        return self.data[np.asarray(row_ids, dtype=np.int64).ravel()]

    def torch(self, device):
        import torch
        return torch.from_numpy(np.ascontiguousarray(self.data).view(np.int16)).view(torch.bfloat16).to(device)


@dataclass
class Workload:
    """One synthetic sparse-attention problem.

    kind 0: BF16 latent cache [num_slots, d_nope + d_rope] = ``kv`` itself.
    kind 1: packed scaled-FP8 cache built from ``kv`` row i into slot ``kv_slot[i]`` (or slot i).
    Paged mode when ``block_table`` is set: indices are logical positions of request
    ``req_of_token[t]``.
    """

    name: str
    kind: int
    d_nope: int
    d_rope: int
    d_v: int
    q: "NormalRows | FixedRows"        # [T*H, D] rows of the query (reshaped to [T, H, D])
    T: int
    H: int
    kv: "NormalRows | FixedRows"       # [num_slots, D] latent rows (slot order)
    num_slots: int
    indices: np.ndarray                # int32 [T, topk]
    sm_scale: float
    block_table: Optional[np.ndarray] = None   # int32 [R, max_pages]
    page_size: int = 0
    req_of_token: Optional[np.ndarray] = None  # int32 [T]
    kv_slot: Optional[np.ndarray] = None       # int64 [num_slots] slot of kv row i (None: identity)
    notes: dict = field(default_factory=dict)

    @property
    def D(self) -> int:
        return self.d_nope + self.d_rope

    @property
    def topk(self) -> int:
        return int(self.indices.shape[1])

    def q_bits(self) -> np.ndarray:
        return self.q.bits().reshape(self.T, self.H, self.D)

    def n_valid(self) -> int:
        return int((self.indices >= 0).sum())


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.default_rng([seed, stream])


def _pad(rows, width: int, rng: Optional[np.random.Generator] = None, scatter=None) -> np.ndarray:
    """Stack per-token valid lists into [T, width] with -1 padding (tail, or scattered for the
    tokens listed in ``scatter``)."""
    out = np.full((len(rows), width), -1, dtype=np.int32)
    scatter = set() if scatter is None else set(int(s) for s in scatter)
    for t, r in enumerate(rows):
        r = np.asarray(r, dtype=np.int32)
        if t in scatter:
            pos = np.sort(rng.choice(width, size=r.size, replace=False))
            out[t, pos] = r
        else:
            out[t, : r.size] = r
    return out


def bf16_direct(T=17, slots=8192, topk=2112, n_valid=2051, H=64, d_nope=256, d_rope=0, d_v=None,
                sm_scale=None, seed=0, scatter_frac=0.0, name="bf16_direct") -> Workload:
    """BF16 direct cache: each token draws n_valid distinct slots uniformly, random order, -1 pad."""
    D = d_nope + d_rope
    d_v = d_nope if d_v is None else d_v
    rng = _rng(seed, 1)
    n_valid = min(n_valid, slots)
    rows = [rng.choice(slots, size=n_valid, replace=False) for _ in range(T)]
    scatter = rng.choice(T, size=int(round(scatter_frac * T)), replace=False) if scatter_frac else None
    idx = _pad(rows, topk, rng, scatter)
    return Workload(name=name, kind=0, d_nope=d_nope, d_rope=d_rope, d_v=d_v,
                    q=NormalRows(seed, 10, T * H, D), T=T, H=H, kv=NormalRows(seed, 11, slots, D),
                    num_slots=slots, indices=idx,
                    sm_scale=(1.0 / np.sqrt(D)) if sm_scale is None else sm_scale)


def fp8_paged(T=8, requests=1, positions=16384, page_size=64, topk=2048, n_valid=2048, H=64,
              d_nope=256, d_rope=0, d_v=None, sm_scale=None, seed=0, recent=0, recent_frac=0.0,
              scatter_frac=0.0, scatter_kv=True, name="fp8_paged") -> Workload:
    """Packed FP8 cache in a paged pool; every request owns positions//page_size random pages.

    Token t belongs to request t % requests. Its n_valid logical positions are drawn without
    replacement: round(recent_frac * n_valid) from the last ``recent`` positions and the rest from
    the positions before them (plain uniform draws when recent_frac == 0).
    """
    D = d_nope + d_rope
    d_v = d_nope if d_v is None else d_v
    assert positions % page_size == 0
    pages_per_req = positions // page_size
    n_pages = requests * pages_per_req
    num_slots = n_pages * page_size
    rng = _rng(seed, 2)
    perm = rng.permutation(n_pages).astype(np.int32)
    block_table = perm.reshape(requests, pages_per_req)
    req = (np.arange(T) % requests).astype(np.int32)
    rows = []
    for t in range(T):
        if recent_frac > 0:
            n_recent = int(round(recent_frac * n_valid))
            a = positions - recent + rng.choice(recent, size=n_recent, replace=False)
            b = rng.choice(positions - recent, size=n_valid - n_recent, replace=False)
            r = np.concatenate([a, b])
            rng.shuffle(r)
        else:
            r = rng.choice(positions, size=n_valid, replace=False)
        rows.append(r)
    scatter = rng.choice(T, size=int(round(scatter_frac * T)), replace=False) if scatter_frac else None
    idx = _pad(rows, topk, rng, scatter)
    kv_slot = None
    if scatter_kv:
        # kv row i is the latent of logical position i % positions of request i // positions,
        # written to its physical slot (the KV write path with out_loc)
        i = np.arange(num_slots, dtype=np.int64)
        r_i, p_i = i // positions, i % positions
        kv_slot = block_table[r_i, p_i // page_size].astype(np.int64) * page_size + p_i % page_size
    return Workload(name=name, kind=1, d_nope=d_nope, d_rope=d_rope, d_v=d_v,
                    q=NormalRows(seed, 20, T * H, D), T=T, H=H, kv=NormalRows(seed, 21, num_slots, D),
                    num_slots=num_slots, indices=idx,
                    sm_scale=(1.0 / np.sqrt(D)) if sm_scale is None else sm_scale,
                    block_table=block_table, page_size=page_size, req_of_token=req, kv_slot=kv_slot)


def fp8_direct(T=1024, slots=65536, topk=2048, n_valid=2048, H=64, d_nope=512, d_rope=64, d_v=512,
               sm_scale=None, seed=0, name="fp8_direct") -> Workload:
    D = d_nope + d_rope
    rng = _rng(seed, 3)
    rows = [rng.choice(slots, size=min(n_valid, slots), replace=False) for _ in range(T)]
    idx = _pad(rows, topk)
    return Workload(name=name, kind=1, d_nope=d_nope, d_rope=d_rope, d_v=d_v,
                    q=NormalRows(seed, 30, T * H, D), T=T, H=H, kv=NormalRows(seed, 31, slots, D),
                    num_slots=slots, indices=idx,
                    sm_scale=(1.0 / np.sqrt(D)) if sm_scale is None else sm_scale)


def prefill_causal(T=8192, topk=2048, window=128, H=64, d_nope=256, seed=0, name="prefill_causal") -> Workload:
    """One sequence of T tokens over a BF16 cache of T slots. Token t < topk takes all of [0, t];
    later tokens take [t-window+1, t] plus topk-window draws without replacement from
    [0, t-window]. Valid entries in random order, -1 tail."""
    rng = _rng(seed, 4)
    idx = np.full((T, topk), -1, dtype=np.int32)
    for t in range(T):
        if t + 1 <= topk:
            r = np.arange(t + 1, dtype=np.int64)
        else:
            r = np.concatenate([np.arange(t - window + 1, t + 1),
                                rng.choice(t - window + 1, size=topk - window, replace=False)])
        rng.shuffle(r)
        idx[t, : r.size] = r
    D = d_nope
    return Workload(name=name, kind=0, d_nope=d_nope, d_rope=0, d_v=d_nope,
                    q=NormalRows(seed, 40, T * H, D), T=T, H=H, kv=NormalRows(seed, 41, T, D),
                    num_slots=T, indices=idx, sm_scale=1.0 / 16.0)


# --------------------------------------------------------------------------- named workloads --
def config(n: int, seed: int = 0) -> Workload:
    """The five named workloads (1-based)."""
    if n == 1:   # BF16 direct 256+0, T=17, 2051 valid of 2112
        return bf16_direct(T=17, slots=8192, topk=2112, n_valid=2051, seed=seed, sm_scale=1 / 16,
                           name="bf16_direct_T17_k2112")
    if n == 2:   # FP8 256+0 paged, T=8, top-k 2048 all valid over 16384 positions
        return fp8_paged(T=8, requests=1, positions=16384, page_size=64, topk=2048, n_valid=2048,
                         seed=seed, sm_scale=1 / 16, name="fp8_paged_T8_k2048")
    if n == 3:   # batched decode: 256 requests x 32768 positions, 70/30 recent/uniform, 5% scattered pads
        return fp8_paged(T=256, requests=256, positions=32768, page_size=64, topk=2112, n_valid=2048,
                         recent=4096, recent_frac=0.7, scatter_frac=0.05, scatter_kv=False,
                         seed=seed, sm_scale=1 / 16, name="fp8_paged_decode_T256_k2112")
    if n == 4:   # prefill, BF16 cache, T=8192 causal top-2048
        return prefill_causal(T=8192, topk=2048, window=128, seed=seed, name="bf16_prefill_T8192_k2048")
    if n == 5:   # 512+64 control, FP8 656-byte rows
        return fp8_direct(T=1024, slots=65536, topk=2048, n_valid=2048, d_nope=512, d_rope=64, d_v=512,
                          seed=seed, sm_scale=1 / 24, name="fp8_512p64_T1024_k2048")
    raise ValueError(n)
