"""CPU oracle for DSA sparse MLA attention (test infrastructure only).

This package is the correctness reference that the CUDA library is checked against. Only
``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference arms import
it; the product path (``dsa_sparse_attention_mla_gb300``) never does, and the two share no code.

The arithmetic lives in ``dsa_oracle.c`` (plain C, fp64 attention, OpenMP over tokens); this
module compiles it with gcc on first use and exposes numpy-facing wrappers. Every wrapper takes
and returns raw bit patterns (bf16 as ``uint16``, packed rows as ``uint8``) so that the exact
bytes handed to the GPU are the bytes the oracle reads.

Sources (sglang PR #38547 "Enable zero-RoPE TileLang DSA on gfx950"): the Contract table (packed
row of 264 / 656 bytes; paged dequant/gather), the Scope list (quant_k_cache, dequant_k_cache)
and the Direct GLM geometry coverage list (the step-by-step reference attention its tests use).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dsa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

CACHE_BF16 = 0
CACHE_FP8_SCALED = 1


def build(force: bool = False) -> str:
    """Compile dsa_oracle.c into oracle/liboracle.so (gcc, OpenMP, no fast-math)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
           "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i64, i32, f64 = ctypes.c_int64, ctypes.c_int, ctypes.c_double
        lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_value.restype = f64
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_float_to_bf16.argtypes = [ctypes.c_float]
        lib.oracle_float_to_bf16.restype = ctypes.c_uint16
        lib.oracle_packed_row_bytes.argtypes = [i32, i32]
        lib.oracle_packed_row_bytes.restype = i64
        lib.oracle_quant_k_cache.argtypes = [P, i64, P, i64, i64, i32, i32, P, P, i64, i32]
        lib.oracle_quant_k_cache.restype = i64
        lib.oracle_gather_dequant.argtypes = [P, i32, i64, i32, i32, P, i64, P, i64, i32, i32, P, P]
        lib.oracle_gather_dequant.restype = i64
        lib.oracle_sparse_attn.argtypes = [P, i64, i64, i32, P, i32, i64, i32, i32, i32, P, i64, i32,
                                           P, i64, i32, i32, P, f64, P, i64, P, P, i32]
        lib.oracle_sparse_attn.restype = i64
        lib.oracle_max_threads.argtypes = []
        lib.oracle_max_threads.restype = i32
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    """Contiguous numpy view with the given dtype (no value conversion for bit patterns)."""
    if a is None:
        return None
    a = np.asarray(a)
    if a.dtype != dtype:
        a = a.astype(dtype)
    return np.ascontiguousarray(a)


def max_threads() -> int:
    return int(_load().oracle_max_threads())


# ------------------------------------------------------------------------------ e4m3 / bf16 --
def e4m3_value(code: int) -> float:
    """Value of one OCP E4M3FN code (NaN for 0x7F / 0xFF)."""
    return float(_load().oracle_e4m3_value(int(code) & 0xFF))


def e4m3_encode(x: float) -> int:
    """Nearest e4m3 code to a float32 value, ties to even, saturating at +-448."""
    return int(_load().oracle_e4m3_encode(float(np.float32(x))))


def e4m3_encode_array(x) -> np.ndarray:
    lib = _load()
    x = np.asarray(x, dtype=np.float32).ravel()
    return np.fromiter((lib.oracle_e4m3_encode(float(v)) for v in x), dtype=np.uint8, count=x.size)


def float_to_bf16(x: float) -> int:
    return int(_load().oracle_float_to_bf16(float(np.float32(x))))


def packed_row_bytes(d_nope: int, d_rope: int) -> int:
    return int(_load().oracle_packed_row_bytes(d_nope, d_rope))


# ----------------------------------------------------------------------------------- pack --
def quant_k_cache(k_nope_bits, k_rope_bits=None, *, out_loc=None, cache=None, num_slots=None,
                  n_threads: int = 0):
    """Pack bf16 latent rows (uint16 bits, [n, d_nope] and [n, d_rope]) into scaled-FP8 rows.

    Returns the uint8 cache [num_slots, row_bytes] (a new zero cache unless one is given).
    """
    k_nope = _c(k_nope_bits, np.uint16)
    n, d_nope = k_nope.shape
    if k_rope_bits is None or np.asarray(k_rope_bits).size == 0:
        k_rope, d_rope = None, 0
    else:
        k_rope = _c(k_rope_bits, np.uint16)
        d_rope = k_rope.shape[1]
    rb = packed_row_bytes(d_nope, d_rope)
    if num_slots is None:
        num_slots = n if cache is None else cache.shape[0]
    if cache is None:
        cache = np.zeros((num_slots, rb), dtype=np.uint8)
    assert cache.dtype == np.uint8 and cache.shape == (num_slots, rb) and cache.flags.c_contiguous
    loc = _c(out_loc, np.int64)
    bad = _load().oracle_quant_k_cache(_ptr(k_nope), d_nope, _ptr(k_rope), d_rope, n, d_nope, d_rope,
                                       _ptr(loc), _ptr(cache), num_slots, n_threads)
    if bad:
        raise ValueError(f"{bad} rows had a destination slot outside [0, {num_slots})")
    return cache


# ------------------------------------------------------------------------------ gather/dequant --
def gather_dequant(cache, kind: int, d_nope: int, d_rope: int, indices, *, block_table=None,
                   page_size: int = 0, req_of_index=None):
    """bf16 bits [n, d_nope + d_rope] for each index (zero row for masked entries)."""
    cache = np.ascontiguousarray(cache)
    num_slots = cache.shape[0]
    idx = _c(indices, np.int32)
    n = idx.size
    bt = _c(block_table, np.int32)
    req = _c(req_of_index, np.int32)
    out = np.zeros((n, d_nope + d_rope), dtype=np.uint16)
    bad = _load().oracle_gather_dequant(_ptr(cache), kind, num_slots, d_nope, d_rope, _ptr(idx), n,
                                        _ptr(bt), 0 if bt is None else bt.shape[1], page_size,
                                        0 if bt is None else bt.shape[1], _ptr(req), _ptr(out))
    return out, int(bad)


# ------------------------------------------------------------------------- gather/requant --
def gather_requant(cache, d_nope: int, d_rope: int, indices, *, block_table=None, page_size: int = 0,
                   req_of_index=None, out_loc=None, out=None, out_slots=None):
    """Packed rows gathered by index and packed again: by definition the pack of the bf16 rows the
    gather/dequant path returns (PR #38547, production-file list: dequant_k_cache's direct, paged
    and gather/dequant/requant paths). A masked or out-of-range index gives the zero row, whose
    pack is all-zero codes and scales.

    Returns (uint8 [n or out_slots, row_bytes], number of indices that addressed no slot)."""
    deq, bad = gather_dequant(cache, CACHE_FP8_SCALED, d_nope, d_rope, indices, block_table=block_table,
                              page_size=page_size, req_of_index=req_of_index)
    n = deq.shape[0]
    if out is None:
        out_slots = n if out_loc is None else int(out_slots)
        out = np.zeros((out_slots, packed_row_bytes(d_nope, d_rope)), dtype=np.uint8)
    out = quant_k_cache(deq[:, :d_nope], deq[:, d_nope:] if d_rope else None, out_loc=out_loc, cache=out,
                        num_slots=out.shape[0])
    return out, bad


# ----------------------------------------------------------------------------------- attention --
def sparse_attn(q_bits, cache, kind: int, d_nope: int, d_rope: int, d_v: int, indices, sm_scale: float,
                *, block_table=None, page_size: int = 0, req_of_token=None, tokens=None,
                n_threads: int = 0):
    """fp64 sparse attention for the requested tokens.

    q_bits: uint16 bf16 bits [T, H, d_nope + d_rope]; cache: uint8 packed rows [slots, row_bytes]
    (kind 1) or uint16 bf16 bits [slots, d_nope + d_rope] (kind 0); indices: int32 [T, topk].
    Returns (out [n_tokens, H, d_v] float64, lse [n_tokens, H] float64, n_out_of_range).
    """
    q = _c(q_bits, np.uint16)
    T, H, D = q.shape
    assert D == d_nope + d_rope
    cache = np.ascontiguousarray(cache)
    num_slots = cache.shape[0]
    idx = _c(indices, np.int32)
    topk = idx.shape[1]
    bt = _c(block_table, np.int32)
    req = _c(req_of_token, np.int32)
    tok = None if tokens is None else _c(tokens, np.int64)
    n_tokens = T if tok is None else tok.size
    out = np.zeros((n_tokens, H, d_v), dtype=np.float64)
    lse = np.zeros((n_tokens, H), dtype=np.float64)
    bad = _load().oracle_sparse_attn(_ptr(q), H * D, D, H, _ptr(cache), kind, num_slots, d_nope, d_rope,
                                     d_v, _ptr(idx), topk, topk, _ptr(bt),
                                     0 if bt is None else bt.shape[1], page_size,
                                     0 if bt is None else bt.shape[1], _ptr(req), float(sm_scale),
                                     _ptr(tok), n_tokens, _ptr(out), _ptr(lse), n_threads)
    return out, lse, int(bad)
