"""GB300-native DSA sparse MLA attention (sm_103a).

Thin Python binding over the C ABI of ``libdsa_gb300.so`` (declared in ``include/dsa.h``).
The functions below carry the C entry points' names and only marshal arguments: they take
torch CUDA tensors for device memory and the current torch stream, pass raw pointers and
sizes, and raise :class:`DsaError` on a non-zero status. Every step of the computation runs
in the library's CUDA kernels; there is no CPU or eager-PyTorch fallback, and a missing
library is an error.

What is computed (sglang PR #38547 "Enable zero-RoPE TileLang DSA on gfx950"): the packed
scaled-FP8 latent cache row (Contract table), quant_k_cache / dequant_k_cache (Scope list)
and the sparse attention over top-k gathered latent rows (Summary; Direct GLM geometry
coverage list).
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "DsaError", "CACHE_BF16", "CACHE_FP8_SCALED", "DEVERR_INDEX_OUT_OF_RANGE", "DEVERR_TIMEOUT",
    "DEVERR_SLOT_OUT_OF_RANGE", "library_path", "load_library", "dsa_status_string",
    "dsa_packed_row_bytes", "dsa_cache_row_bytes", "dsa_quant_k_cache", "dsa_gather_dequant", "dsa_gather_requant",
    "dsa_sparse_attn_workspace_size", "dsa_sparse_attn", "dsa_sparse_attn_static_ws", "dsa_topk_select", "DsaAttnArgs",
]

CACHE_BF16 = 0
CACHE_FP8_SCALED = 1
DEVERR_INDEX_OUT_OF_RANGE = 0x1
DEVERR_TIMEOUT = 0x2
DEVERR_SLOT_OUT_OF_RANGE = 0x4

_HERE = os.path.dirname(os.path.abspath(__file__))
_lock = threading.Lock()
_LIB = None


def library_path() -> str:
    return os.path.join(_HERE, "libdsa_gb300.so")


class DsaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {dsa_status_string(status)} (status {status})")


class DsaAttnArgs(ctypes.Structure):
    """ctypes mirror of ``dsa_attn_args_t``."""

    _fields_ = [
        ("q", ctypes.c_void_p), ("q_stride_t", ctypes.c_int64), ("q_stride_h", ctypes.c_int64),
        ("T", ctypes.c_int64), ("H", ctypes.c_int),
        ("cache", ctypes.c_void_p), ("kind", ctypes.c_int), ("num_slots", ctypes.c_int64),
        ("d_nope", ctypes.c_int), ("d_rope", ctypes.c_int), ("d_v", ctypes.c_int),
        ("indices", ctypes.c_void_p), ("idx_stride_t", ctypes.c_int64), ("topk", ctypes.c_int),
        ("block_table", ctypes.c_void_p), ("bt_stride", ctypes.c_int64),
        ("page_size", ctypes.c_int), ("max_pages", ctypes.c_int),
        ("req_of_token", ctypes.c_void_p), ("sm_scale", ctypes.c_float),
        ("out", ctypes.c_void_p), ("out_stride_t", ctypes.c_int64), ("out_stride_h", ctypes.c_int64),
        ("lse", ctypes.c_void_p), ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
        ("error_word", ctypes.c_void_p),
    ]


def load_library():
    """Load libdsa_gb300.so (built in-tree by ``__graft_entry__.build()``)."""
    global _LIB
    with _lock:
        if _LIB is not None:
            return _LIB
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build the CUDA library first (__graft_entry__.build())")
        lib = ctypes.CDLL(path)
        P, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        lib.dsa_status_string.argtypes = [i32]
        lib.dsa_status_string.restype = ctypes.c_char_p
        lib.dsa_last_cuda_error.argtypes = []
        lib.dsa_last_cuda_error.restype = i32
        lib.dsa_packed_row_bytes.argtypes = [i32, i32]
        lib.dsa_packed_row_bytes.restype = i64
        lib.dsa_cache_row_bytes.argtypes = [i32, i32, i32]
        lib.dsa_cache_row_bytes.restype = i64
        lib.dsa_quant_k_cache.argtypes = [P, i64, P, i64, i64, i32, i32, P, P, i64, P, P]
        lib.dsa_quant_k_cache.restype = i32
        lib.dsa_gather_dequant.argtypes = [P, i32, i64, i32, i32, P, i64, P, i64, i32, i32, P, P, P, P]
        lib.dsa_gather_dequant.restype = i32
        lib.dsa_gather_requant.argtypes = [P, i64, i32, i32, P, i64, P, i64, i32, i32, P, P, P, i64, P, P]
        lib.dsa_gather_requant.restype = i32
        lib.dsa_sparse_attn_workspace_size.argtypes = [ctypes.POINTER(DsaAttnArgs), ctypes.POINTER(ctypes.c_size_t)]
        lib.dsa_sparse_attn_workspace_size.restype = i32
        lib.dsa_sparse_attn.argtypes = [ctypes.POINTER(DsaAttnArgs), P]
        lib.dsa_sparse_attn.restype = i32
        lib.dsa_sparse_attn_static_ws.argtypes = [ctypes.POINTER(DsaAttnArgs), P]
        lib.dsa_sparse_attn_static_ws.restype = i32
        lib.dsa_topk_select.argtypes = [P, i64, i64, i64, P, i32, P, i64, P]
        lib.dsa_topk_select.restype = i32
        lib.dsa_blockscale_bytes.argtypes = [i64, i64]
        lib.dsa_blockscale_bytes.restype = i64
        lib.dsa_quant_fp8_blockscale.argtypes = [P, i64, i64, i64, i32, P, P, P]
        lib.dsa_quant_fp8_blockscale.restype = i32
        lib.dsa_proj_gemm.argtypes = [P, P, P, P, i64, i64, i64, P, i64, P, ctypes.c_size_t, P]
        lib.dsa_proj_gemm.restype = i32
        _LIB = lib
        return lib


def _check(status: int, where: str):
    if status != 0:
        raise DsaError(status, where)


def dsa_status_string(status: int) -> str:
    return load_library().dsa_status_string(int(status)).decode()


def dsa_packed_row_bytes(d_nope: int, d_rope: int) -> int:
    return int(load_library().dsa_packed_row_bytes(d_nope, d_rope))


def dsa_cache_row_bytes(kind: int, d_nope: int, d_rope: int) -> int:
    return int(load_library().dsa_cache_row_bytes(kind, d_nope, d_rope))


# ----------------------------------------------------------------------------- helpers --
def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device):
    import torch

    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _need_cuda(name, t, dtype=None):
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must have dtype {dtype}, got {t.dtype}")


# --------------------------------------------------------------------------- entry points --
def dsa_quant_k_cache(k_nope, k_rope=None, *, out_loc=None, cache=None, num_slots=None, error_word=None):
    """Pack bf16 latent rows into scaled-FP8 rows; returns the uint8 cache [num_slots, row_bytes]."""
    import torch

    _need_cuda("k_nope", k_nope, torch.bfloat16)
    _need_cuda("k_rope", k_rope, torch.bfloat16)
    _need_cuda("out_loc", out_loc, torch.int64)
    n, d_nope = k_nope.shape
    d_rope = 0 if k_rope is None or k_rope.numel() == 0 else k_rope.shape[1]
    if d_rope == 0:
        k_rope = None
    rb = dsa_packed_row_bytes(d_nope, d_rope)
    if cache is None:
        num_slots = n if num_slots is None else num_slots
        cache = torch.zeros((num_slots, rb), dtype=torch.uint8, device=k_nope.device)
    _need_cuda("cache", cache, torch.uint8)
    if num_slots is None:
        num_slots = cache.shape[0]
    if k_nope.stride(1) != 1 or (k_rope is not None and k_rope.stride(1) != 1):
        raise ValueError("rows must be contiguous along d")
    if out_loc is not None:
        out_loc = out_loc.contiguous()
    st = load_library().dsa_quant_k_cache(
        _ptr(k_nope), k_nope.stride(0), _ptr(k_rope), 0 if k_rope is None else k_rope.stride(0), n, d_nope, d_rope,
        _ptr(out_loc), _ptr(cache), num_slots, _ptr(error_word), _stream(k_nope.device))
    _check(st, "dsa_quant_k_cache")
    return cache


def dsa_gather_dequant(cache, kind: int, d_nope: int, d_rope: int, indices, *, block_table=None, page_size=0,
                       req_of_index=None, out=None, error_word=None):
    """bf16 rows [n, d_nope + d_rope] gathered (and dequantised) by index."""
    import torch

    _need_cuda("cache", cache)
    _need_cuda("indices", indices, torch.int32)
    _need_cuda("block_table", block_table, torch.int32)
    _need_cuda("req_of_index", req_of_index, torch.int32)
    indices = indices.contiguous().view(-1)
    n = indices.numel()
    if out is None:
        out = torch.empty((n, d_nope + d_rope), dtype=torch.bfloat16, device=indices.device)
    _need_cuda("out", out, torch.bfloat16)
    bt_stride = 0 if block_table is None else block_table.stride(0)
    max_pages = 0 if block_table is None else block_table.shape[1]
    st = load_library().dsa_gather_dequant(
        _ptr(cache), kind, cache.shape[0], d_nope, d_rope, _ptr(indices), n, _ptr(block_table), bt_stride, page_size,
        max_pages, _ptr(None if req_of_index is None else req_of_index.contiguous()), _ptr(out), _ptr(error_word),
        _stream(indices.device))
    _check(st, "dsa_gather_dequant")
    return out


def dsa_gather_requant(cache, d_nope: int, d_rope: int, indices, *, block_table=None, page_size=0,
                       req_of_index=None, out_loc=None, out=None, out_slots=None, error_word=None):
    """Packed rows gathered by index and packed again (uint8 [n, row_bytes], or written into
    rows out_loc of ``out``)."""
    import torch

    _need_cuda("cache", cache, torch.uint8)
    _need_cuda("indices", indices, torch.int32)
    _need_cuda("block_table", block_table, torch.int32)
    _need_cuda("req_of_index", req_of_index, torch.int32)
    _need_cuda("out_loc", out_loc, torch.int64)
    indices = indices.contiguous().view(-1)
    n = indices.numel()
    rb = dsa_packed_row_bytes(d_nope, d_rope)
    if out is None:
        out = torch.empty((n if out_loc is None else int(out_slots), rb), dtype=torch.uint8, device=indices.device)
    _need_cuda("out", out, torch.uint8)
    bt_stride = 0 if block_table is None else block_table.stride(0)
    max_pages = 0 if block_table is None else block_table.shape[1]
    st = load_library().dsa_gather_requant(
        _ptr(cache), cache.shape[0], d_nope, d_rope, _ptr(indices), n, _ptr(block_table), bt_stride, page_size,
        max_pages, _ptr(None if req_of_index is None else req_of_index.contiguous()),
        _ptr(None if out_loc is None else out_loc.contiguous()), _ptr(out), out.shape[0], _ptr(error_word),
        _stream(indices.device))
    _check(st, "dsa_gather_requant")
    return out


_WS = {}


def _workspace(device, nbytes: int):
    """The default workspace of the current stream on ``device``: one zero-filled buffer per
    (device, stream), so that calls on different streams, which may run at the same time on the
    GPU, never share one (calls on one stream run in order, so they can). The library leaves a
    workspace with no flag set after every call that completes without a timeout."""
    import torch

    index = device.index if device.index is not None else torch.cuda.current_device()
    key = (index, torch.cuda.current_stream(index).cuda_stream)
    with _lock:
        ws = _WS.get(key)
        if ws is None or ws.numel() < nbytes:
            ws = torch.zeros(nbytes, dtype=torch.uint8, device=torch.device("cuda", index))
            _WS[key] = ws
    return ws


def _attn_args(q, cache, kind, indices, sm_scale, d_nope, d_rope, d_v, block_table, page_size, req_of_token, out,
               lse, workspace, error_word) -> DsaAttnArgs:
    a = DsaAttnArgs()
    T, H, D = q.shape
    a.q = q.data_ptr()
    a.q_stride_t, a.q_stride_h = q.stride(0), q.stride(1)
    a.T, a.H = T, H
    a.cache = cache.data_ptr()
    a.kind = kind
    a.num_slots = cache.shape[0]
    a.d_nope, a.d_rope, a.d_v = d_nope, d_rope, d_v
    a.indices = indices.data_ptr()
    a.idx_stride_t = indices.stride(0)
    a.topk = indices.shape[1]
    if block_table is not None:
        a.block_table = block_table.data_ptr()
        a.bt_stride = block_table.stride(0)
        a.page_size = page_size
        a.max_pages = block_table.shape[1]
    if req_of_token is not None:
        a.req_of_token = req_of_token.data_ptr()
    a.sm_scale = float(sm_scale)
    a.out = out.data_ptr()
    a.out_stride_t, a.out_stride_h = out.stride(0), out.stride(1)
    if lse is not None:
        a.lse = lse.data_ptr()
    if workspace is not None:
        a.workspace = workspace.data_ptr()
        a.workspace_bytes = workspace.numel() * workspace.element_size()
    if error_word is not None:
        a.error_word = error_word.data_ptr()
    return a


def dsa_sparse_attn_workspace_size(d_v: int = 256) -> int:
    """Workspace bytes dsa_sparse_attn needs on the current device."""
    a = DsaAttnArgs()
    a.H, a.d_v = 64, d_v
    n = ctypes.c_size_t(0)
    _check(load_library().dsa_sparse_attn_workspace_size(ctypes.byref(a), ctypes.byref(n)),
           "dsa_sparse_attn_workspace_size")
    return int(n.value)


def _check_attn_inputs(q, cache, kind, indices, block_table, req_of_token, out, lse, error_word):
    import torch

    _need_cuda("q", q, torch.bfloat16)
    _need_cuda("cache", cache, torch.uint8 if kind == CACHE_FP8_SCALED else torch.bfloat16)
    _need_cuda("indices", indices, torch.int32)
    _need_cuda("block_table", block_table, torch.int32)
    _need_cuda("req_of_token", req_of_token, torch.int32)
    _need_cuda("out", out, torch.bfloat16)
    _need_cuda("lse", lse, torch.float32)
    _need_cuda("error_word", error_word, torch.int32)
    for name, t in (("cache", cache), ("indices", indices), ("block_table", block_table),
                    ("req_of_token", req_of_token), ("out", out), ("lse", lse), ("error_word", error_word)):
        if t is not None and t.device != q.device:
            raise ValueError(f"{name} is on {t.device}, q on {q.device}: every tensor must be on one device")
    if q.dim() != 3 or indices.dim() != 2:
        raise ValueError("q must be [T, H, D] and indices [T, topk]")
    if q.stride(2) != 1 or indices.stride(1) != 1:
        raise ValueError("q and indices must be contiguous along their last dimension")
    if req_of_token is not None and not req_of_token.is_contiguous():
        raise ValueError("req_of_token must be contiguous")
    if lse is not None and not lse.is_contiguous():
        raise ValueError("lse must be a contiguous [T, H] tensor")


def _prepare_attn(q, cache, kind, indices, d_v, block_table, req_of_token, out, lse, error_word):
    import torch

    if kind == CACHE_BF16 and cache.dim() == 3:
        cache = cache.view(cache.shape[0], -1)
    if out is None:
        out = torch.empty((q.shape[0], q.shape[1], d_v), dtype=torch.bfloat16, device=q.device)
    _check_attn_inputs(q, cache, kind, indices, block_table, req_of_token, out, lse, error_word)
    return cache, out


def dsa_sparse_attn(q, cache, kind: int, indices, sm_scale: float, *, d_nope: int = 256, d_rope: int = 0,
                    d_v: int = None, block_table=None, page_size: int = 0, req_of_token=None, out=None, lse=None,
                    workspace=None, error_word=None):
    """Sparse MLA attention: out[t, h] = softmax_j(sm_scale * q[t,h].k_j) @ k_j[:d_v] over valid indices.

    Without ``workspace`` the call takes the default workspace of the current stream (one per
    device and stream)."""
    import torch

    d_v = d_nope if d_v is None else d_v
    cache, out = _prepare_attn(q, cache, kind, indices, d_v, block_table, req_of_token, out, lse, error_word)
    if workspace is None:
        workspace = _workspace(q.device, dsa_sparse_attn_workspace_size(d_v))
    _need_cuda("workspace", workspace, torch.uint8)
    a = _attn_args(q, cache, kind, indices, sm_scale, d_nope, d_rope, d_v, block_table, page_size, req_of_token,
                   out, lse, workspace, error_word)
    _check(load_library().dsa_sparse_attn(ctypes.byref(a), _stream(q.device)), "dsa_sparse_attn")
    return out


def dsa_sparse_attn_static_ws(q, cache, kind: int, indices, sm_scale: float, *, d_nope: int = 256, d_rope: int = 0,
                              d_v: int = None, block_table=None, page_size: int = 0, req_of_token=None, out=None,
                              lse=None, error_word=None):
    """dsa_sparse_attn without a workspace: the library's fixed device scratch is used, so the
    call allocates no device memory (``out`` aside, when the caller passes none). For callers
    that cannot allocate device memory when they call; the first call on a device does one-time
    set-up. Calls whose kernels may overlap on the GPU share the one scratch array and race on it."""
    d_v = d_nope if d_v is None else d_v
    cache, out = _prepare_attn(q, cache, kind, indices, d_v, block_table, req_of_token, out, lse, error_word)
    a = _attn_args(q, cache, kind, indices, sm_scale, d_nope, d_rope, d_v, block_table, page_size, req_of_token,
                   out, lse, None, error_word)
    _check(load_library().dsa_sparse_attn_static_ws(ctypes.byref(a), _stream(q.device)), "dsa_sparse_attn_static_ws")
    return out


def dsa_topk_select(scores, K: int, *, lengths=None, out=None):
    """int32 [T, K]: per row, the positions of its K largest scores (ties: lower position first),
    in that order, then -1 (positions at or past lengths[t] are not considered)."""
    import torch

    _need_cuda("scores", scores, torch.float32)
    _need_cuda("lengths", lengths, torch.int32)
    if scores.dim() != 2 or scores.stride(1) != 1:
        raise ValueError("scores must be [T, S], contiguous along S")
    T, S = scores.shape
    if out is None:
        out = torch.empty((T, K), dtype=torch.int32, device=scores.device)
    _need_cuda("out", out, torch.int32)
    if out.dim() != 2 or out.shape[0] != T or out.shape[1] < K or out.stride(1) != 1:
        raise ValueError("out must be [T, >=K] int32, contiguous along its last dimension")
    if lengths is not None:
        lengths = lengths.contiguous()
        if lengths.numel() != T:
            raise ValueError("lengths must have one entry per row")
    st = load_library().dsa_topk_select(_ptr(scores), T, S, scores.stride(0), _ptr(lengths), int(K), _ptr(out),
                                        out.stride(0), _stream(scores.device))
    _check(st, "dsa_topk_select")
    return out


def dsa_blockscale_bytes(rows: int, cols: int) -> int:
    return int(load_library().dsa_blockscale_bytes(rows, cols))


def dsa_quant_fp8_blockscale(x, block_rows: int, *, codes=None, scales=None):
    """(codes uint8 [R, C], scales uint8 [dsa_blockscale_bytes(R, C)]) of bf16 x [R, C]: e4m3 codes
    with one power-of-two scale per block_rows x 128 block (128: weights, 1: activations), the
    scales in the projection GEMM's block-scale layout."""
    import torch

    _need_cuda("x", x, torch.bfloat16)
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be [rows, cols], contiguous along cols")
    R, C = x.shape
    nb = dsa_blockscale_bytes(R, C)
    if nb < 0:
        raise ValueError("cols must be a positive multiple of 128")
    if codes is None:
        codes = torch.empty((R, C), dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty(nb, dtype=torch.uint8, device=x.device)
    _need_cuda("codes", codes, torch.uint8)
    _need_cuda("scales", scales, torch.uint8)
    if tuple(codes.shape) != (R, C) or not codes.is_contiguous() or scales.numel() < nb or not scales.is_contiguous():
        raise ValueError("codes must be contiguous [rows, cols] and scales hold dsa_blockscale_bytes(rows, cols)")
    st = load_library().dsa_quant_fp8_blockscale(_ptr(x), R, C, x.stride(0), int(block_rows), _ptr(codes), _ptr(scales),
                                                 _stream(x.device))
    _check(st, "dsa_quant_fp8_blockscale")
    return codes, scales


_GEMM_WS = {}


def _gemm_workspace(device, nbytes: int = 32 << 20):
    """The GEMM's scratch for the current stream on ``device`` (its own buffer: the attention's
    default workspace must keep its flags)."""
    import torch

    index = device.index if device.index is not None else torch.cuda.current_device()
    key = (index, torch.cuda.current_stream(index).cuda_stream)
    with _lock:
        ws = _GEMM_WS.get(key)
        if ws is None:
            ws = torch.empty(nbytes, dtype=torch.uint8, device=torch.device("cuda", index))
            _GEMM_WS[key] = ws
    return ws


def dsa_proj_gemm(x_codes, x_scales, w_codes, w_scales, *, out=None, workspace=None):
    """bf16 [M, N] = X W^T over block-scaled FP8 operands (x from block_rows=1 [M, K], w from
    block_rows=128 [N, K])."""
    import torch

    for name, t in (("x_codes", x_codes), ("x_scales", x_scales), ("w_codes", w_codes), ("w_scales", w_scales)):
        _need_cuda(name, t, torch.uint8)
    M, K = x_codes.shape
    N, K2 = w_codes.shape
    if K2 != K:
        raise ValueError("x and w must share K")
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=x_codes.device)
    _need_cuda("out", out, torch.bfloat16)
    if out.dim() != 2 or tuple(out.shape) != (M, N) or out.stride(1) != 1:
        raise ValueError("out must be [M, N] bf16, contiguous along N")
    if workspace is None:
        workspace = _gemm_workspace(x_codes.device)
    _need_cuda("workspace", workspace, torch.uint8)
    st = load_library().dsa_proj_gemm(_ptr(x_codes), _ptr(x_scales), _ptr(w_codes), _ptr(w_scales), M, N, K, _ptr(out),
                                      out.stride(0), _ptr(workspace), workspace.numel(), _stream(x_codes.device))
    _check(st, "dsa_proj_gemm")
    return out
