"""The C ABI library loads, exports every entry point include/dsa.h declares, lays out its
argument struct as the header says, and rejects bad arguments before touching the GPU."""
import ctypes
import os
import re
import subprocess


import dsa_sparse_attention_mla_gb300 as dsa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dsa.h")


def _declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"DSA_API\s+[\w\s\*]+?\b(dsa_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = _declared()
    for n in ["dsa_quant_k_cache", "dsa_gather_dequant", "dsa_gather_requant", "dsa_sparse_attn", "dsa_sparse_attn_workspace_size",
              "dsa_topk_select", "dsa_quant_fp8_blockscale", "dsa_proj_gemm", "dsa_blockscale_bytes",
              "dsa_packed_row_bytes", "dsa_cache_row_bytes", "dsa_status_string", "dsa_last_cuda_error"]:
        assert n in names


def test_library_exports_every_declared_symbol(dsa_lib):
    out = subprocess.run(["nm", "-D", "--defined-only", dsa.library_path()], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\bT\s+(\w+)", out))
    for n in _declared():
        assert n in exported, n
        assert getattr(dsa_lib, n) is not None


def test_struct_layout_matches_header(tmp_path):
    fields = [f[0] for f in dsa.DsaAttnArgs._fields_]
    src = tmp_path / "layout.c"
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "dsa.h"\nint main(void){\n'
                   'printf("%zu\\n", sizeof(dsa_attn_args_t));\n' +
                   "".join(f'printf("%zu\\n", offsetof(dsa_attn_args_t, {f}));\n' for f in fields) + "return 0;}\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    vals = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    assert vals[0] == ctypes.sizeof(dsa.DsaAttnArgs)
    for f, off in zip(fields, vals[1:]):
        assert getattr(dsa.DsaAttnArgs, f).offset == off, f


def test_row_bytes_and_status_strings(dsa_lib):
    assert dsa.dsa_packed_row_bytes(256, 0) == 264
    assert dsa.dsa_packed_row_bytes(512, 64) == 656
    assert dsa.dsa_packed_row_bytes(100, 0) == -1
    assert dsa.dsa_cache_row_bytes(dsa.CACHE_BF16, 256, 0) == 512
    assert dsa.dsa_cache_row_bytes(dsa.CACHE_FP8_SCALED, 512, 64) == 656
    for s in range(6):
        assert dsa.dsa_status_string(s).startswith("DSA_")


def test_argument_errors_need_no_gpu(dsa_lib):
    L = dsa_lib
    P = ctypes.c_void_p
    fake = P(0x10000)
    # negative count, unsupported geometry, missing pointer: rejected before any CUDA call
    assert L.dsa_quant_k_cache(fake, 256, None, 0, -1, 256, 0, None, fake, 10, None, None) == 1
    assert L.dsa_quant_k_cache(fake, 256, None, 0, 4, 384, 0, None, fake, 10, None, None) == 2
    assert L.dsa_quant_k_cache(None, 256, None, 0, 4, 256, 0, None, fake, 10, None, None) == 1
    assert L.dsa_quant_k_cache(fake, 256, fake, 64, 4, 256, 0, None, fake, 10, None, None) == 1
    assert L.dsa_quant_k_cache(fake, 256, None, 0, 0, 256, 0, None, fake, 10, None, None) == 0
    assert L.dsa_gather_dequant(fake, 7, 10, 256, 0, fake, 4, None, 0, 0, 0, None, fake, None, None) == 1
    assert L.dsa_gather_dequant(fake, 1, 10, 128, 0, fake, 4, None, 0, 0, 0, None, fake, None, None) == 2
    i64 = ctypes.c_int64
    assert L.dsa_gather_requant(fake, i64(10), 256, 0, fake, i64(-1), None, i64(0), 0, 0, None, None, fake, i64(10),
                                None, None) == 1
    assert L.dsa_gather_requant(fake, i64(10), 384, 0, fake, i64(4), None, i64(0), 0, 0, None, None, fake, i64(10),
                                None, None) == 2
    assert L.dsa_gather_requant(fake, i64(10), 256, 0, fake, i64(4), None, i64(0), 0, 0, None, None, fake, i64(2),
                                None, None) == 1  # more results than output rows, no out_loc
    assert L.dsa_gather_requant(fake, i64(10), 256, 0, fake, i64(0), None, i64(0), 0, 0, None, None, fake, i64(10),
                                None, None) == 0
    # top-k selection: bad width, bad stride, missing pointer; nothing to do
    assert L.dsa_topk_select(fake, i64(4), i64(100), i64(100), None, 0, fake, i64(8), None) == 1
    assert L.dsa_topk_select(fake, i64(4), i64(100), i64(100), None, 16385, fake, i64(16385), None) == 1
    assert L.dsa_topk_select(fake, i64(4), i64(100), i64(99), None, 8, fake, i64(8), None) == 1
    assert L.dsa_topk_select(fake, i64(4), i64(100), i64(100), None, 8, fake, i64(7), None) == 1
    assert L.dsa_topk_select(None, i64(4), i64(100), i64(100), None, 8, fake, i64(8), None) == 1
    assert L.dsa_topk_select(fake, i64(4), i64(1 << 31), i64(1 << 31), None, 8, fake, i64(8), None) == 2
    assert L.dsa_topk_select(fake, i64(0), i64(100), i64(100), None, 8, fake, i64(8), None) == 0
    a = dsa.DsaAttnArgs()
    a.H, a.d_nope, a.d_rope, a.d_v, a.topk, a.T = 64, 256, 0, 256, 2048, 4
    a.q = a.cache = a.indices = a.out = a.workspace = 0x10000
    a.num_slots, a.sm_scale = 100, 0.0625
    a.q_stride_h, a.q_stride_t, a.idx_stride_t = 256, 64 * 256, 2048
    a.out_stride_h, a.out_stride_t = 256, 64 * 256
    good = dsa.DsaAttnArgs.from_buffer_copy(a)
    for field, val, want in [("H", 32, 2), ("d_nope", 128, 2), ("topk", 0, 1), ("sm_scale", float("inf"), 1), ("sm_scale", float("nan"), 1),
                             ("q_stride_h", 100, 1), ("kind", 9, 1), ("out", 0, 1), ("T", -1, 1)]:
        b = dsa.DsaAttnArgs.from_buffer_copy(good)
        setattr(b, field, val)
        assert L.dsa_sparse_attn(ctypes.byref(b), None) == want, field
    b = dsa.DsaAttnArgs.from_buffer_copy(good)
    b.T = 0
    assert L.dsa_sparse_attn(ctypes.byref(b), None) == 0


def test_blockscale_sizes_and_argument_errors(dsa_lib):
    assert dsa.dsa_blockscale_bytes(1, 128) == 512
    assert dsa.dsa_blockscale_bytes(129, 256) == 2 * 2 * 512
    assert dsa.dsa_blockscale_bytes(8, 100) == -1
    P = ctypes.c_void_p(16)
    # bad block size, cols not a multiple of 128: rejected before any device work
    assert dsa_lib.dsa_quant_fp8_blockscale(P, 4, 128, 128, 7, P, P, None) == 1
    assert dsa_lib.dsa_quant_fp8_blockscale(P, 4, 100, 128, 1, P, P, None) == 1
    assert dsa_lib.dsa_quant_fp8_blockscale(P, 4, 128, 120, 1, P, P, None) == 1
    # N and K multiples of 128, output stride at least N
    assert dsa_lib.dsa_proj_gemm(P, P, P, P, 4, 100, 128, P, 128, None, 0, None) == 1
    assert dsa_lib.dsa_proj_gemm(P, P, P, P, 4, 128, 100, P, 128, None, 0, None) == 1
    assert dsa_lib.dsa_proj_gemm(P, P, P, P, 4, 256, 128, P, 128, None, 0, None) == 1
    assert dsa_lib.dsa_proj_gemm(P, P, P, P, 0, 128, 128, P, 128, None, 0, None) == 0
