"""The fixed-scratch entry point dsa_sparse_attn_static_ws, called through the C ABI.

It serves callers that cannot allocate device memory when they call the library (engines that
reserve all device memory up front, runtimes with a fixed memory plan, latency-critical paths
where an allocation could stall the device): the split-token scratch comes from a device array
inside the library. Two calls in a row must each match the workspace-taking dsa_sparse_attn
within the attention tolerance of the other GPU tests (here they are in fact bit-identical:
same grid, same schedule). The workload (8 tokens, top-k 2112) splits every token over several
CTAs, so the shared scratch and its flags are exercised, and the second call checks that the
first left them in a usable state. This file is collected last on purpose.
"""
import ctypes

import pytest
import torch

import dsa_sparse_attention_mla_gb300 as dsa
from dsa_sparse_attention_mla_gb300 import workloads as W

from _helpers import bf16_dev, check_close, f32_of, oracle_cache

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("kind", [0, 1])
def test_static_scratch_matches_workspace_entry_point(gpu, kind):
    wl = W.fp8_paged(T=8, requests=2, positions=4096, page_size=64, topk=2112, n_valid=2051, seed=77,
                     sm_scale=1 / 16, scatter_frac=0.5)
    wl.kind = kind
    cache = oracle_cache(wl)
    q = bf16_dev(wl.q_bits(), gpu)
    dcache = bf16_dev(cache, gpu) if kind == 0 else torch.from_numpy(cache).to(gpu)
    idx = torch.from_numpy(wl.indices).to(gpu)
    bt = torch.from_numpy(wl.block_table).to(gpu)
    req = torch.from_numpy(wl.req_of_token).to(gpu)
    ref = dsa.dsa_sparse_attn(q, dcache, kind, idx, wl.sm_scale, block_table=bt, page_size=wl.page_size,
                              req_of_token=req)
    lib = dsa.load_library()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        out = torch.full_like(ref, float("nan"))
        err = torch.zeros(1, dtype=torch.int32, device=gpu)
        a = dsa._attn_args(q, dcache, kind, idx, wl.sm_scale, 256, 0, 256, bt, wl.page_size, req, out, None, None,
                           err)
        st = lib.dsa_sparse_attn_static_ws(ctypes.byref(a), stream)
        assert st == 0, dsa.dsa_status_string(st)
        torch.cuda.synchronize()
        assert err.item() == 0, f"call {call}: device error word {err.item()}"
        check_close(f32_of(out), f32_of(ref), f"static scratch, call {call}")


def test_static_scratch_argument_errors(dsa_lib):
    a = dsa.DsaAttnArgs()
    a.H, a.d_nope, a.d_rope, a.d_v, a.topk, a.T = 32, 256, 0, 256, 2048, 4
    assert dsa_lib.dsa_sparse_attn_static_ws(ctypes.byref(a), None) == 2   # unsupported head count
    a.H, a.T = 64, 0
    assert dsa_lib.dsa_sparse_attn_static_ws(ctypes.byref(a), None) == 0   # nothing to do
    assert dsa_lib.dsa_sparse_attn_static_ws(None, None) == 1


def test_static_scratch_with_the_work_balanced_split(gpu):
    """Long causal lists (T=3072): the launch takes the work-balanced split, whose slice counts
    and range bounds also live in the fixed scratch; two calls equal the workspace entry point
    bit for bit (same bounds, same schedule)."""
    wl = W.prefill_causal(T=3072, topk=2048, window=128, seed=31, name="prefill_causal_T3072")
    cache = oracle_cache(wl)
    q = bf16_dev(wl.q_bits(), gpu)
    dcache = bf16_dev(cache, gpu)
    idx = torch.from_numpy(wl.indices).to(gpu)
    ref = dsa.dsa_sparse_attn(q, dcache, 0, idx, wl.sm_scale)
    lib = dsa.load_library()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        out = torch.full_like(ref, float("nan"))
        err = torch.zeros(1, dtype=torch.int32, device=gpu)
        a = dsa._attn_args(q, dcache, 0, idx, wl.sm_scale, 256, 0, 256, None, 0, None, out, None, None, err)
        st = lib.dsa_sparse_attn_static_ws(ctypes.byref(a), stream)
        assert st == 0, dsa.dsa_status_string(st)
        torch.cuda.synchronize()
        assert err.item() == 0
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), f"call {call}"
