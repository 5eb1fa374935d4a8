"""dsa_sparse_attn under concurrency and replay.

- Two streams at once, each with the binding's default workspace: the binding keeps one
  workspace per (device, stream), so calls that overlap on the GPU never share split-token
  scratch; both results must match the oracle.
- A recorded launch replayed with new inputs: the merge flags of a call carry a tag fixed when
  the launch is recorded, and the kernel clears every flag it consumes, so each replay merges
  only the partial results that replay wrote. Every replay must equal a direct call on the same
  inputs bit for bit (same grid, same schedule).
"""
import numpy as np
import pytest
import torch

import dsa_sparse_attention_mla_gb300 as dsa
from dsa_sparse_attention_mla_gb300 import workloads as W

from _helpers import bf16_dev, check_close, f32_of, oracle_cache, run_oracle

pytestmark = pytest.mark.gpu


def _inputs(wl, device):
    cache = oracle_cache(wl)
    q = bf16_dev(wl.q_bits(), device)
    dcache = bf16_dev(cache, device) if wl.kind == 0 else torch.from_numpy(cache).to(device)
    idx = torch.from_numpy(wl.indices).to(device)
    bt = None if wl.block_table is None else torch.from_numpy(wl.block_table).to(device)
    req = None if wl.req_of_token is None else torch.from_numpy(wl.req_of_token).to(device)
    return cache, q, dcache, idx, bt, req


def test_two_streams_default_workspaces(gpu):
    """Two split-heavy batches (few tokens, every token over several CTAs) launched on two streams
    with no ordering between them; each stream's calls use that stream's default workspace."""
    wls = [W.bf16_direct(T=6, slots=5000, topk=2112, n_valid=2051, seed=61, sm_scale=1 / 16, scatter_frac=0.3),
           W.fp8_paged(T=8, requests=2, positions=4096, page_size=64, topk=2112, n_valid=2051, seed=62,
                       sm_scale=1 / 16, scatter_frac=0.3)]
    ins = [_inputs(wl, gpu) for wl in wls]
    streams = [torch.cuda.Stream(gpu) for _ in wls]
    torch.cuda.synchronize()
    outs = [[], []]
    for rep in range(4):
        for k, (wl, (_, q, dcache, idx, bt, req)) in enumerate(zip(wls, ins)):
            with torch.cuda.stream(streams[k]):
                outs[k].append(dsa.dsa_sparse_attn(q, dcache, wl.kind, idx, wl.sm_scale, block_table=bt,
                                                   page_size=wl.page_size, req_of_token=req))
    torch.cuda.synchronize()
    for k, wl in enumerate(wls):
        ref, _, bad = run_oracle(wl, ins[k][0])
        assert bad == 0
        for o in outs[k]:
            check_close(f32_of(o), ref, f"{wl.name} on stream {k}")


@pytest.mark.parametrize("kind", [0, 1])
def test_recorded_launch_replayed_with_new_inputs(gpu, kind):
    """Record one dsa_sparse_attn call (caller workspace) in a CUDA graph, then replay it three
    times after copying new queries and index lists into the recorded input buffers."""
    base = W.fp8_paged(T=8, requests=2, positions=4096, page_size=64, topk=2112, n_valid=2051, seed=70,
                       sm_scale=1 / 16, scatter_frac=0.3)
    base.kind = kind
    cache, q, dcache, idx, bt, req = _inputs(base, gpu)
    ws = torch.zeros(dsa.dsa_sparse_attn_workspace_size(256), dtype=torch.uint8, device=gpu)
    out = torch.empty((base.T, 64, 256), dtype=torch.bfloat16, device=gpu)
    err = torch.zeros(1, dtype=torch.int32, device=gpu)

    def call():
        dsa.dsa_sparse_attn(q, dcache, kind, idx, base.sm_scale, block_table=bt, page_size=base.page_size,
                            req_of_token=req, out=out, workspace=ws, error_word=err)

    side = torch.cuda.Stream(gpu)
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call()  # the first call on the device does its one-time set-up outside the recording
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    torch.cuda.synchronize()
    for rep in range(3):
        wl = W.fp8_paged(T=8, requests=2, positions=4096, page_size=64, topk=2112, n_valid=2051, seed=71 + rep,
                         sm_scale=1 / 16, scatter_frac=0.3)
        q.copy_(bf16_dev(wl.q_bits(), gpu))
        idx.copy_(torch.from_numpy(wl.indices).to(gpu))
        g.replay()
        torch.cuda.synchronize()
        assert err.item() == 0, f"replay {rep}: device error word {err.item()}"
        replayed = out.clone()
        direct = dsa.dsa_sparse_attn(q, dcache, kind, idx, base.sm_scale, block_table=bt, page_size=base.page_size,
                                     req_of_token=req)
        torch.cuda.synchronize()
        assert torch.equal(replayed.view(torch.int16), direct.view(torch.int16)), f"replay {rep}"
        wl.kind = kind
        wl.block_table, wl.req_of_token = base.block_table, base.req_of_token  # the recorded cache and table
        ref, _, bad = run_oracle(wl, cache)
        assert bad == 0
        check_close(f32_of(replayed), ref, f"replay {rep}")
