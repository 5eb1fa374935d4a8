"""Benchmark: DSA sparse MLA attention on one GB300 (or N independent replicas).

Default workload: batched decode over a packed scaled-FP8 paged cache, 256+0 latent geometry,
256 requests x 32768 positions (8,388,608 slots, 2.2 GB of 264-byte rows), one query token per
request, top-k 2048 valid entries per token in a 2112-wide list (70% from the last 4096
positions, 30% uniform over the rest; 5% of tokens with the -1 padding scattered), 64 heads,
sm_scale 1/16. One step = one dsa_sparse_attn call over the whole batch.

Prints ONE JSON line (rank 0). Timing: W untimed warm-up steps, then K timed steps; every step is
bracketed by CUDA events on the launching stream and a 512 MB buffer is written between steps
(outside the events) so the L2 (129 MB) holds none of the step's inputs. ``value`` = tokens per
second over the K steps (all ranks, max time over ranks). ``e2e`` repeats the measurement through
the same call with the step's inputs (q, indices) copied from pinned host memory and the output
copied back inside the timed region. ``cpu_baseline`` times the CPU oracle on a bounded sample.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config 1..5] [--impl reference]
  python bench.py --op requant|proj|topk|pack|dequant     (the other entry points, one JSON line each)
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

L2_FLUSH_BYTES = 512 << 20
NOMINAL_HBM_GBS = 7900.0
NOMINAL_BF16_TFLOPS = 2250.0
METRIC = "sparse-attn tokens/s (256+0 FP8, T=256)"


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


def max_over_ranks(value: float, world: int) -> float:
    """The largest of every rank's value (the job's time is its slowest rank's). The exchange
    tensor lives where the process group's backend wants it: the GPU for NCCL, the host for gloo."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist

    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(world: int, tokens_per_rank: int, steps: int, total_ms: float) -> float:
    """Whole-job tokens/s: every rank processes its own copy of the workload (weak scaling), and
    the job takes the slowest rank's time."""
    return world * tokens_per_rank * steps / (total_ms / 1000.0)


def _recorded_traffic(workload):
    """DRAM bytes per launch of the attention kernel for this workload, from the ncu capture
    recorded under profiles/, or None when there is none or the kernel sources have changed
    since it was taken (the record carries a hash of the source files of the measured kernels)."""
    import hashlib

    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    src = os.path.join(ROOT, "dsa_sparse_attention_mla_gb300", "csrc")
    # the record names the source files of the kernels it measured (every file when it names none)
    names = rec.get("sources") or [n for n in os.listdir(src) if n.endswith((".cu", ".cuh", ".h", ".cpp"))]
    h = hashlib.sha256()
    for name in sorted(names):
        path = os.path.join(src, name)
        if not os.path.exists(path):
            return None
        h.update(name.encode())
        with open(path, "rb") as f:
            h.update(f.read())
    if h.hexdigest() != rec.get("csrc_sha256"):
        return None
    w = rec.get("workloads", {}).get(workload)
    return None if w is None else int(w["traffic"])


def kernels_per_call(wl, sm_count):
    """Kernel launches of one dsa_sparse_attn call, by the launcher's own rule: the 256+0 kernel
    (d_nope 256, no rope) takes a work-balanced split, two small pre-pass kernels, when its
    CTAs hold at least 64 (token, 128-entry) units each; every other call is one launch."""
    if wl.d_nope != 256 or wl.d_rope != 0:
        return 1
    nt = (wl.indices.shape[1] + 127) // 128
    u = wl.T * nt
    g = min(sm_count, (u + 3) // 4)
    k = max(1, nt // 4)
    if wl.T * k <= sm_count:
        g = wl.T * k
    while g > 1 and (nt + u // g - 1) // (u // g) + 1 > 17:
        g -= 1
    gap = (nt + 14) // 15
    return 3 if (1 < g <= 192 and u // g >= 64 and u >= g * gap) else 1


def algorithmic_work(wl):
    """Algorithmic bytes and FLOPs of one full call (per the data each token must touch once):
    gathered rows (valid entries x row bytes) + q + out + the index list + the block table;
    FLOPs = 2 * H * n_valid * (D_K + d_v)."""
    n_valid = int((wl.indices >= 0).sum())
    rb = (wl.d_nope + 4 * (wl.d_nope // 128) + 2 * wl.d_rope) if wl.kind == 1 else 2 * wl.D
    rows = n_valid * rb
    q = wl.T * wl.H * wl.D * 2
    out = wl.T * wl.H * wl.d_v * 2
    idx = wl.indices.size * 4
    bt = 0 if wl.block_table is None else wl.block_table.size * 4
    flops = 2.0 * wl.H * n_valid * (wl.D + wl.d_v)
    # each distinct cache row once: what HBM must deliver when repeated gathers hit L2
    idx_all = wl.indices.astype(np.int64)
    valid = idx_all >= 0
    if wl.block_table is None:
        phys = idx_all[valid]
    else:
        req = np.broadcast_to(wl.req_of_token.astype(np.int64)[:, None], idx_all.shape)[valid]
        pos = idx_all[valid]
        phys = wl.block_table[req, pos // wl.page_size].astype(np.int64) * wl.page_size + pos % wl.page_size
    unique_rows = int(np.unique(phys).size) * rb
    return {"bytes": rows + q + out + idx + bt, "row_bytes": rows, "flops": flops, "n_valid": n_valid,
            "unique_bytes": unique_rows + q + out + idx + bt}


def roofline(work, seconds, hbm_gbs, tensor_tflops):
    """The roofline of one call: the slower of the tensor-core term (FLOPs at the bf16 peak) and
    the memory term (each distinct row once, plus q, out and the index lists, at the HBM peak).
    Decode gathers distinct rows from a table far larger than the L2, so its memory term is all
    of its gathered bytes; causal prefill re-gathers rows of a 4 MB table that the L2 holds, so
    it is bound by the tensor core. `achieved` and `frac` are on the bounding term."""
    t_mem = work["unique_bytes"] / (hbm_gbs * 1e9)
    t_tc = work["flops"] / (tensor_tflops * 1e12)
    gbs = work["bytes"] / seconds / 1e9
    tflops = work["flops"] / seconds / 1e12
    if t_tc > t_mem:
        return {"bound": "tensor", "achieved": tflops, "peak": tensor_tflops, "unit": "TFLOP/s",
                "frac": tflops / tensor_tflops, "gathered_gbs": gbs, "roofline_us": t_tc * 1e6}
    return {"bound": "hbm", "achieved": gbs, "peak": hbm_gbs, "unit": "GB/s", "frac": gbs / hbm_gbs,
            "tflops": tflops, "tensor_frac_of_bf16_burst": tflops / tensor_tflops, "roofline_us": t_mem * 1e6}


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        import torch

        try:
            self.gpu_id = "GPU-" + str(torch.cuda.get_device_properties(device).uuid)
        except Exception:
            self.gpu_id = str(device.index or 0)
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_id}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, pw, reasons = [], None, [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
                pw.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(pw) if pw else None}


# ------------------------------------------------------------------------------ GPU inputs --
def build_device_inputs(wl, device):
    """Resident inputs for one workload: the cache is generated and packed on the GPU."""
    import torch

    import dsa_sparse_attention_mla_gb300 as dsa

    q = wl.q.torch(device).view(wl.T, wl.H, wl.D)
    if wl.kind == 0:
        cache = wl.kv.torch(device)
    else:
        rb = dsa.dsa_packed_row_bytes(wl.d_nope, wl.d_rope)
        cache = torch.empty((wl.num_slots, rb), dtype=torch.uint8, device=device)
        chunk = 1 << 20
        loc_all = None if wl.kv_slot is None else torch.from_numpy(wl.kv_slot).to(device)
        from dsa_sparse_attention_mla_gb300.workloads import normal_bf16_torch

        for r0 in range(0, wl.num_slots, chunk):
            n = min(chunk, wl.num_slots - r0)
            rows = normal_bf16_torch(wl.kv.seed, wl.kv.stream, r0 * wl.D, n * wl.D, device).view(n, wl.D)
            loc = (torch.arange(r0, r0 + n, device=device, dtype=torch.int64) if loc_all is None else loc_all[r0:r0 + n])
            dsa.dsa_quant_k_cache(rows[:, : wl.d_nope], rows[:, wl.d_nope:] if wl.d_rope else None, out_loc=loc,
                                  cache=cache, num_slots=wl.num_slots)
        torch.cuda.synchronize(device)
    idx = torch.from_numpy(wl.indices).to(device)
    bt = None if wl.block_table is None else torch.from_numpy(wl.block_table).to(device)
    req = None if wl.req_of_token is None else torch.from_numpy(wl.req_of_token).to(device)
    return q, cache, idx, bt, req


def run_gpu(args, wl, rank, world, device, config):
    import torch

    import dsa_sparse_attention_mla_gb300 as dsa

    q, cache, idx, bt, req = build_device_inputs(wl, device)
    out = torch.empty((wl.T, wl.H, wl.d_v), dtype=torch.bfloat16, device=device)
    err = torch.zeros(1, dtype=torch.int32, device=device)
    ws = torch.zeros(dsa.dsa_sparse_attn_workspace_size(wl.d_v), dtype=torch.uint8, device=device)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)

    def step(o=out, qq=q, ii=idx):
        dsa.dsa_sparse_attn(qq, cache, wl.kind, ii, wl.sm_scale, d_nope=wl.d_nope, d_rope=wl.d_rope, d_v=wl.d_v,
                            block_table=bt, page_size=wl.page_size, req_of_token=req, out=o, workspace=ws,
                            error_word=err)

    for _ in range(args.warmup):
        flush.fill_(1)
        step()
    torch.cuda.synchronize(device)

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(device)
    with ClockSampler(device) as clk:
        t_wall0 = time.perf_counter()
        for i in range(args.steps):
            flush.fill_(i & 0xFF)
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize(device)
        t_wall = time.perf_counter() - t_wall0
    if world > 1:
        torch.distributed.barrier()
    times = [s.elapsed_time(e) for s, e in zip(starts, ends)]  # ms
    total_ms = max_over_ranks(float(sum(times)), world)
    if err.item() != 0:
        raise RuntimeError(f"device error word {err.item()} during the benchmark")

    # ---- end to end: host-resident q and indices in, output back to host, copies timed
    e2e_steps = max(3, min(args.steps, 200))
    q_h = q.cpu().pin_memory()
    idx_h = idx.cpu().pin_memory()
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    q_d, idx_d = torch.empty_like(q), torch.empty_like(idx)
    e_s = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps)]
    e_e = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps)]
    for i in range(e2e_steps + 2):
        flush.fill_(3)
        if i >= 2:
            e_s[i - 2].record(stream)
        q_d.copy_(q_h, non_blocking=True)
        idx_d.copy_(idx_h, non_blocking=True)
        step(out, q_d, idx_d)
        out_h.copy_(out, non_blocking=True)
        if i >= 2:
            e_e[i - 2].record(stream)
    torch.cuda.synchronize(device)
    e2e_ms = float(sum(s.elapsed_time(e) for s, e in zip(e_s, e_e)) / e2e_steps)
    h2d = q.numel() * q.element_size() + idx.numel() * idx.element_size()
    d2h = out.numel() * out.element_size()

    # ---- end to end, pipelined: step i+1's inputs are copied in (one copy stream) and step i-1's
    # output read back (another) while step i computes, over two buffer sets. Every step still
    # copies its own inputs from pinned host memory and reads its own result back. The steps
    # rotate among four independently drawn index sets of the same workload, so consecutive
    # steps' gathered rows (four times a step's) cannot be served from L2 without a flush.
    from dsa_sparse_attention_mla_gb300 import workloads as W

    idx_sets = [idx_h] + [torch.from_numpy(W.config(config, seed=sd).indices).pin_memory() for sd in (1, 2, 3)]
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    qd = [torch.empty_like(q) for _ in range(2)]
    idd = [torch.empty_like(idx) for _ in range(2)]
    od = [torch.empty_like(out) for _ in range(2)]
    oh = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_cmp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def pipeline(n, first=0):
        for i in range(first, first + n):
            k = i & 1
            with torch.cuda.stream(s_in):
                if i - first >= 2:
                    s_in.wait_event(ev_cmp[k])  # step i-2 no longer reads buffer set k
                qd[k].copy_(q_h, non_blocking=True)
                idd[k].copy_(idx_sets[i % 4], non_blocking=True)
                ev_in[k].record(s_in)
            stream.wait_event(ev_in[k])
            if i - first >= 2:
                stream.wait_event(ev_out[k])  # step i-2's output has been read back
            step(od[k], qd[k], idd[k])
            ev_cmp[k].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_cmp[k])
                oh[k].copy_(od[k], non_blocking=True)
                ev_out[k].record(s_out)

    pipeline(4)
    torch.cuda.synchronize(device)
    p_start, p_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    p_start.record(s_in)
    pipeline(e2e_steps, first=4)
    p_end.record(s_out)
    torch.cuda.synchronize(device)
    e2e_pipe_ms = p_start.elapsed_time(p_end) / e2e_steps
    return {"total_ms": total_ms, "times": times, "t_wall": t_wall, "clocks": clk.summary(), "e2e_ms": e2e_ms,
            "e2e_pipe_ms": e2e_pipe_ms, "h2d": h2d, "d2h": d2h}


def run_requant(args, device):
    """Timing of dsa_gather_requant on the decode workload's gathered rows: every valid entry of
    the 256 tokens (paged, 524,288 rows of 264 bytes) gathered, widened and re-packed into a
    contiguous buffer. One JSON line like the attention bench's, HBM-bound."""
    import torch

    import dsa_sparse_attention_mla_gb300 as dsa
    from dsa_sparse_attention_mla_gb300 import workloads as W

    wl = W.config(3, seed=0)
    _, cache, _, bt, _ = build_device_inputs(wl, device)
    valid = wl.indices >= 0
    pos = torch.from_numpy(wl.indices[valid].astype(np.int32)).to(device)
    req = torch.from_numpy(np.broadcast_to(wl.req_of_token[:, None], wl.indices.shape)[valid].astype(np.int32)).to(device)
    n = int(pos.numel())
    rb = dsa.dsa_packed_row_bytes(wl.d_nope, wl.d_rope)
    out = torch.empty((n, rb), dtype=torch.uint8, device=device)
    err = torch.zeros(1, dtype=torch.int32, device=device)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)

    def step():
        dsa.dsa_gather_requant(cache, wl.d_nope, wl.d_rope, pos, block_table=bt, page_size=wl.page_size,
                               req_of_index=req, out=out, error_word=err)

    for _ in range(args.warmup):
        flush.fill_(1)
        step()
    torch.cuda.synchronize(device)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(device) as clk:
        for i in range(args.steps):
            flush.fill_(i & 0xFF)
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize(device)
    times = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    if err.item() != 0:
        raise RuntimeError(f"device error word {err.item()} during the benchmark")
    ms = float(sum(times)) / args.steps
    nbytes = n * (2 * rb + 4 + 4)  # row read + row written + logical position + request
    hbm = _peaks()[0]
    achieved = nbytes / (ms / 1000.0) / 1e9
    # CPU baseline: the oracle's gather_requant on a bounded sample of the same rows
    import oracle
    from oracle.workload_inputs import cache_for_tokens

    tok = np.arange(8)
    host_cache = cache_for_tokens(wl, tok)
    v8 = wl.indices[tok] >= 0
    hp = wl.indices[tok][v8].astype(np.int32)
    hr = np.broadcast_to(wl.req_of_token[tok][:, None], v8.shape)[v8].astype(np.int32)
    t0 = time.perf_counter()
    oracle.gather_requant(host_cache, wl.d_nope, wl.d_rope, hp, block_table=wl.block_table, page_size=wl.page_size,
                          req_of_index=hr)
    cpu_rows_s = hp.size / (time.perf_counter() - t0)
    line = {
        "metric": "gather-requant rows/s (256+0 FP8 paged)", "value": n / (ms / 1000.0), "unit": "rows/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "u8", "data": "synthetic",
        "config": {"workload": "requant_" + wl.name, "rows": n, "row_bytes": rb,
                   "l2": "512 MB buffer written between timed steps (outside the events)"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                     "traffic": _recorded_traffic("requant_" + wl.name), "algorithmic_bytes_per_launch": nbytes},
        "cpu_baseline": {"value": cpu_rows_s, "unit": "rows/s", "cores": 1, "kind": "oracle",
                         "sample": f"{hp.size} rows of 8 tokens", "cpu": cpu_model()},
        "gpu_launches": args.steps, "clocks": clk.summary(),
        "step_ms": {"median": statistics.median(times), "min": min(times), "max": max(times)},
    }
    print(json.dumps(line))


def run_topk(args, device):
    """Timing of dsa_topk_select, the selection that produces the attention's index lists, on
    two shapes: decode (256 rows of scores over 32768 positions, every position visible, K 2048)
    and causal prefill (8192 rows over 8192 positions, row t seeing positions 0 .. t, K 2048).
    Scores are seeded standard normals drawn on the device. One JSON line (decode) with the
    prefill shape alongside; HBM-bound: the visible scores are read once and the lists written."""
    import torch

    import dsa_sparse_attention_mla_gb300 as dsa

    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)
    hbm = _peaks()[0]

    def shape(T, S, K, causal, seed):
        gen = torch.Generator(device=device)
        gen.manual_seed(seed)
        scores = torch.randn((T, S), generator=gen, dtype=torch.float32, device=device)
        lengths = (torch.arange(T, dtype=torch.int32, device=device) + 1).clamp_(max=S) if causal else None
        out = torch.empty((T, K), dtype=torch.int32, device=device)

        def step():
            dsa.dsa_topk_select(scores, K, lengths=lengths, out=out)

        for _ in range(args.warmup):
            flush.fill_(1)
            step()
        torch.cuda.synchronize(device)
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        with ClockSampler(device) as clk:
            for i in range(args.steps):
                flush.fill_(i & 0xFF)
                starts[i].record(stream)
                step()
                ends[i].record(stream)
            torch.cuda.synchronize(device)
        times = [a.elapsed_time(b) for a, b in zip(starts, ends)]
        ms = float(sum(times)) / args.steps
        visible = sum(min(t + 1, S) for t in range(T)) if causal else T * S
        nbytes = 4 * visible + 4 * T * K + (4 * T if causal else 0)
        achieved = nbytes / (ms / 1000.0) / 1e9
        name = f"topk_{'prefill' if causal else 'decode'}_T{T}_S{S}_k{K}"
        res = {"metric": f"top-k selection rows/s ({name})", "value": T / (ms / 1000.0), "unit": "rows/s",
               "ms_per_step": ms, "dtype": "f32 scores, int32 lists",
               "config": {"workload": name, "rows": T, "positions": S, "k": K, "causal": causal,
                          "l2": "512 MB buffer written between timed steps (outside the events)"},
               "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                            "traffic": None, "algorithmic_bytes_per_launch": nbytes},
               "gpu_launches": args.steps, "clocks": clk.summary(),
               "step_ms": {"median": statistics.median(times), "min": min(times), "max": max(times)}}
        return res, scores, lengths

    dec, scores, _ = shape(256, 32768, 2048, False, 11)
    pre, _, _ = shape(8192, 8192, 2048, True, 12)
    # CPU baseline: the oracle's stable sort on a bounded sample of the decode rows
    from oracle.selection import topk_select

    host = scores[:16].cpu().numpy()
    t0 = time.perf_counter()
    topk_select(host, 2048)
    cpu_rows_s = host.shape[0] / (time.perf_counter() - t0)
    line = dict(dec)
    line.update({"n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
                 "scaling": "weak", "vs_baseline": None, "data": "synthetic",
                 "cpu_baseline": {"value": cpu_rows_s, "unit": "rows/s", "cores": 1, "kind": "oracle",
                                  "sample": "16 of the 256 decode rows", "cpu": cpu_model()},
                 "prefill": pre})
    print(json.dumps(line))


def _time_op(args, device, step):
    """Mean time (ms) of `step` over args.steps calls between CUDA events on the current stream,
    after args.warmup untimed calls, with the 512 MB L2 flush between calls (outside the events);
    returns (ms, step times, clock summary)."""
    import torch

    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)
    for _ in range(args.warmup):
        flush.fill_(1)
        step()
    torch.cuda.synchronize(device)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(device) as clk:
        for i in range(args.steps):
            flush.fill_(i & 0xFF)
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize(device)
    times = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    return float(sum(times)) / args.steps, times, clk.summary()


def run_cache_ops(args, device):
    """Timing of the two cache kernels at the decode workload's sizes: --op pack packs 1,048,576
    bf16 latent rows (256+0) into 264-byte rows scattered through a random slot map
    (dsa_quant_k_cache); --op dequant gathers and widens the 524,288 rows the 256 decode tokens
    name (dsa_gather_dequant, paged). One JSON line each, HBM-bound."""
    import torch

    import dsa_sparse_attention_mla_gb300 as dsa
    import oracle
    from dsa_sparse_attention_mla_gb300 import workloads as W

    hbm = _peaks()[0]
    err = torch.zeros(1, dtype=torch.int32, device=device)
    if args.op == "pack":
        n = 1 << 20
        gen = torch.Generator(device=device)
        gen.manual_seed(21)
        kv = torch.randn((n, 256), generator=gen, device=device).to(torch.bfloat16)
        loc = torch.randperm(n, generator=gen, device=device)
        cache = torch.empty((n, 264), dtype=torch.uint8, device=device)

        def step():
            dsa.dsa_quant_k_cache(kv, out_loc=loc, cache=cache, error_word=err)

        ms, times, clk = _time_op(args, device, step)
        nbytes = n * (512 + 264 + 8)
        host_kv = kv[:4096].view(torch.int16).cpu().numpy().view(np.uint16)
        t0 = time.perf_counter()
        oracle.quant_k_cache(host_kv, num_slots=4096, n_threads=1)
        cpu_v = 4096 / (time.perf_counter() - t0)
        name, metric, sample = "pack_256p0_rows1048576", "pack rows/s (256+0, 264-byte rows)", "4096 rows"
    else:
        wl = W.config(3, seed=0)
        _, cache, _, bt, _ = build_device_inputs(wl, device)
        valid = wl.indices >= 0
        pos = torch.from_numpy(wl.indices[valid].astype(np.int32)).to(device)
        req = torch.from_numpy(np.broadcast_to(wl.req_of_token[:, None], wl.indices.shape)[valid].astype(np.int32)).to(device)
        n = int(pos.numel())
        out = torch.empty((n, 256), dtype=torch.bfloat16, device=device)

        def step():
            dsa.dsa_gather_dequant(cache, wl.kind, wl.d_nope, wl.d_rope, pos, block_table=bt, page_size=wl.page_size,
                                   req_of_index=req, out=out, error_word=err)

        ms, times, clk = _time_op(args, device, step)
        nbytes = n * (264 + 512 + 4 + 4)
        from oracle.workload_inputs import cache_for_tokens

        tok = np.arange(8)
        host_cache = cache_for_tokens(wl, tok)
        v8 = wl.indices[tok] >= 0
        hp = wl.indices[tok][v8].astype(np.int32)
        hr = np.broadcast_to(wl.req_of_token[tok][:, None], v8.shape)[v8].astype(np.int32)
        t0 = time.perf_counter()
        oracle.gather_dequant(host_cache, oracle.CACHE_FP8_SCALED, wl.d_nope, wl.d_rope, hp, block_table=wl.block_table,
                              page_size=wl.page_size, req_of_index=hr)
        cpu_v = hp.size / (time.perf_counter() - t0)
        name, metric = "dequant_" + wl.name, "gather-dequant rows/s (256+0 FP8 paged)"
        sample = f"{hp.size} rows of 8 tokens"
    if err.item() != 0:
        raise RuntimeError(f"device error word {err.item()} during the benchmark")
    achieved = nbytes / (ms / 1000.0) / 1e9
    line = {
        "metric": metric, "value": n / (ms / 1000.0), "unit": "rows/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": name, "rows": n, "l2": "512 MB buffer written between timed steps (outside the events)"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                     "traffic": None, "algorithmic_bytes_per_launch": nbytes},
        "cpu_baseline": {"value": cpu_v, "unit": "rows/s", "cores": 1, "kind": "oracle", "sample": sample,
                         "cpu": cpu_model()},
        "gpu_launches": args.steps, "clocks": clk,
        "step_ms": {"median": statistics.median(times), "min": min(times), "max": max(times)},
    }
    print(json.dumps(line))


def run_proj(args, device):
    """Timing of the FP8 block-scaled projection GEMM at prefill size (8192 tokens): q_b_proj
    (K 2048 -> N 16384 = 64 heads x 256) and o_proj (K 16384 -> N 6144); the pages name the layers
    but give no widths, so these are read from the attention's geometry. Weights are quantised
    once; each timed step quantises the activations (1 x 128 blocks) and runs the GEMM. Bound:
    the FP8 tensor peak, taken as twice the measured bf16 burst (the nominal 4.5 / 2.25 ratio)."""
    import torch

    import dsa_sparse_attention_mla_gb300 as dsa

    M = 8192
    shapes = [("q_b_proj", 2048, 16384), ("o_proj", 16384, 6144)]
    gen = torch.Generator(device=device).manual_seed(0)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)
    fp8_peak = 2.0 * _peaks()[1]
    out = []
    for name, K, N in shapes:
        x = torch.randn((M, K), generator=gen, device=device).to(torch.bfloat16)
        w = (torch.randn((N, K), generator=gen, device=device) * 0.02).to(torch.bfloat16)
        wc, ws = dsa.dsa_quant_fp8_blockscale(w, 128)
        xc = torch.empty((M, K), dtype=torch.uint8, device=device)
        xs = torch.empty(dsa.dsa_blockscale_bytes(M, K), dtype=torch.uint8, device=device)
        y = torch.empty((M, N), dtype=torch.bfloat16, device=device)

        def step():
            dsa.dsa_quant_fp8_blockscale(x, 1, codes=xc, scales=xs)
            dsa.dsa_proj_gemm(xc, xs, wc, ws, out=y)

        for _ in range(args.warmup):
            flush.fill_(1)
            step()
        torch.cuda.synchronize(device)
        n = max(3, min(args.steps, 200))
        t_all, t_gemm = [], []
        with ClockSampler(device) as clk:
            for i in range(n):
                flush.fill_(i & 0xFF)
                a, b, c = (torch.cuda.Event(enable_timing=True) for _ in range(3))
                a.record(stream)
                dsa.dsa_quant_fp8_blockscale(x, 1, codes=xc, scales=xs)
                b.record(stream)
                dsa.dsa_proj_gemm(xc, xs, wc, ws, out=y)
                c.record(stream)
                torch.cuda.synchronize(device)
                t_all.append(a.elapsed_time(c))
                t_gemm.append(b.elapsed_time(c))
        ms, ms_g = statistics.median(t_all), statistics.median(t_gemm)
        flops = 2.0 * M * N * K
        out.append({"layer": name, "M": M, "K": K, "N": N, "ms_per_step": ms, "gemm_ms": ms_g,
                    "tflops": flops / (ms / 1e3) / 1e12, "gemm_tflops": flops / (ms_g / 1e3) / 1e12,
                    "roofline": {"bound": "tensor", "achieved": flops / (ms_g / 1e3) / 1e12, "peak": fp8_peak,
                                 "unit": "TFLOP/s", "frac": flops / (ms_g / 1e3) / 1e12 / fp8_peak,
                                 "peak_source": "2 x measured bf16 burst"},
                    "clocks": clk.summary()})
    # CPU baseline: the oracle's product on a sample of 4 rows of the first layer
    from oracle import projection as P

    K, N = shapes[0][1], 256
    rng = np.random.default_rng(0)
    xb = P.f64_to_bf16(rng.standard_normal((4, K)))
    wb = P.f64_to_bf16(rng.standard_normal((N, K)) * 0.02)
    xc_h, xe_h = P.quant_blockscale(xb, 1)
    wc_h, we_h = P.quant_blockscale(wb, 128)
    t0 = time.perf_counter()
    P.proj_gemm(xc_h, xe_h, wc_h, we_h)
    cpu = 2.0 * 4 * N * K / (time.perf_counter() - t0)
    tot_flops = sum(2.0 * M * o["N"] * o["K"] for o in out)
    tot_ms = sum(o["ms_per_step"] for o in out)
    line = {"metric": "FP8 block-scaled projection GEMM TFLOP/s (q_b_proj + o_proj, 8192 tokens)",
            "value": tot_flops / (tot_ms / 1e3) / 1e12, "unit": "TFLOP/s", "n_gpus": 1, "steps": n,
            "warmup": args.warmup, "ms_per_step": tot_ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "e4m3", "data": "synthetic",
            "config": {"workload": "fp8_blockscale_proj_M8192", "layers": out,
                       "l2": f"{L2_FLUSH_BYTES >> 20} MB buffer written between timed steps (outside the events)"},
            "cpu_baseline": {"value": cpu / 1e12, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
                             "sample": "4 rows x 256 columns of q_b_proj (fp64 numpy product, quantisation excluded)",
                             "cpu": cpu_model()},
            "gpu_launches": n * 2 * len(shapes)}
    print(json.dumps(line))


# ---------------------------------------------------------------------------- CPU oracle --
class OracleRunner:
    """The CPU oracle (as it stands) on the workload. The packed cache rows the tokens name are
    generated and packed by the oracle on the host: no oracle input comes from the GPU path."""

    def __init__(self, wl, tokens=None):
        import oracle
        from oracle.workload_inputs import cache_for_tokens

        self.oracle = oracle
        self.wl = wl
        self.q = wl.q_bits()
        self.cache = cache_for_tokens(wl, np.arange(wl.T) if tokens is None else np.asarray(tokens))
        self.order = np.random.default_rng(1234).permutation(wl.T)
        self.threads = oracle.max_threads()

    def run(self, tokens) -> float:
        wl = self.wl
        t0 = time.perf_counter()
        self.oracle.sparse_attn(self.q, self.cache, wl.kind, wl.d_nope, wl.d_rope, wl.d_v, wl.indices, wl.sm_scale,
                                block_table=wl.block_table, page_size=wl.page_size, req_of_token=wl.req_of_token,
                                tokens=np.asarray(tokens, dtype=np.int64))
        return time.perf_counter() - t0

    def sample(self, seconds: float):
        """tokens/s on a bounded sample sized to about ``seconds`` of host time."""
        probe = self.order[: min(self.wl.T, max(self.threads, 8))]
        per_tok = self.run(probe) / len(probe)
        n = int(min(self.wl.T, max(len(probe), seconds / max(per_tok, 1e-9))))
        dt = self.run(self.order[:n])
        return n / dt, min(self.threads, n), f"{n} of {self.wl.T} tokens (seeded random subset), full top-k lists"


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo; 'unknown' where neither names one)."""
    try:
        r = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10)
        for line in r.stdout.splitlines():
            k, _, v = line.partition(":")
            if k.strip() == "Model name" and v.strip():
                return v.strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                k, _, v = line.partition(":")
                if k.strip() == "model name" and v.strip():
                    return v.strip()
    except OSError:
        pass
    import platform

    return platform.machine() or "unknown"


def measure(args, wl, rank, world, device, config=None):
    """Times one workload (kernel-only and end to end) and returns its JSON line on rank 0."""
    import torch

    config = args.config if config is None else config
    work = algorithmic_work(wl)
    r = run_gpu(args, wl, rank, world, device, config)
    if rank != 0:
        return None
    hbm, bf16, bf16_sus, peak_src = _peaks()
    ms_per_step = r["total_ms"] / args.steps
    value = job_value(world, wl.T, args.steps, r["total_ms"])
    roof = roofline(work, ms_per_step / 1000.0, hbm, bf16)
    roof.update({"traffic": _recorded_traffic(wl.name), "peak_source": peak_src,
                 "algorithmic_bytes_per_launch": work["bytes"], "unique_bytes_per_launch": work["unique_bytes"],
                 "flops_per_launch": work["flops"]})
    # the same achieved figure against the GB300 nominal peaks (HBM3e 7.9 TB/s, dense bf16 2.25 PFLOP/s)
    nominal = NOMINAL_HBM_GBS if roof["bound"] == "hbm" else NOMINAL_BF16_TFLOPS
    roof["frac_of_nominal"] = roof["achieved"] / nominal
    roof["nominal_peak"] = nominal
    cpu_v, cores, sample = OracleRunner(wl).sample(args.cpu_seconds)
    metric = METRIC if config == 3 else f"sparse-attn tokens/s ({wl.name})"
    return {
        "metric": metric, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        # the products' operand type: e4m3 codes (FP8 cache: both products on the tensor core's
        # 8-bit kind, fp32 accumulation) or bf16
        "vs_baseline": None, "dtype": "e4m3" if wl.kind == 1 else "bf16", "data": "synthetic",
        "config": workload_config(wl, work),
        "roofline": roof,
        "cpu_baseline": {"value": cpu_v, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample,
                         "cpu": cpu_model()},
        "e2e": {"value": world * wl.T / (r["e2e_pipe_ms"] / 1000.0), "unit": "tokens/s", "h2d_bytes_per_step": r["h2d"],
                "mode": "pipelined: step i+1's inputs copied in and step i-1's output read back while step i "
                        "computes (two copy streams, two buffer sets), index sets rotating among 4",
                "serial_value": world * wl.T / (r["e2e_ms"] / 1000.0),
                "d2h_bytes_per_step": r["d2h"]},
        "gpu_launches": args.steps * kernels_per_call(wl, torch.cuda.get_device_properties(device).multi_processor_count),
        "clocks": r["clocks"],
        "step_ms": {"median": statistics.median(r["times"]), "min": min(r["times"]), "max": max(r["times"])},
    }


def measure_latency(args, wl, device):
    """Device time of one call on a small batch, L2 flushed before each: replayed from a CUDA
    graph (the kernels alone, no host marshalling between the events) and launched directly
    (host marshalling included, as one isolated call sees it)."""
    import torch

    import dsa_sparse_attention_mla_gb300 as dsa

    q, cache, idx, bt, req = build_device_inputs(wl, device)
    out = torch.empty((wl.T, wl.H, wl.d_v), dtype=torch.bfloat16, device=device)
    err = torch.zeros(1, dtype=torch.int32, device=device)
    ws = torch.zeros(dsa.dsa_sparse_attn_workspace_size(wl.d_v), dtype=torch.uint8, device=device)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    s = torch.cuda.Stream(device)

    def step():
        dsa.dsa_sparse_attn(q, cache, wl.kind, idx, wl.sm_scale, d_nope=wl.d_nope, d_rope=wl.d_rope, d_v=wl.d_v,
                            block_table=bt, page_size=wl.page_size, req_of_token=req, out=out, workspace=ws,
                            error_word=err)

    n = max(10, min(args.steps, 200))
    with torch.cuda.stream(s):
        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize(device)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            step()
        torch.cuda.synchronize(device)
        res = {}
        for mode in ("graph", "launch"):
            ts = []
            for i in range(n):
                flush.fill_(i & 0xFF)
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(s)
                g.replay() if mode == "graph" else step()
                b.record(s)
                torch.cuda.synchronize(device)
                ts.append(a.elapsed_time(b) * 1000.0)
            res[mode] = statistics.median(ts)
    if err.item() != 0:
        raise RuntimeError(f"device error word {err.item()} during the latency measurement")
    work = algorithmic_work(wl)
    return {"workload": wl.name, "tokens": wl.T, "us_per_call_graph": res["graph"], "us_per_call_launch": res["launch"],
            "calls": n, "roofline_us": max(work["unique_bytes"] / (_peaks()[0] * 1e9),
                                           work["flops"] / (_peaks()[1] * 1e12)) * 1e6,
            "gpu_launches_per_call": kernels_per_call(wl, torch.cuda.get_device_properties(device).multi_processor_count)}


def workload_config(wl, work):
    return {"workload": wl.name, "tokens_per_step": wl.T, "heads": wl.H, "d_nope": wl.d_nope, "d_rope": wl.d_rope,
            "d_v": wl.d_v, "topk": wl.topk, "valid_entries": work["n_valid"],
            "cache": f"fp8_{wl.d_nope + 4 * (wl.d_nope // 128) + 2 * wl.d_rope}B" if wl.kind else "bf16",
            "slots": wl.num_slots, "page_size": wl.page_size or None,
            "l2": f"{L2_FLUSH_BYTES >> 20} MB buffer written between timed steps (outside the events)"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--op", default="attn", choices=["attn", "requant", "proj", "topk", "pack", "dequant"],
                    help="requant: time dsa_gather_requant on the decode workload's rows instead; proj: the "
                         "FP8 block-scaled projection GEMM; topk: the top-k selection at decode and prefill shapes; "
                         "pack / dequant: the cache pack and the gather-dequant helper")
    ap.add_argument("--no-prefill", dest="prefill", action="store_false",
                    help="with the default decode workload, skip the second (T=8192 prefill) measurement")
    ap.add_argument("--no-extra", dest="extra", action="store_false",
                    help="with the default decode workload, skip the 512+64 control and small-batch latency")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    from dsa_sparse_attention_mla_gb300 import workloads as W

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    wl = W.config(args.config, seed=0)
    metric = METRIC if args.config == 3 else f"sparse-attn tokens/s ({wl.name})"

    if args.impl == "reference":
        # The reference arm is the CPU oracle as it stands, on rank 0 only; each step runs a
        # bounded sample of the workload's tokens so the whole run stays within a few minutes.
        if rank != 0:
            return
        runner = OracleRunner(wl)
        per_tok = runner.run(runner.order[:1])
        budget = 150.0
        n = int(max(1, min(wl.T, budget / ((args.steps + args.warmup) * max(per_tok, 1e-9)))))
        tot_t, tot_n = 0.0, 0
        for i in range(args.warmup + args.steps):
            toks = np.roll(runner.order, -i * n)[:n]
            dt = runner.run(toks)
            if i >= args.warmup:
                tot_t += dt
                tot_n += n
        v = tot_n / tot_t
        cores = min(runner.threads, n)
        sample = f"{n} of {wl.T} tokens per step (seeded rotation), full top-k lists"
        line = {"impl": "reference", "metric": metric, "value": v, "unit": "tokens/s", "n_gpus": 0,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * wl.T / v,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": workload_config(wl, algorithmic_work(wl)),
                "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample,
                                 "cpu": cpu_model()},
                "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import torch

    if world > 1:
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    device = torch.device("cuda", local_rank)
    import __graft_entry__

    __graft_entry__.build() if rank == 0 else None
    if world > 1:
        torch.distributed.barrier()
    if args.op in ("requant", "proj", "topk", "pack", "dequant"):
        if rank == 0:
            {"requant": run_requant, "proj": run_proj, "topk": run_topk, "pack": run_cache_ops,
             "dequant": run_cache_ops}[args.op](args, device)
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    line = measure(args, wl, rank, world, device)
    if args.config == 3 and args.prefill:
        # the second headline workload, timed in the same run (every rank takes part in its
        # barriers): BF16 causal prefill, T=8192
        wl4 = W.config(4, seed=0)
        sub = measure(args, wl4, rank, world, device, config=4)
        if line is not None and sub is not None:
            line["prefill"] = {k: sub[k] for k in ("metric", "value", "unit", "ms_per_step", "dtype", "config",
                                                   "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks",
                                                   "step_ms")}
    if args.config == 3 and args.extra:
        # the 512+64 control (FP8 656-byte rows, T=1024), timed like the headline workload
        wl5 = W.config(5, seed=0)
        sub = measure(args, wl5, rank, world, device, config=5)
        if line is not None and sub is not None:
            line["control"] = {k: sub[k] for k in ("metric", "value", "unit", "ms_per_step", "dtype", "config",
                                                   "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks",
                                                   "step_ms")}
        # small batches (T=17 BF16 direct, T=8 FP8 paged): device time per call
        if rank == 0 and line is not None:
            line["small_batch"] = [measure_latency(args, W.config(c, seed=0), device) for c in (1, 2)]
    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
