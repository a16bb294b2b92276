#!/usr/bin/env python3
"""Benchmark of the structured-mask attention forward on GB300.

One step = one pass of the whole hot path over one batch: build the block
mask (tile summaries, exact classification, compacted lists, longest-first
order) once, then run the attention forward of every layer of the step
(``--layers``, default 64; the layers of a model share one mask, which is
built once per step and reused, the xorl issue's "Proposed work", item 3), on
inputs already resident in HBM.  Every layer reads the workload's Q, K, V
(805 MB on the default workload, larger than L2).  Metric: effective TFLOP/s
counting only unmasked score FLOPs, 4*D*H*nnz per forward (2*D for q.k and
2*D for p.v per visible pair), and its fraction of the measured dense bf16
tensor peak.

After the forward's timed steps, the backward (dQ, dK, dV for a seeded
upstream gradient, on the forward's own O and LSE) is timed back to back for
at least a second and reported under "backward", in effective TFLOP/s
(10*D*H*nnz, the usual 2.5x the forward's count); ``--no-backward`` skips it.
``per_config`` times the forward (and backward) of the other block-mask
workloads (1: one 64-token causal sequence in fp32, forward only, on the
CUDA-core path; 2: varlen causal, 3: shared prefix, 4: strip thinking), each
back to back for at least a second with its own clock samples.

Default workload: the 32768-token causal+document mask (12 documents, H=32,
D=128, bf16), the largest configuration.  ``--impl reference`` times the fp64
CPU oracle on the host cores on a bounded sample of the same workload.
Multi-GPU (torchrun): every rank runs an independent replica of the workload
(weak scaling); the forward has no exchange step.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "masked attn fwd TFLOP/s (unmasked FLOPs) & % of GB300 bf16 tensor peak"
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(value: float, ws: int) -> float:
    """Max over ranks (the job finishes when the slowest rank does)."""
    if ws == 1:
        return value
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_throughput(flops_per_step_per_rank: float, ws: int, seconds_per_step: float) -> float:
    """Whole-job TFLOP/s: every rank's units divided by the slowest rank's time."""
    return flops_per_step_per_rank * ws / seconds_per_step / 1e12


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


class ClockSampler:
    """nvidia-smi samples during the timed region (SM clock, reasons)."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]
        return False

    def summary(self, window=None):
        """Median SM clock and the throttle reasons seen; ``window`` = (t0, t1)
        in host wall-clock seconds keeps only the samples taken inside it (the
        timed region)."""
        import datetime
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in getattr(self, "lines", []):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                t = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                clk, top = float(parts[2]), float(parts[3])
            except ValueError:
                continue
            if window is not None and not (window[0] <= t <= window[1]):
                continue
            sm.append(clk)
            mx = top
            for name, val in zip(names, parts[6:10]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def workload_config(w, nnz, extra=None):
    cfg = {"workload": w.name, "kind": w.kind, "total_tokens": w.total_tokens,
           "batch": w.batch, "seqlens": w.seqlens, "num_heads": w.num_heads,
           "head_dim": w.head_dim, "unmasked_pairs_per_head": nnz,
           "flops_per_step": 4 * w.head_dim * w.num_heads * nnz,
           "l2": "inputs larger than L2 (Q+K+V = %.0f MB)" %
                 (3 * w.total_tokens * w.num_heads * w.head_dim * 2 / 1e6)}
    if extra:
        cfg.update(extra)
    return cfg


# Visible (query, key) pairs per head of each workload: the nnz of the metric's
# 4*D*H*nnz.  Closed forms: workload 2 and 5 are sums of L(L+1)/2 over the
# (seeded) sequence / document lengths; workload 3 is P(P+1)/2 + n(sP + s(s+1)/2)
# with P=2048, n=16, s=512; workload 4 is 8 L(L+1)/2 + L*384*(0+1+...+7) with
# L=1152.  tests/test_bench_host.py checks each against the oracle's count.
UNMASKED_PAIRS = {1: 2080, 2: 8_172_171, 3: 20_976_640, 4: 17_699_328, 5: 67_979_834,
                  6: 20_977_152, 7: 16_334_146, 8: 53_960_250}


def count_pairs(w, c):
    return UNMASKED_PAIRS[c]


# the fp32 path runs on CUDA cores: 152 SMs x 128 fp32 lanes x 2 FLOP per FFMA x 2.07 GHz
FP32_FFMA_PEAK = 152 * 128 * 2 * 2.07e9 / 1e12


# kernels the library launches: a block-mask build (five kernels) and the backward
BUILD_LAUNCHES = 5
BWD_KERNELS = ["bwd_zero_kernel", "bwd_prep_kernel", "bwd_mult_kernel", "attn_bwd_kernel", "bwd_dq_convert_kernel"]


TRAFFIC_PROFILE = os.path.join(ROOT, "profiles", "attn_fwd_bf16_causal_document_32k_h8_full.md")
FWD_SOURCE = os.path.join(ROOT, "block_sparse_masked_mask_gb300", "csrc", "attn_fwd_bf16.cu")


def profiled_traffic(workload: int, num_heads: int):
    """DRAM bytes per forward launch from the committed ncu capture (8 heads of
    the 32k causal+document mask), scaled by the head count; None when the
    workload differs or the kernel source changed since the capture."""
    import hashlib
    if workload != 5 or not os.path.exists(TRAFFIC_PROFILE):
        return None, None
    fields = {}
    with open(TRAFFIC_PROFILE) as f:
        for line in f:
            if ":" in line and not line.startswith(("|", "#", " ", "*")):
                k, _, v = line.partition(":")
                fields[k.strip()] = v.strip()
    with open(FWD_SOURCE, "rb") as f:
        sha = hashlib.sha256(f.read()).hexdigest()
    if fields.get("source_sha256") != sha:
        return None, None
    heads = int(fields["heads"])
    t = int(fields["traffic_bytes_per_launch_h8"]) * num_heads / heads
    return t, f"ncu dram__bytes_read.sum + dram__bytes_write.sum at {heads} heads, scaled to {num_heads}"


def cpu_baseline(w, budget_s: float, seed: int = 0):
    """The fp64 oracle on the host cores over a bounded sample of rows of head 0."""
    import oracle
    rng = np.random.default_rng(seed)
    T = w.total_tokens
    t0 = time.perf_counter()
    flops = 0
    rows_done = 0
    block = 256
    qh, kh, vh = w.q[:, :1], w.k[:, :1], w.v[:, :1]
    while time.perf_counter() - t0 < budget_s:
        r0 = int(rng.integers(0, max(1, T - block)))
        rows = np.arange(r0, min(T, r0 + block))
        oracle.attention(qh, kh, vh, w.kind, w.cu_seqlens, w.meta(), rows=rows)
        # visible pairs of the sampled rows
        for b in range(w.batch):
            s0, s1 = int(w.cu_seqlens[b]), int(w.cu_seqlens[b + 1])
            sel = rows[(rows >= s0) & (rows < s1)]
            if len(sel):
                m = oracle.sequence_mask(w.kind, w.cu_seqlens, b, w.meta(), rows=sel - s0)
                flops += 4 * w.head_dim * int(m.sum())
        rows_done += len(rows)
    el = time.perf_counter() - t0
    return {"value": flops / el / 1e12, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{rows_done} query rows of head 0 in random {block}-row blocks, "
                      f"{el:.1f} s of fp64 numpy work (BLAS thread pool over all cores)"}


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    from block_sparse_masked_mask_gb300 import workloads as W
    w = W.make_workload(args.workload, tensors=True)
    nnz = count_pairs(w, args.workload)
    import oracle
    rng = np.random.default_rng(0)
    block = 256
    qh, kh, vh = w.q[:, :1], w.k[:, :1], w.v[:, :1]

    def step():
        r0 = int(rng.integers(0, max(1, w.total_tokens - block)))
        rows = np.arange(r0, min(w.total_tokens, r0 + block))
        oracle.attention(qh, kh, vh, w.kind, w.cu_seqlens, w.meta(), rows=rows)
        f = 0
        for b in range(w.batch):
            s0, s1 = int(w.cu_seqlens[b]), int(w.cu_seqlens[b + 1])
            sel = rows[(rows >= s0) & (rows < s1)]
            if len(sel):
                f += 4 * w.head_dim * int(oracle.sequence_mask(w.kind, w.cu_seqlens, b, w.meta(),
                                                                rows=sel - s0).sum())
        return f

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    flops = sum(step() for _ in range(args.steps))
    el = time.perf_counter() - t0
    val = flops / el / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": workload_config(w, nnz, {"sample": f"each step: {block} random query rows of head 0"}),
        "cpu_baseline": {"value": val, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                         "sample": f"{args.steps} steps of {block} query rows of head 0"},
        "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def time_loop(fn, stream, dev, min_seconds: float, batch: int = 8, batch_ms: float = 5.0):
    """Run ``fn`` back to back for at least ``min_seconds`` of device time, in
    batches bracketed by CUDA events on ``stream``; returns the per-call device
    times (ms, one batch mean per entry), the call count and the host
    wall-clock window of the timed calls.  A batch is sized to about
    ``batch_ms`` of device time (at least ``batch`` calls), so that the host's
    time to issue the first call of a batch, which the start event sees as
    device idle time, is a small part of it even for short calls."""
    per_call, calls = [], 0
    torch.cuda.synchronize(dev)
    # size the batches from one untimed batch
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(batch):
        fn()
    e1.record(stream)
    e1.synchronize()
    est = e0.elapsed_time(e1) / batch
    batch = max(batch, min(512, int(batch_ms / max(est, 1e-3))))
    t0 = time.time()
    while True:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(batch):
            fn()
        e1.record(stream)
        e1.synchronize()
        per_call.append(e0.elapsed_time(e1) / batch)
        calls += batch
        if sum(per_call) * batch >= min_seconds * 1e3:
            break
    return per_call, calls, (t0, time.time())


def time_workload(c, dev, stream, peak, min_seconds, backward=True):
    """Forward (and backward) of workload ``c`` back to back for at least
    ``min_seconds`` each, mask built once, with clock samples of each timed
    region."""
    from block_sparse_masked_mask_gb300 import api
    from block_sparse_masked_mask_gb300 import workloads as W
    w = W.make_workload(c, tensors=True)
    nnz = count_pairs(w, c)
    flops = 4 * w.head_dim * w.num_heads * nnz
    dm = w.device_meta(dev)
    mkw = w.api_kwargs(dm)
    q, k, v = w.q.to(dev), w.k.to(dev), w.v.to(dev)
    bm = api.attn_block_mask_build(w.kind, dm["cu_seqlens"], w.total_tokens, w.max_seqlen, **mkw)
    out, lse = api.attn_fwd(q, k, v, bm, w.kind, dm["cu_seqlens"], w.max_seqlen, **mkw)

    def fwd():
        api.attn_fwd(q, k, v, bm, w.kind, dm["cu_seqlens"], w.max_seqlen, out=out, lse=lse, **mkw)

    for _ in range(5):
        fwd()
    with ClockSampler(dev.index) as clk:
        time.sleep(0.3)
        ms, calls, win = time_loop(fwd, stream, dev, min_seconds)
    fwd_ms = sum(ms) / len(ms)
    fp32 = w.dtype == torch.float32
    fpeak = FP32_FFMA_PEAK if fp32 else peak
    res = {"workload": w.name, "kind": w.kind, "dtype": "f32" if fp32 else "bf16",
           "total_tokens": w.total_tokens,
           "num_heads": w.num_heads, "head_dim": w.head_dim, "unmasked_pairs_per_head": nnz,
           "fwd_ms_mean": fwd_ms, "fwd_calls_timed": calls,
           "fwd_tflops": flops / fwd_ms / 1e9, "fwd_frac": flops / fwd_ms / 1e9 / fpeak,
           "fwd_clocks": clk.summary(win)}
    if fp32:
        res["fwd_peak"] = ("CUDA-core FFMA, derived: 152 SMs x 128 fp32 lanes x 2 FLOP x 2.07 GHz = "
                           f"{FP32_FFMA_PEAK:.1f} TFLOP/s; one 64-token sequence is launch-latency bound")
    if backward and not fp32:  # the backward is bf16 only
        do = W.grad_output(w, seed=1).to(dev)
        gq, gk, gv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        bws = torch.empty(api.attn_bwd_workspace_size(bm, w.num_heads, w.head_dim), dtype=torch.uint8, device=dev)

        def bwd():
            api.attn_bwd(q, k, v, out, lse, do, bm, w.kind, dm["cu_seqlens"], w.max_seqlen,
                         dq=gq, dk=gk, dv=gv, workspace=bws, **mkw)

        for _ in range(3):
            bwd()
        with ClockSampler(dev.index) as clk:
            time.sleep(0.3)
            ms, calls, win = time_loop(bwd, stream, dev, min_seconds)
        bwd_ms = sum(ms) / len(ms)
        res.update({"bwd_ms_mean": bwd_ms, "bwd_calls_timed": calls,
                    "bwd_tflops_effective": 2.5 * flops / bwd_ms / 1e9,
                    "bwd_frac_effective": 2.5 * flops / bwd_ms / 1e9 / peak,
                    "bwd_clocks": clk.summary(win)})
    status = api.attn_get_status(bm)
    if status != 0:
        raise RuntimeError(f"workload {c}: device status {api.attn_status_string(status)}")
    return res


def run_ours(args):
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from block_sparse_masked_mask_gb300 import api
    from block_sparse_masked_mask_gb300 import workloads as W

    w = W.make_workload(args.workload, tensors=True)
    if args.heads:
        w.num_heads = args.heads
        w.q, w.k, w.v = (t[:, :args.heads].contiguous() for t in (w.q, w.k, w.v))
    nnz = count_pairs(w, args.workload)
    flops_fwd = 4 * w.head_dim * w.num_heads * nnz
    L = args.layers
    flops = flops_fwd * L  # per step
    dm = w.device_meta(dev)
    q, k, v = w.q.to(dev), w.k.to(dev), w.v.to(dev)
    T, H, D = q.shape
    out = torch.empty_like(q)
    lse = torch.empty((H, T), dtype=torch.float32, device=dev)
    ws_bytes = api.attn_block_mask_workspace_size(w.batch, T, w.max_seqlen)
    workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    mkw = w.api_kwargs(dm)

    def step(ev=None):
        """One mask build, then the forward of each of the step's layers."""
        bm = api.attn_block_mask_build(w.kind, dm["cu_seqlens"], T, w.max_seqlen,
                                       workspace=workspace, **mkw)
        if ev is not None:
            ev.record(stream)
        for _ in range(L):
            api.attn_fwd(q, k, v, bm, w.kind, dm["cu_seqlens"], w.max_seqlen, out=out, lse=lse, **mkw)
        return bm

    for _ in range(args.warmup):
        bm = step()
    status = api.attn_get_status(bm)
    if status != 0:
        raise RuntimeError(f"device status {api.attn_status_string(status)}")
    hdr = bm.header().tolist()

    # ---- timed region: K steps, events on the launching stream
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    mids = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(ws)
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        time.sleep(0.3)
        t_wall0 = time.time()
        for i in range(args.steps):
            starts[i].record(stream)
            step(mids[i])
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
        t_wall1 = time.time()
    barrier(ws)
    total_ms = starts[0].elapsed_time(ends[-1])
    fwd_ms = [mids[i].elapsed_time(ends[i]) / L for i in range(args.steps)]
    build_ms = [starts[i].elapsed_time(mids[i]) for i in range(args.steps)]
    sec_per_step = reduce_max(total_ms / 1e3 / args.steps, ws)
    value = aggregate_throughput(flops, ws, sec_per_step)
    status = api.attn_get_status(bm)
    if status != 0:
        raise RuntimeError(f"device status {api.attn_status_string(status)}")

    peaks, peak_kind = load_peaks()
    fwd_avg_s = sum(fwd_ms) / len(fwd_ms) / 1e3
    achieved = flops_fwd / fwd_avg_s / 1e12
    # The forward is timed inside a long step (back-to-back launches over a
    # second or more, under the power cap): the sustained tensor peak is its
    # denominator; a short run (well under a second) is compared with the burst
    # peak.  Both fractions are reported.
    burst = float(peaks["bf16_tflops"])
    sustained = float(peaks.get("bf16_tflops_sustained", burst))
    long_step = total_ms >= 1000.0
    peak = sustained if long_step else burst
    roofline = {"bound": "tensor", "kernel": "attn_fwd_bf16_kernel<128, false>", "achieved": achieved,
                "peak": peak, "unit": UNIT, "frac": achieved / peak,
                "peak_source": f"{peak_kind} bf16_tflops" + ("_sustained (timed region "
                               f"{total_ms / 1e3:.2f} s)" if long_step else " (burst)"),
                "frac_of_burst": achieved / burst,
                "frac_of_sustained": achieved / sustained,
                "traffic": None}
    traffic, traffic_src = profiled_traffic(args.workload, w.num_heads)
    if traffic is not None:
        roofline["traffic"] = traffic
        roofline["traffic_source"] = traffic_src

    # ---- the backward on the same workload: dQ, dK, dV of the forward just
    # timed, for a seeded upstream gradient, inputs resident, back to back for
    # at least a second
    bwd = None
    if not args.no_backward:
        do = W.grad_output(w, seed=1).to(dev)
        gq, gk, gv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        bws = torch.empty(api.attn_bwd_workspace_size(bm, H, D), dtype=torch.uint8, device=dev)

        def bwd_step():
            api.attn_bwd(q, k, v, out, lse, do, bm, w.kind, dm["cu_seqlens"], w.max_seqlen,
                         dq=gq, dk=gk, dv=gv, workspace=bws, **mkw)

        for _ in range(args.warmup):
            bwd_step()
        with ClockSampler(local) as bclk:
            time.sleep(0.3)
            bwd_ms, bwd_calls, bwin = time_loop(bwd_step, stream, dev, args.min_seconds)
        status = api.attn_get_status(bm)
        if status != 0:
            raise RuntimeError(f"device status {api.attn_status_string(status)}")
        bwd_s = sum(bwd_ms) / len(bwd_ms) / 1e3
        eff = 2.5 * flops_fwd / bwd_s / 1e12
        bwd = {"ms_mean": bwd_s * 1e3, "ms_min_batch": min(bwd_ms), "calls_timed": bwd_calls,
               "tflops_effective": eff, "frac_effective": eff / peak,
               "flops_effective_per_step": 2.5 * flops_fwd,
               "flop_counting": "effective = 10*D*H*nnz (five products per visible tile pair: "
                                "S, dP, dV, dK, dQ; the usual 2.5x the forward)",
               "kernels": BWD_KERNELS,
               "workspace_bytes": bws.numel(),
               "clocks": bclk.summary(bwin)}

    # ---- the other block-mask workloads, each timed for at least a second
    per_config = None
    if rank == 0 and ws == 1 and not args.no_per_config and args.workload == 5 and not args.heads:
        per_config = {str(c): time_workload(c, dev, stream, peak, args.min_seconds,
                                            backward=not args.no_backward) for c in (1, 2, 3, 4)}

    # ---- end to end through the public API with host buffers.  Every step copies
    # its inputs (Q, K, V and the mask metadata) from pinned host memory and reads
    # O and LSE back.  Two streams and two device buffer sets: the host->device
    # copy of step i+1 runs while step i builds its mask, runs the forward and
    # copies its result back.  (One forward per step: each layer of a real model
    # has its own inputs.)
    pin = lambda t: t.pin_memory()
    hq, hk, hv = pin(w.q), pin(w.k), pin(w.v)
    hmeta = {k2: (None if t is None else pin(t.cpu())) for k2, t in dm.items()}
    ho = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    hl = [torch.empty(lse.shape, dtype=lse.dtype).pin_memory() for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in [hq, hk, hv] + [t for t in hmeta.values() if t is not None])
    d2h = ho[0].numel() * ho[0].element_size() + hl[0].numel() * hl[0].element_size()
    dq = [torch.empty_like(q) for _ in range(2)]
    dk = [torch.empty_like(k) for _ in range(2)]
    dv = [torch.empty_like(v) for _ in range(2)]
    dmeta = [{k2: (None if t is None else torch.empty_like(t, device=dev)) for k2, t in hmeta.items()}
             for _ in range(2)]
    dout = [out, torch.empty_like(out)]
    dlse = [lse, torch.empty_like(lse)]
    dws = [workspace, torch.empty_like(workspace)]
    copy_s, comp_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    h2d_done = [torch.cuda.Event() for _ in range(2)]
    comp_done = [torch.cuda.Event() for _ in range(2)]

    def e2e_step(i):
        b = i & 1
        with torch.cuda.stream(copy_s):
            copy_s.wait_event(comp_done[b])  # the step that last read these buffers is done
            dq[b].copy_(hq, non_blocking=True)
            dk[b].copy_(hk, non_blocking=True)
            dv[b].copy_(hv, non_blocking=True)
            for k2, t in hmeta.items():
                if t is not None:
                    dmeta[b][k2].copy_(t, non_blocking=True)
            h2d_done[b].record(copy_s)
        with torch.cuda.stream(comp_s):
            comp_s.wait_event(h2d_done[b])
            m = dmeta[b]
            mk = w.api_kwargs(m)
            bm2 = api.attn_block_mask_build(w.kind, m["cu_seqlens"], T, w.max_seqlen,
                                            workspace=dws[b], **mk)
            api.attn_fwd(dq[b], dk[b], dv[b], bm2, w.kind, m["cu_seqlens"], w.max_seqlen,
                         out=dout[b], lse=dlse[b], **mk)
            ho[b].copy_(dout[b], non_blocking=True)
            hl[b].copy_(dlse[b], non_blocking=True)
            comp_done[b].record(comp_s)

    e2e_steps = max(1, min(args.steps, 10))
    for i in range(2):
        e2e_step(i)
    barrier(ws)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    copy_s.wait_event(e0)
    comp_s.wait_event(e0)
    for i in range(e2e_steps):
        e2e_step(i)
    stream.wait_stream(copy_s)
    stream.wait_stream(comp_s)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_sec = reduce_max(e0.elapsed_time(e1) / 1e3 / e2e_steps, ws)
    e2e = {"value": aggregate_throughput(flops_fwd, ws, e2e_sec), "unit": UNIT,
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_sec * 1e3,
           "pipeline": "two streams: the host->device copy of step i+1 overlaps step i; "
                       "one mask build and one forward per step"}

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, args.cpu_seconds)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": sec_per_step * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": workload_config(w, nnz, {
                "parallelism": f"replicas{ws}",
                "layers_per_step": L,
                "step": f"one block-mask build + {L} forward passes sharing it",
                "flops_per_step": flops,
                "tiles_empty_partial_full": hdr[4:7],
                "skipped_tile_ratio": hdr[4] / max(1, sum(hdr[4:7])),
                "timed_region_s": total_ms / 1e3,
                "fwd_ms_mean": sum(fwd_ms) / len(fwd_ms), "fwd_ms_min_step": min(fwd_ms),
                "build_ms_mean": sum(build_ms) / len(build_ms),
                "fwd_tflops": achieved, "pct_of_peak_fwd": 100 * achieved / peak}),
            "roofline": roofline,
            "cpu_baseline": cpu,
            "clocks": clk.summary((t_wall0, t_wall1)),
            "e2e": e2e,
            "gpu_launches": (BUILD_LAUNCHES + L) * args.steps,
            "backward": bwd,
            "per_config": per_config,
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=5, choices=[2, 3, 4, 5, 6, 7, 8],
                    help="workload number (2-5: the bf16 block-mask workloads; 6: strip-thinking with "
                         "duplicated answers; 7: non-causal varlen; 8: dense causal+document+padding)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="time budget of the oracle CPU-baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-backward", action="store_true",
                    help="skip the backward measurement that follows the forward's")
    ap.add_argument("--heads", type=int, default=None,
                    help="override the head count (a smaller case of the same mask for profiling)")
    ap.add_argument("--layers", type=int, default=64,
                    help="forward passes per step, all sharing the step's one mask build")
    ap.add_argument("--min-seconds", type=float, default=1.0,
                    help="least device time of each back-to-back timing (backward, per_config)")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the timings of workloads 1-4")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        return run_reference(args)
    from block_sparse_masked_mask_gb300 import build as _b
    _b.ensure_built()
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
