#!/usr/bin/env python3
"""Benchmark: causal flash-attention forward + backward on one GB300.

One step = one pass of the whole hot path over one batch: the forward
(xfa_fwd) and the three backward stages (D pre-pass, backward kernel, dQ
conversion) on the S=8192, bh=32, hd=128 bf16 workload with inputs resident
in HBM.  Each launch is bracketed by CUDA events on the launching stream.
The inputs (4 x 64 MiB) are larger than L2 (129 MB); no extra flush.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

``--impl reference`` times the CPU oracle (fp64, all host cores) on a bounded
sample of the same workload.  Prints one JSON line.
"""
from __future__ import annotations

import argparse
import csv
import io
import json
import math
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from bwd_xfa_fwd_gb300 import inputs  # noqa: E402

METRIC = "causal attn fwd / bwd TFLOP/s at 1 GB300 and fraction of bf16 tensor peak"
FAMILIES = {"auto": 0, "simt": 1, "tcgen05": 2, "tcgen05_det": 3}   # xfa_impl codes
WORKLOAD_ID = 5
DROPOUT_SEED = 0x5EED   # seed of the optional dropout mode (--dropout)
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


KERNEL_SOURCES = {
    "tc_fwd": ("bwd_xfa_fwd_gb300/csrc/tc_fwd.cu", "bwd_xfa_fwd_gb300/csrc/ptx.cuh"),
    "tc_bwd": ("bwd_xfa_fwd_gb300/csrc/tc_bwd.cu", "bwd_xfa_fwd_gb300/csrc/ptx.cuh"),
    "rowdot": ("bwd_xfa_fwd_gb300/csrc/aux.cu", "bwd_xfa_fwd_gb300/csrc/ptx.cuh"),
}


def source_hash(name):
    """Hash of the code of a kernel's sources: // comments, blank lines and indentation are left
    out, so an edit of the comments or the layout does not void a recorded capture, any edit of
    the code does."""
    import hashlib
    import re
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[name]:
        with open(os.path.join(ROOT, rel)) as f:
            code = [re.sub(r"//.*$", "", line).strip() for line in f]
        h.update("\n".join(line for line in code if line).encode())
    return h.hexdigest()[:16]


def recorded_traffic(name, workload):
    """DRAM bytes per launch recorded by an ncu capture (profiles/dram_traffic.json),
    or None when there is none for this workload or the kernel source changed since."""
    try:
        with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    e = rec.get(workload, {}).get(name)
    if not e or e.get("source_hash") != source_hash(name):
        return None
    return e["dram_bytes_per_launch"]


def measure_graph(torch, step, K, flops):
    """The same step captured once in a CUDA graph and replayed K times: the library neither
    allocates nor synchronises, so a whole forward + backward is capturable, and replaying
    it removes the per-call host cost that dominates small problems."""
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()                       # warm on a side stream before capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        step()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(K):
        g.replay()
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / K
    return {"ms_per_step": ms, "value": flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "replays": K}


def max_over_ranks(value: float, device=None) -> float:
    """The largest `value` over all ranks of the default process group (the
    value itself when no group is initialised)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), int(
        os.environ.get("LOCAL_RANK", "0"))


L2_BYTES = 129 * 10**6
# Steps of the end-to-end leg, whatever --steps is: the first upload and the last download
# are not overlapped with compute, so a short leg would measure the pipeline's fill and drain.
E2E_STEPS = 64
SIMT_FMA_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12   # the SIMT kernels' arithmetic bound


def data_note(w):
    """The `data` entry of a JSON line: how the workload's inputs are drawn."""
    def n(std):
        return "N(0,1)" if std == 1.0 else f"N(0,{std:g}^2)"
    dist = (f"Q, K ~ {n(w.qk_std)}, V ~ {n(w.v_std)}, dO ~ {n(w.do_std)}" if (w.qk_std, w.v_std, w.do_std) != (1, 1, 1)
            else "Q, K, V, dO ~ N(0,1)")
    return (f"synthetic, seed {w.seed}: {dist}" + (", rounded to bf16" if w.dtype == "bf16" else "")
            + "; recipe in bwd_xfa_fwd_gb300/inputs.py")


def workload_config(w):
    elt = 2 if w.dtype == "bf16" else 4
    one = w.bh * w.S * w.hd * elt   # Q, K, V and dO, each streamed every step
    l2 = (f"inputs (4 x {one / 2**20:.0f} MiB {w.dtype}) larger than L2 (129 MB); no flush" if 4 * one > L2_BYTES
          else f"inputs (4 x {one / 2**20:.2f} MiB {w.dtype}) fit in L2 (129 MB): timed warm, a profiling case")
    return {"workload": w.name, "B": w.B, "H": w.H, "S": w.S, "hd": w.hd, "dtype": w.dtype,
            "scale": w.scale, "causal": True, "layout": "[bh,S,hd] row-major", "l2": l2}


def resolved_family(w, family):
    """The kernel family a call runs: 'tc' (bf16 tcgen05), 'tc_det', 'tf32x3' (fp32 tcgen05)
    or 'simt' -- as the library's dispatch resolves xfa_impl for this dtype and hd."""
    if family == "simt":
        return "simt"
    if w.dtype == "bf16" and w.hd in (64, 128):
        return "tc_det" if family == "tcgen05_det" else "tc"
    if w.dtype == "f32" and w.hd in (32, 64):
        return "tf32x3"
    return "simt"


def kernel_labels(w, fam):
    """(forward kernel, backward main-stage kernels, launches per step) of a family."""
    if fam == "tc":
        return f"tc_fwd_kernel<{w.hd}>", f"tc_bwd_kernel<{w.hd}>", 4          # fwd, prep, bwd, convert
    if fam == "tc_det":
        return f"tc_fwd_kernel<{w.hd}>", f"tc_bwd_kernel<{w.hd}> + tc_dq_kernel<{w.hd}>", 4
    if fam == "tf32x3":
        return f"tf_fwd_kernel<{w.hd}>", f"tf_bwd_kv_kernel<{w.hd}> + tf_bwd_q_kernel<{w.hd}>", 4
    conv = 1 if w.dtype == "bf16" else 0
    return f"simt_fwd_kernel<{w.dtype},{w.hd}>", f"simt_bwd_kernel<{w.dtype},{w.hd}>", 3 + conv


def tensor_peak(pk, pk_kind, fam):
    """(peak TFLOP/s, source) the family's contractions are measured against.  3xTF32 forms
    each fp32 product with three tf32 MMAs: its ceiling is the tf32 rate (the measured bf16
    rate times the nominal dense tf32 / bf16 ratio, 1.1 / 2.25 PFLOP/s) over three."""
    bf16 = float(pk["bf16_tflops"])
    if fam == "simt":
        return SIMT_FMA_TFLOPS, "FFMA: 152 SMs x 128 fp32 FMA/clk x 2 FLOP x 2.07 GHz (maximum SM clock)"
    if fam == "tf32x3":
        return bf16 * (1.1 / 2.25) / 3.0, f"{pk_kind} bf16_tflops x nominal tf32/bf16 (1.1/2.25) / 3 MMAs per product"
    return bf16, f"{pk_kind} bf16_tflops"


class ClockSampler:
    """nvidia-smi clock/throttle sampling while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.result = self._collect()

    def _collect(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = [r for r in csv.reader(io.StringIO(out)) if len(r) >= 9]
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.strip() == "Active"})
        loaded = [s for s in sm if smax and s > 0.5 * max(smax)] or sm
        return {"sm_mhz": float(np.median(loaded)) if loaded else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons, "samples": len(rows)}


def make_device_inputs(w, torch):
    x = inputs.workload_inputs(w)
    dev = {}
    for n in ("q", "k", "v", "dout"):
        if w.dtype == "f32":
            dev[n] = torch.from_numpy(np.ascontiguousarray(x[n].stored)).cuda()
        else:
            bits = torch.from_numpy(np.ascontiguousarray(x[n].stored).view(np.int16))
            dev[n] = bits.view(torch.bfloat16).cuda()
    return x, dev


def cpu_baseline_leg(w, heads=tuple(range(8))):
    """The oracle as it stands, on all host cores, on a bounded sample: the
    forward + backward of ``heads`` of the full-size workload."""
    import oracle
    x = inputs.workload_inputs(w, bh=max(heads) + 1)
    t0 = time.perf_counter()
    oracle.attention(x["q"].exact, x["k"].exact, x["v"].exact, x["dout"].exact, w.scale, heads=list(heads))
    dt = time.perf_counter() - t0
    flops = (w.fwd_flops() + w.bwd_flops()) * len(heads) / w.bh
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.threads(), "kind": "oracle",
            "sample": f"fwd+bwd of heads {list(heads)} of {w.name} (S={w.S}, hd={w.hd}), fp64, "
                      f"{dt:.1f} s; FLOPs counted by the causal convention", "seconds": dt}


REFERENCE_BUDGET_S = 120.0   # wall time the reference arm's warm-up + timed steps aim for
REFERENCE_CAL_ROWS = 2048    # rows of the calibration run (the time is extrapolated as S'^2)


def run_reference(args, w):
    """The reference arm: the oracle as it stands on the host cores, W warm-up and K timed
    steps.  A step is the forward + backward of a bounded sample of the workload: the
    first S' query rows and keys of one head (heads taken in turn), itself a causal
    problem of the same inputs.  S' (a multiple of 128, at most S) is sized from one
    calibration run so that the W + K steps take about REFERENCE_BUDGET_S seconds."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    K, W = args.steps, args.warmup
    x = inputs.workload_inputs(w)

    def sample(head, s_rows):
        return tuple(x[n].exact[head, :s_rows] for n in ("q", "k", "v", "dout"))

    t0 = time.perf_counter()
    oracle.attention_head(*sample(0, REFERENCE_CAL_ROWS), scale=w.scale)
    t_cal = time.perf_counter() - t0
    s_rows = int(REFERENCE_CAL_ROWS * math.sqrt(REFERENCE_BUDGET_S / ((K + W) * t_cal))) // 128 * 128
    s_rows = max(128, min(w.S, s_rows))
    for i in range(W):
        oracle.attention_head(*sample(i % w.bh, s_rows), scale=w.scale)
    t0 = time.perf_counter()
    for i in range(K):
        oracle.attention_head(*sample((W + i) % w.bh, s_rows), scale=w.scale)
    dt = time.perf_counter() - t0
    flops = 3.5 * 2.0 * s_rows * s_rows * w.hd   # fwd 2*S'^2*hd, bwd 2.5x, per sampled head
    value = flops * K / dt / 1e12
    sample_txt = (f"per step: fwd+bwd of the first {s_rows} query rows and keys of one head of {w.name} "
                  f"(heads in turn), fp64; {K} timed steps in {dt:.1f} s after {W} warm-up; FLOPs counted by the "
                  f"causal convention")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": K, "warmup": W, "ms_per_step": dt / K * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": data_note(w),
            "config": workload_config(w),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.threads(), "kind": "oracle",
                             "sample": sample_txt},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def measure_e2e(torch, binding, w, dev, ws, impl, K, flops, world):
    names_in = ("q", "k", "v", "dout")
    host_in = {n: dev[n].cpu().pin_memory() for n in names_in}
    bufs = []
    for _ in range(2):
        din = {n: torch.empty_like(dev[n]) for n in names_in}
        dout = (torch.empty_like(dev["q"]), torch.empty(dev["q"].shape[:-1], device="cuda", dtype=torch.float32),
                torch.empty_like(dev["q"]), torch.empty_like(dev["q"]), torch.empty_like(dev["q"]))
        hout = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in dout]
        bufs.append((din, dout, hout))
    wss = [ws, torch.empty_like(ws)]
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in bufs[0][2])
    up, comp, down = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()  # noqa: E731
    uploaded = [ev(), ev()]
    computed = [ev(), ev()]
    downloaded = [ev(), ev()]
    for e in computed + downloaded:
        e.record(torch.cuda.current_stream())

    def step(i):
        s = i % 2
        din, dout, hout = bufs[s]
        with torch.cuda.stream(up):
            up.wait_event(computed[s])              # step i-2 no longer reads these inputs
            for n in names_in:
                din[n].copy_(host_in[n], non_blocking=True)
            uploaded[s].record(up)
        with torch.cuda.stream(comp):
            comp.wait_event(uploaded[s])
            comp.wait_event(downloaded[s])          # step i-2's outputs have been read back
            o, l = binding.fwd(din["q"], din["k"], din["v"], w.scale, impl, out=dout[0], lse=dout[1])
            binding.bwd(din["q"], din["k"], din["v"], o, din["dout"], l, w.scale, impl, workspace=wss[s],
                        grads=dout[2:])
            computed[s].record(comp)
        with torch.cuda.stream(down):
            down.wait_event(computed[s])
            for h, d in zip(hout, dout):
                h.copy_(d, non_blocking=True)
            downloaded[s].record(down)

    for i in range(2):
        step(i)
    torch.cuda.synchronize()
    ke = E2E_STEPS
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    for e in computed + downloaded:   # start the clock with no step in flight
        up.wait_event(e)
    t0.record(up)
    for i in range(ke):
        step(i)
    t1.record(down)                   # after the last step's download
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / ke
    return {"value": flops * world / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms, "steps": ke,
            "pipelining": "upload / compute / download streams, two buffer sets; the clock runs from the first "
                          "upload to the last download"}


def run_ours(args, w):
    import torch
    from bwd_xfa_fwd_gb300 import binding, build

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    build.build()
    lib = binding.load()
    torch.cuda.init()
    _, dev = make_device_inputs(w, torch)
    q, k, v, do = dev["q"], dev["k"], dev["v"], dev["dout"]
    out, lse = torch.empty_like(q), torch.empty(q.shape[:-1], device="cuda", dtype=torch.float32)
    grads = tuple(torch.empty_like(q) for _ in range(3))
    ws = torch.empty(binding.workspace_bytes(w.bh, w.S, w.hd, q.dtype), device="cuda", dtype=torch.uint8)
    keep = (torch.empty(binding.dropout_keep_bytes(w.bh, w.S), device="cuda", dtype=torch.uint8)
            if args.dropout and args.keep_bits != "none" else None)
    stream = torch.cuda.current_stream()

    impl = FAMILIES[args.family]
    fill = bool(args.dropout) and args.keep_bits == "fill"
    stages = ("fwd", "prep", "main", "finish") + (("keep_fill",) if fill else ())
    K = args.steps
    ev = {s: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
          for s in stages}

    def step(i=None):
        def mark(stage, edge):
            if i is not None:
                ev[stage][i][edge].record(stream)

        def hook(name):
            if name == "prep":
                mark("prep", 0)
            elif name == "main":
                mark("prep", 1)
                mark("main", 0)
            elif name == "finish":
                mark("main", 1)
                mark("finish", 0)
            else:
                mark("finish", 1)

        if fill:
            # the keep decisions drawn by their own kernel, then read by both attention kernels
            mark("keep_fill", 0)
            binding.dropout_keep_fill(w.bh, w.S, args.dropout, DROPOUT_SEED, keep)
            mark("keep_fill", 1)
        mark("fwd", 0)
        if args.dropout:
            # dropout on the attention probabilities: the backward is one xfa_bwd_dropout call
            # (its pre-pass, kernel and conversion), timed as "main"; with --keep-bits store the forward
            # caches its keep decisions for the backward (xfa_fwd_dropout_keep / xfa_bwd_dropout_cached),
            # with --keep-bits fill both read those of xfa_dropout_keep_fill (xfa_fwd_dropout_cached)
            binding.fwd(q, k, v, w.scale, impl, out=out, lse=lse, dropout_p=args.dropout, seed=DROPOUT_SEED,
                        keep_bits=keep, keep_cached=fill)
            mark("fwd", 1)
            mark("prep", 0)
            mark("prep", 1)
            mark("main", 0)
            binding.bwd(q, k, v, out, do, lse, w.scale, impl, workspace=ws, grads=grads, dropout_p=args.dropout,
                        seed=DROPOUT_SEED, keep_bits=keep)
            mark("main", 1)
            mark("finish", 0)
            mark("finish", 1)
            return
        binding.fwd(q, k, v, w.scale, impl, out=out, lse=lse)
        mark("fwd", 1)
        binding.bwd_stages(q, k, v, out, do, lse, w.scale, ws, grads, impl=impl, hook=hook)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if binding.status() != binding.XFA_OK:
        raise RuntimeError("kernel status not ok after warm-up")
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clk:
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for i in range(K):
            step(i)
        t_end.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    if binding.status() != binding.XFA_OK:
        raise RuntimeError("kernel status not ok after the timed region")
    total_ms = max_over_ranks(t_start.elapsed_time(t_end), device="cuda")
    per = {s: float(np.mean([a.elapsed_time(b) for a, b in ev[s]])) for s in stages}
    ms_step = total_ms / K
    f_fwd, f_bwd = w.fwd_flops(), w.bwd_flops()
    bwd_ms = per["prep"] + per["main"] + per["finish"]

    graph = measure_graph(torch, step, K, f_fwd + f_bwd) if args.graph else None

    # End to end through the C ABI with host buffers.  Every step copies its inputs
    # (Q, K, V, dO) from pinned host memory to the device and reads O, L, dQ, dK, dV
    # back into pinned host memory.  Steps are software-pipelined over three streams
    # (upload, compute, download) with double-buffered device tensors, so step i's
    # compute overlaps step i+1's upload and step i-1's download.
    e2e = None
    if not args.no_e2e and not args.dropout:
        e2e = measure_e2e(torch, binding, w, dev, ws, impl, K, f_fwd + f_bwd, world)

    pk, pk_kind = peaks()
    rfam = resolved_family(w, args.family)
    k_fwd, k_bwd, launches = kernel_labels(w, rfam)
    peak_tc, peak_src = tensor_peak(pk, pk_kind, rfam)
    main_tflops = f_bwd / (per["main"] * 1e-3) / 1e12
    elt = 2 if w.dtype == "bf16" else 4
    # The D pre-pass by the method's own byte count: read O and dO, write D.
    d_bytes = w.bh * w.S * (2 * w.hd * elt + 4)
    # What the same launch does besides, for the fused dQ route: read L, write -L*log2(e) and
    # clear the fp32 dQ accumulator the backward kernel reduces into.
    clears_acc = rfam in ("tc", "simt")   # the fused tcgen05 and the SIMT backward reduce dQ into fp32
    extra_bytes = w.bh * w.S * (4 + 4 + (4 * w.hd if clears_acc else 0))
    prep_gbs = lambda b: b / (per["prep"] * 1e-3) / 1e9   # noqa: E731
    line = {
        "metric": METRIC,
        "value": (f_fwd + f_bwd) * world / (ms_step * 1e-3) / 1e12,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": w.dtype,
        "data": data_note(w),
        "config": dict(workload_config(w),
                       **({"dropout_p": args.dropout, "dropout_seed": DROPOUT_SEED} if args.dropout else {}),
                       **({"dropout_keep_bits": args.keep_bits} if args.dropout and args.keep_bits != "none" else {})),
        "kernel_family": args.family,
        "fwd_tflops": f_fwd / (per["fwd"] * 1e-3) / 1e12,
        "bwd_tflops": f_bwd / (bwd_ms * 1e-3) / 1e12,
        "fwd_frac_of_peak": f_fwd / (per["fwd"] * 1e-3) / 1e12 / peak_tc,
        "bwd_frac_of_peak": f_bwd / (bwd_ms * 1e-3) / 1e12 / peak_tc,
        "peak_tensor_tflops": peak_tc,
        "peak_kind": peak_src,
        "stage_ms": per,
        "roofline": {"kernel": k_bwd + (" with its pre-pass and conversion (xfa_bwd_dropout)"
                                        if args.dropout else " (xfa_bwd_main)"),
                     "bound": "alu" if rfam == "simt" else "tensor", "achieved": main_tflops,
                     "peak": peak_tc, "unit": "TFLOP/s", "frac": main_tflops / peak_tc,
                     "traffic": (recorded_traffic("tc_bwd", w.name) if rfam == "tc" and not args.dropout
                                 else None),
                     "peak_source": peak_src},
        "roofline_fwd": {"kernel": k_fwd + " (xfa_fwd)", "bound": "alu" if rfam == "simt" else "tensor",
                         "achieved": f_fwd / (per["fwd"] * 1e-3) / 1e12, "peak": peak_tc, "unit": "TFLOP/s",
                         "frac": f_fwd / (per["fwd"] * 1e-3) / 1e12 / peak_tc,
                         "traffic": (recorded_traffic("tc_fwd", w.name) if rfam in ("tc", "tc_det")
                                     and not args.dropout else None)},
        "roofline_prep": None if args.dropout else {
            "kernel": "rowdot_kernel (xfa_bwd_prep): the D pre-pass, bytes of O, dO read and D written",
            "bound": "hbm", "achieved": prep_gbs(d_bytes), "peak": float(pk["hbm_gbs"]), "unit": "GB/s",
            "frac": prep_gbs(d_bytes) / float(pk["hbm_gbs"]), "bytes": d_bytes,
            "same_launch": {"what": "L read, -L*log2(e) written" + (", fp32 dQ accumulator cleared"
                                                                    if clears_acc else ""),
                            "bytes": extra_bytes, "achieved_all_bytes": prep_gbs(d_bytes + extra_bytes),
                            "frac_all_bytes": prep_gbs(d_bytes + extra_bytes) / float(pk["hbm_gbs"])},
            "traffic": recorded_traffic("rowdot", w.name)},
        "e2e": e2e,
        "graph": graph,
        "gpu_launches": (launches + (1 if fill else 0)) * K,   # + the keep-bit fill kernel with --keep-bits fill
        "clocks": clk.result,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        base = cpu_baseline_leg(w)
        line["cpu_baseline"] = {k: base[k] for k in ("value", "unit", "cores", "kind", "sample")}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing leg")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--dropout", type=float, default=0.0,
                    help="dropout rate on the attention probabilities (0: none, the benchmark's default)")
    ap.add_argument("--keep-bits", choices=("none", "store", "fill"), default="none", nargs="?", const="store",
                    help="with --dropout: cache the keep decisions instead of drawing them twice -- 'store': the "
                         "forward stores them for the backward; 'fill': xfa_dropout_keep_fill draws them (timed "
                         "as the keep_fill stage) and both kernels read them")
    ap.add_argument("--family", choices=sorted(FAMILIES), default="auto",
                    help="kernel family (xfa_impl): auto, tcgen05 (bf16: dQ by fp32 reductions; fp32 with "
                         "hd 32/64: the 3xTF32 kernels), tcgen05_det (bf16: dQ by a separate pass, "
                         "bit-reproducible), simt")
    ap.add_argument("--workload", type=int, default=WORKLOAD_ID, choices=sorted(inputs.WORKLOADS),
                    help="workload id (default: the S=8192 benchmark workload; others for profiling)")
    ap.add_argument("--graph", action="store_true",
                    help="also time the step captured in a CUDA graph and replayed (added as \"graph\")")
    ap.add_argument("--shape", default=None,
                    help="B,H,S,hd,dtype: a seeded synthetic shape of the same recipe instead of --workload "
                         "(profiling; scale 1/sqrt(hd), seed 0)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    w = inputs.WORKLOADS[args.workload]
    if args.shape:
        try:
            B, H, S, hd, dt = args.shape.split(",")
            w = inputs.Workload(f"causal_{dt}_bh{int(B) * int(H)}_s{int(S)}_hd{int(hd)}", int(B), int(H), int(S),
                                int(hd), dt, 1.0 / math.sqrt(int(hd)), seed=0)
        except ValueError:
            ap.error("--shape wants B,H,S,hd,dtype (dtype f32 or bf16)")
        if w.dtype not in ("f32", "bf16"):
            ap.error("--shape dtype must be f32 or bf16")
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
