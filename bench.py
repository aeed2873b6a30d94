#!/usr/bin/env python
"""Throughput benchmark of the log-linear Mamba-2 forward on GB300.

Workload (one step = one loglinear_fwd over one batch, with the Fenwick state export):
``pages``: B=4 per GPU, H=48 heads in 24 Q/K groups, T=8192, d_k=128, d_v=64, chunk 64,
14 lambda levels, bf16 q/k/v/o, fp32 a/lambda, seeded synthetic inputs resident in HBM.

    python bench.py [--gpus N --steps K --warmup W] [--impl reference]

Prints one JSON line (rank 0).  ``value`` is forward tokens/s over all ranks (each rank
runs its own batch: weak scaling, no data-path collective); ``e2e`` is the same metric
through loglinear_fwd_host with pinned host buffers (copies inside the timed region);
``roofline`` is the dominant kernel's algorithmic HBM bytes per launch over its average
CUDA-event duration, against the measured copy bandwidth; ``cpu_baseline`` is the fp64
CPU oracle (recurrent form) timed on this host's cores on a bounded sample.  With
``--impl reference`` the oracle itself is timed per step instead (the reference arm).
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "log-linear Mamba-2 fwd tokens/s at T=8K–131K on 1 GB300; % of roofline"
L2_BYTES = 129 * 2 ** 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extras", action="store_true", help="skip the long/decode/e2e extras")
    ap.add_argument("--ncu-case", nargs="?", const="fwd",
                    choices=["fwd", "bwd", "gdn", "decode", "decode64", "long"],
                    help="profiling case, no timing, no JSON: on the pages workload at batch 1 "
                         "(inputs 225 MB > L2) three forwards (fwd, the default), two backwards "
                         "(bwd) or two Gated DeltaNet forwards (gdn); decode: three decode steps "
                         "of the decode workload at batch 8 (states 214 MB > L2); decode64: 64 "
                         "steps of the decode workload itself (batch 64, positions 32768..32831); "
                         "long: two forwards of the long workload's shape with 4 of its 48 heads")
    return ap.parse_args()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def job_time(ms: float, world: int, dist=None, device=None) -> float:
    """Per-step time of the whole job: the slowest rank's (max over ranks; a no-op at N=1)."""
    if world <= 1:
        return ms
    import torch

    tt = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return float(tt.item())


def job_value(units_per_rank: int, world: int, ms: float) -> float:
    """Whole-job throughput: the units all ranks processed over the job's per-step time."""
    return world * units_per_rank / (ms / 1e3)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d.get("bf16_tflops", 1900.0)), "measured"
    return 6800.0, 1900.0, "fallback"


def workload_desc(w):
    return (f"{w.name}: B={w.batch} H={w.heads} ({w.groups} Q/K groups) T={w.T} d_k={w.d_k} "
            f"d_v={w.d_v} chunk={w.chunk} levels={w.levels} bf16 q/k/v/o, fp32 a/lambda")


def algorithmic_bytes(w, kernel: str) -> int:
    """Algorithmic HBM bytes one launch of `kernel` must move for workload w (inputs read
    once, outputs written once; chunk/block states are implementation traffic)."""
    B, T, H, G, L = w.batch, w.T, w.heads, w.groups, w.levels
    es = 2 if "bfloat16" in str(w.dtype) else 4
    q = k = B * T * G * w.d_k * es
    v = o = B * T * H * w.d_v * es
    a = B * T * H * 4
    lam = B * T * H * L * 4
    if kernel in ("gen_output", "tc_output"):
        return q + k + v + lam + a + o  # a is read as its chunk-local log cumsum
    if kernel in ("gen_chunk_state", "tc_state"):
        return k + v + a
    return q + k + v + a + lam + o  # whole path


# ---- clocks -------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self._t.join(timeout=5)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


def traffic_for(kernel: str, w, key: str | None = None, algorithmic: float | None = None):
    """ncu DRAM bytes per launch from profiles/traffic.json, if the kernel's source is
    unchanged since the capture (scaled to this workload's units: the record holds bytes
    per token of all heads, or, with `algorithmic` given, DRAM bytes per algorithmic byte
    over a run of launches).  key names the record (default: the kernel's name)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(key or kernel)
    if not d:
        return None
    srcs = d["source"] if isinstance(d["source"], list) else [d["source"]]
    h = hashlib.sha256()
    for name in srcs:  # every file the kernel is compiled from, in order
        src = os.path.join(ROOT, "structured_mask_linear_gb300", "csrc", name)
        if not os.path.exists(src):
            return None
        h.update(open(src, "rb").read())
    if h.hexdigest() != d["source_sha256"]:
        return None
    if algorithmic is not None:
        return d["bytes_per_algorithmic_byte"] * algorithmic if "bytes_per_algorithmic_byte" in d else None
    return d["bytes_per_token"] * w.batch * w.T


# ---- CPU oracle baseline --------------------------------------------------------------
def cpu_oracle_run(w, heads: int, T: int, seed: int = 0):
    """Times the oracle's recurrent form on batch 0, heads [0, heads), first T tokens."""
    import torch

    from oracle import oracle
    from structured_mask_linear_gb300.inputs import make_inputs, to_numpy64, workload

    ws = workload(w.name, batch=1, heads=heads, T=T, decode_steps=0,
                  heads_per_group=min(w.heads_per_group, heads))
    x = make_inputs(ws, "cpu", seed=seed)
    arrs = [to_numpy64(t) for t in (x.q, x.k, x.v, x.a, x.lam)]
    t0 = time.perf_counter()
    oracle.form_r(*arrs)
    dt = time.perf_counter() - t0
    return dt, oracle.num_threads()


def cpu_oracle_other(w, what: str, T: int = 2048, seed: int = 0):
    """The oracle beside a next-row GPU path, on a bounded sample: batch element 0, all
    heads, the first T tokens.  what: "backward" (gradients of sum(dO * o)) or "gdn"
    (log-linear Gated DeltaNet forward).  Returns a cpu-baseline object in all-head
    tokens per second."""
    import numpy as np
    import torch

    from oracle import oracle
    from structured_mask_linear_gb300.inputs import make_inputs, to_numpy64, workload

    ws = workload(w.name, batch=1, T=T, levels=max(w.levels, T.bit_length() + 1))
    x = make_inputs(ws, "cpu", seed=seed)
    arrs = [to_numpy64(t) for t in (x.q, x.k, x.v, x.a, x.lam)]
    rng = np.random.default_rng(seed)
    if what == "backward":
        dO = rng.standard_normal(arrs[2].shape)
        t0 = time.perf_counter()
        oracle.backward(*arrs, dO)
        form = "backward of the quadratic form"
    else:
        k = arrs[1] / np.linalg.norm(arrs[1], axis=-1, keepdims=True)
        beta = 1.0 / (1.0 + np.exp(-rng.standard_normal(arrs[3].shape)))
        t0 = time.perf_counter()
        oracle.gdn_forward(arrs[0], k, arrs[2], arrs[3], beta, arrs[4])
        form = "gated delta rule then the quadratic form"
    dt = time.perf_counter() - t0
    return {"value": T / dt, "unit": "tokens/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{form}, fp64, batch element 0 (all {w.heads} heads), first {T} tokens: "
                      f"{dt:.2f} s"}


def cpu_baseline(w):
    dt, cores = cpu_oracle_run(w, w.heads, w.T)
    return {"value": w.T / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"recurrent Fenwick form, fp64, batch element 0 of the workload "
                      f"(all {w.heads} heads, T={w.T}): {w.T} tokens in {dt:.2f} s"}


def run_reference(args):
    ws_, rank, _ = dist_env()
    if rank != 0:
        return
    from structured_mask_linear_gb300.inputs import workload

    w = workload("pages")
    import multiprocessing

    heads = max(2, min(w.heads, (multiprocessing.cpu_count() // 2) * 2))
    # calibrate the per-step sample so that warmup + steps stay within ~3 minutes
    T = 1024
    dt, cores = cpu_oracle_run(w, heads, T)
    budget = 150.0 / max(1, args.steps + args.warmup)
    while T * 2 <= w.T and dt * 2.2 < budget:
        T *= 2
        dt, cores = cpu_oracle_run(w, heads, T)
    for _ in range(max(0, args.warmup - 1)):
        cpu_oracle_run(w, heads, T)
    times = []
    for _ in range(args.steps):
        d, cores = cpu_oracle_run(w, heads, T)
        times.append(d)
    total = sum(times)
    tokens = T * heads / w.heads  # token-equivalents of all heads
    value = tokens * args.steps / total
    sample = (f"per step: recurrent Fenwick form (fp64) on batch 0, {heads} of {w.heads} heads, "
              f"first {T} of {w.T} tokens = {tokens:.0f} all-head token equivalents")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload_desc(w), "global_batch": w.batch,
                       "seq_len": w.T, "parallelism": "host cores (OpenMP over heads)"},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---- GPU arm --------------------------------------------------------------------------
def ncu_case(what: str = "fwd"):
    import torch

    import structured_mask_linear_gb300 as sml
    from structured_mask_linear_gb300.inputs import make_inputs, workload

    sml.lib()
    if what in ("decode", "decode64"):
        wd = workload("decode", batch=8) if what == "decode" else workload("decode")
        n = 3 if what == "decode" else 64
        st, lsc, q, k, v, a, lam = decode_inputs(torch, wd, "cuda", steps=n)
        for i in range(n):
            sml.loglinear_decode_step(wd.T + i, q[i], k[i], v[i], a[i], lam[i], st, lsc)
        torch.cuda.synchronize()
        assert sml.loglinear_check_status() == 0
        return
    if what == "long":
        wl = workload("long", heads=4)
        x = make_inputs(wl, "cuda", seed=1)
        for _ in range(2):
            sml.loglinear_fwd(x.q, x.k, x.v, x.a, x.lam, chunk=wl.chunk)
        torch.cuda.synchronize()
        assert sml.loglinear_check_status() == 0
        return
    w = workload("pages", batch=1)
    x = make_inputs(w, "cuda", seed=0)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(99)
    if what == "fwd":
        st = torch.empty((1, w.heads, w.T.bit_length() + 1, w.d_k, w.d_v), device="cuda")
        for _ in range(3):
            sml.loglinear_fwd(x.q, x.k, x.v, x.a, x.lam, chunk=w.chunk, states_out=st,
                              state_levels=w.T.bit_length() + 1)
    elif what == "bwd":
        dO = torch.randn(x.v.shape, generator=gen, device="cuda").to(x.v.dtype)
        for _ in range(2):
            sml.loglinear_bwd(x.q, x.k, x.v, x.a, x.lam, dO, chunk=w.chunk)
    else:
        kn = x.k.float()
        kn = (kn / kn.norm(dim=-1, keepdim=True)).to(x.k.dtype)
        beta = torch.sigmoid(torch.randn(x.a.shape, generator=gen, device="cuda"))
        for _ in range(2):
            sml.loglinear_gdn_fwd(x.q, kn, x.v, x.a, beta, x.lam, chunk=w.chunk)
    torch.cuda.synchronize()
    assert sml.loglinear_check_status() == 0


def main():
    args = parse()
    if args.ncu_case:
        ncu_case(args.ncu_case)
        return
    if args.impl == "reference":
        run_reference(args)
        return
    import torch
    import torch.distributed as dist

    import structured_mask_linear_gb300 as sml
    from structured_mask_linear_gb300.inputs import make_inputs, workload

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    sml.lib()
    hbm_peak, _, peak_src = peaks()

    w = workload("pages")
    x = make_inputs(w, dev, seed=rank)
    B, T, H = w.batch, w.T, w.heads
    SL = T.bit_length() + 1
    shape = sml.fwd_shape(x.q, x.v, x.lam, w.chunk)
    names = sml.loglinear_fwd_kernel_names(shape, with_export=True)
    nk = len(names)
    o = torch.empty_like(x.v)
    wsb = torch.empty(sml.loglinear_fwd_workspace_bytes(shape), dtype=torch.uint8, device=dev)
    st = torch.empty((B, H, SL, w.d_k, w.d_v), device=dev)
    lsc = torch.empty((B, H, SL), device=dev)
    stream = torch.cuda.current_stream()

    def step(events=None):
        if events is None:
            sml.loglinear_fwd(x.q, x.k, x.v, x.a, x.lam, chunk=w.chunk, o=o, workspace=wsb,
                              states_out=st, state_logscale_out=lsc, state_levels=SL)
        else:
            sml.loglinear_fwd_profiled(x.q, x.k, x.v, x.a, x.lam, events, chunk=w.chunk, o=o,
                                       workspace=wsb, states_out=st, state_logscale_out=lsc,
                                       state_levels=SL)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    if sml.loglinear_check_status() != 0:
        raise RuntimeError("device status error during warm-up")
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nk + 1)] for _ in range(args.steps)]
    for row in evs:  # torch creates the CUDA event on its first record
        for e in row:
            e.record(stream)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    # pass 1: the step as a user runs it (no events between kernels, so each launch may
    # overlap the end of the one before): value and ms_per_step
    n0 = sml.loglinear_launch_count()
    t_start.record(stream)
    for i in range(args.steps):
        step()
    t_end.record(stream)
    torch.cuda.synchronize()
    n1 = sml.loglinear_launch_count()
    # pass 2: the same steps with CUDA events between the kernels: per-kernel durations
    for i in range(args.steps):
        step(evs[i])
    torch.cuda.synchronize()
    clk = clocks.stop()
    if world > 1:
        dist.barrier()
    if sml.loglinear_check_status() != 0:
        raise RuntimeError("device status error in the timed region")
    ms = job_time(t_start.elapsed_time(t_end) / args.steps, world, dist, dev)
    value = job_value(B * T, world, ms)
    per_kernel = [statistics.mean(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(args.steps))
                  for j in range(nk)]
    dom = max(range(nk), key=lambda j: per_kernel[j])
    dom_name = names[dom]
    dom_bytes = algorithmic_bytes(w, dom_name)
    achieved = dom_bytes / (per_kernel[dom] / 1e3) / 1e9
    path_bytes = algorithmic_bytes(w, "path")
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": workload_desc(w), "global_batch": B * world, "seq_len": T,
                   "parallelism": f"replicas: each of {world} GPU(s) runs its own batch",
                   "l2": f"inputs {path_bytes / 1e9:.2f} GB per step > L2 {L2_BYTES >> 20} MiB; no flush"},
        "roofline": {"bound": "hbm", "kernel": dom_name, "achieved": achieved, "peak": hbm_peak,
                     "unit": "GB/s", "frac": achieved / hbm_peak, "peak_source": peak_src,
                     "traffic": traffic_for(dom_name, w),
                     "algorithmic_bytes_per_launch": dom_bytes},
        "path_roofline": {"achieved": path_bytes / (ms / 1e3) / 1e9, "peak": hbm_peak,
                          "unit": "GB/s", "frac": path_bytes / (ms / 1e3) / 1e9 / hbm_peak,
                          "algorithmic_bytes_per_step": path_bytes},
        "kernels_ms": {n: round(t, 4) for n, t in zip(names, per_kernel)},
        "kernels_ms_note": ("a second pass of the same steps with CUDA events between the "
                            "kernels (which serialises them); ms_per_step is the first pass"),
        "gpu_launches": int(n1 - n0),
        "clocks": clk,
        "path": sml.loglinear_fwd_path(shape),
    }
    del evs
    if world == 1 and not args.no_extras:
        line["e2e"] = e2e_measure(sml, torch, x, w, dev, min(args.steps, 20))
        line["long"] = long_measure(sml, torch, dev)
        line["decode"] = decode_measure(sml, torch, dev, hbm_peak)
        line["comparators"] = comparators_measure(sml, torch, x, w, ms)
        line["backward"] = backward_measure(sml, torch, x, w, hbm_peak)
        line["gated_deltanet"] = gdn_measure(sml, torch, x, w, hbm_peak)
    else:
        line["e2e"] = e2e_measure(sml, torch, x, w, dev, min(args.steps, 10))
        if world > 1:
            e_ms = job_time(line["e2e"]["ms_per_step"], world, dist, dev)
            line["e2e"]["value"] = job_value(B * T, world, e_ms)
    if rank == 0 and world == 1:
        line["cpu_baseline"] = cpu_baseline(w)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def e2e_measure(sml, torch, x, w, dev, steps):
    hq, hk, hv, ha, hl = (t.cpu().pin_memory() for t in (x.q, x.k, x.v, x.a, x.lam))
    ho = torch.empty(x.v.shape, dtype=x.v.dtype).pin_memory()
    shape = sml.fwd_shape(x.q, x.v, x.lam, w.chunk)
    arena = torch.empty(sml.loglinear_fwd_host_arena_bytes(shape), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    for _ in range(3):
        sml.loglinear_fwd_host(hq, hk, hv, ha, hl, ho, arena, chunk=w.chunk)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        sml.loglinear_fwd_host(hq, hk, hv, ha, hl, ho, arena, chunk=w.chunk)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    bi = sum(t.numel() * t.element_size() for t in (hq, hk, hv, ha, hl))
    bo = ho.numel() * ho.element_size()
    return {"value": w.batch * w.T / (ms / 1e3), "unit": "tokens/s", "ms_per_step": ms,
            "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo, "steps": steps,
            "api": "loglinear_fwd_host (pinned host buffers)"}


def gdn_measure(sml, torch, x, w, hbm_peak, steps=3):
    """Log-linear Gated DeltaNet forward on the same workload (keys L2-normalised per
    token, beta = sigmoid(z)): the delta-rule values kernel plus the level-fused forward.
    Algorithmic bytes: q, k, v, a, beta, lambda read once, o written once."""
    gen = torch.Generator(device=x.v.device)
    gen.manual_seed(6)
    kn = x.k.float()
    kn = (kn / kn.norm(dim=-1, keepdim=True)).to(x.k.dtype)
    beta = torch.sigmoid(torch.randn(x.a.shape, generator=gen, device=x.a.device))
    shape = sml.fwd_shape(x.q, x.v, x.lam, w.chunk)
    ws = torch.empty(sml.lib().loglinear_gdn_fwd_workspace_bytes(ctypes.byref(shape)), dtype=torch.uint8,
                     device=x.v.device)
    o = torch.empty_like(x.v)
    call = lambda: sml.loglinear_gdn_fwd(x.q, kn, x.v, x.a, beta, x.lam, chunk=w.chunk, o=o, workspace=ws)
    call()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        call()
    e1.record()
    torch.cuda.synchronize()
    if sml.loglinear_check_status() != 0:
        raise RuntimeError("device status error in the Gated DeltaNet forward")
    ms = e0.elapsed_time(e1) / steps
    el = lambda t: t.numel() * t.element_size()
    nbytes = el(x.q) + el(kn) + 2 * el(x.v) + el(x.a) + el(beta) + el(x.lam)
    res = {"workload": workload_desc(w) + ", keys L2-normalised, beta = sigmoid(z)",
           "ms_per_step": ms, "unit": "tokens/s", "value": w.batch * w.T / (ms / 1e3), "steps": steps,
           "roofline": {"bound": "hbm", "achieved": nbytes / (ms / 1e3) / 1e9, "peak": hbm_peak,
                        "unit": "GB/s", "frac": nbytes / (ms / 1e3) / 1e9 / hbm_peak,
                        "algorithmic_bytes_per_step": nbytes}}
    del ws, o, kn, beta
    torch.cuda.empty_cache()
    res["cpu_oracle"] = cpu_oracle_other(w, "gdn")
    return res


def backward_measure(sml, torch, x, w, hbm_peak, steps=3):
    """loglinear_bwd on the same workload (gradients of sum(dO * o) for q, k, v, log a,
    lambda), CUDA events around whole calls, inputs in HBM.  Algorithmic bytes: q, k, v,
    a, lambda, dO read once; dq, dk, dv, d(log a), dlambda written once."""
    gen = torch.Generator(device=x.v.device)
    gen.manual_seed(5)
    dO = torch.randn(x.v.shape, generator=gen, device=x.v.device).to(x.v.dtype)
    shape = sml.fwd_shape(x.q, x.v, x.lam, w.chunk)
    ws = torch.empty(sml.lib().loglinear_bwd_workspace_bytes(ctypes.byref(shape)), dtype=torch.uint8,
                     device=x.v.device)
    call = lambda: sml.loglinear_bwd(x.q, x.k, x.v, x.a, x.lam, dO, chunk=w.chunk, workspace=ws)
    call()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        call()
    e1.record()
    torch.cuda.synchronize()
    if sml.loglinear_check_status() != 0:
        raise RuntimeError("device status error in the backward")
    ms = e0.elapsed_time(e1) / steps
    el = lambda t: t.numel() * t.element_size()
    nbytes = 2 * (el(x.q) + el(x.k) + el(x.v) + el(x.a) + el(x.lam)) + el(dO)
    res = {"workload": workload_desc(w), "ms_per_step": ms, "unit": "tokens/s",
           "value": w.batch * w.T / (ms / 1e3), "steps": steps,
           "path": "tensor cores: tc_bwd_intra, tc_bwd_q, tc_bwd_kv (csrc/tc_bwd.cu), sums in csrc/backward.cu",
           "roofline": {"bound": "hbm", "achieved": nbytes / (ms / 1e3) / 1e9, "peak": hbm_peak,
                        "unit": "GB/s", "frac": nbytes / (ms / 1e3) / 1e9 / hbm_peak,
                        "algorithmic_bytes_per_step": nbytes}}
    del ws, dO
    torch.cuda.empty_cache()
    res["cpu_oracle"] = cpu_oracle_other(w, "backward")
    return res


def comparators_measure(sml, torch, x, w, fused_ms, steps=5):
    """The same workload through the two comparators: the forward without level fusion
    (one output pass per level) and the lambda-constant special case (Mamba-2 SSD, with a
    sequential state pass over tiles).  CUDA events around whole calls, inputs in HBM."""
    res = {"fused_ms": fused_ms}
    shape = sml.fwd_shape(x.q, x.v, x.lam, w.chunk)
    dev = x.q.device
    o = torch.empty_like(x.v)
    ws_n = torch.empty(sml.lib().loglinear_fwd_naive_workspace_bytes(ctypes.byref(shape)),
                       dtype=torch.uint8, device=dev)
    ws_s = torch.empty(sml.lib().ssd_fwd_workspace_bytes(ctypes.byref(shape)), dtype=torch.uint8,
                       device=dev)
    for key, call in (("naive_per_level_ms",
                       lambda: sml.loglinear_fwd_naive(x.q, x.k, x.v, x.a, x.lam, chunk=w.chunk, o=o,
                                                       workspace=ws_n)),
                      ("ssd_ms", lambda: sml.ssd_fwd(x.q, x.k, x.v, x.a, chunk=w.chunk, o=o,
                                                     workspace=ws_s))):
        for _ in range(3):
            call()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            call()
        e1.record()
        torch.cuda.synchronize()
        res[key] = e0.elapsed_time(e1) / steps
    if sml.loglinear_check_status() != 0:
        raise RuntimeError("device status error in the comparators")
    res["level_fusion_speedup"] = res["naive_per_level_ms"] / fused_ms
    res["loglinear_over_ssd_time"] = fused_ms / res["ssd_ms"]
    res["note"] = (f"workspaces and outputs allocated before timing; steps={steps}; fused_ms is "
                   "the main line's ms_per_step")
    del o, ws_n, ws_s
    torch.cuda.empty_cache()
    return res


def long_measure(sml, torch, dev, steps=5):
    """The long workload (B=1, H=48, T=131072): whole-step time, then the same steps with
    CUDA events between the kernels for the dominant kernel's roofline, and the oracle's
    recurrent form on a bounded sample of the same workload."""
    from structured_mask_linear_gb300.inputs import make_inputs, workload

    w = workload("long")
    x = make_inputs(w, dev, seed=1)
    o = torch.empty_like(x.v)
    shape = sml.fwd_shape(x.q, x.v, x.lam, w.chunk)
    wsb = torch.empty(sml.loglinear_fwd_workspace_bytes(shape), dtype=torch.uint8, device=dev)
    names = sml.loglinear_fwd_kernel_names(shape, with_export=False)
    for _ in range(3):
        sml.loglinear_fwd(x.q, x.k, x.v, x.a, x.lam, chunk=w.chunk, o=o, workspace=wsb)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        sml.loglinear_fwd(x.q, x.k, x.v, x.a, x.lam, chunk=w.chunk, o=o, workspace=wsb)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)] for _ in range(steps)]
    for row in evs:  # torch creates the CUDA event on its first record
        for e in row:
            e.record()
    torch.cuda.synchronize()
    for row in evs:
        sml.loglinear_fwd_profiled(x.q, x.k, x.v, x.a, x.lam, row, chunk=w.chunk, o=o, workspace=wsb)
    torch.cuda.synchronize()
    if sml.loglinear_check_status() != 0:
        raise RuntimeError("device status error in the long workload")
    per_kernel = [statistics.mean(r[j].elapsed_time(r[j + 1]) for r in evs) for j in range(len(names))]
    dom = max(range(len(names)), key=lambda j: per_kernel[j])
    hbm_peak, _, peak_src = peaks()
    pb = algorithmic_bytes(w, "path")
    db = algorithmic_bytes(w, names[dom])
    ach = db / (per_kernel[dom] / 1e3) / 1e9
    res = {"workload": workload_desc(w), "value": w.batch * w.T / (ms / 1e3), "unit": "tokens/s",
           "ms_per_step": ms, "steps": steps,
           "path_frac": pb / (ms / 1e3) / 1e9 / hbm_peak,
           "kernels_ms": {n: round(t, 4) for n, t in zip(names, per_kernel)},
           "roofline": {"bound": "hbm", "kernel": names[dom], "achieved": ach, "peak": hbm_peak,
                        "unit": "GB/s", "frac": ach / hbm_peak, "peak_source": peak_src,
                        "traffic": traffic_for(names[dom], w, key=names[dom] + ":long"),
                        "algorithmic_bytes_per_launch": db}}
    del x, o, wsb, evs
    torch.cuda.empty_cache()
    res["cpu_baseline"] = cpu_baseline_sampled(w)
    return res


def cpu_baseline_sampled(w, T: int | None = None):
    """The oracle's recurrent form on batch element 0, as many heads as host cores (even,
    at most H), the first T tokens (default all): all-head token equivalents per second."""
    import multiprocessing

    from oracle import oracle

    heads = max(2, min(w.heads, (multiprocessing.cpu_count() // 2) * 2))
    T = w.T if T is None else T
    dt, cores = cpu_oracle_run(w, heads, T)
    return {"value": T * heads / w.heads / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"recurrent Fenwick form, fp64, batch element 0, {heads} of {w.heads} heads, "
                      f"first {T} tokens: {dt:.2f} s, scaled to all {w.heads} heads"}


def decode_inputs(torch, w, dev, steps):
    """Random fp32 states at every level (the live levels of each position decide the
    work; state values do not) and per-step token inputs for `steps` decode steps."""
    B, H, G, L = w.batch, w.heads, w.groups, w.levels
    gen = torch.Generator(device=dev)
    gen.manual_seed(7)
    st = torch.randn((B, H, L, w.d_k, w.d_v), generator=gen, device=dev) * 1e-2
    lsc = torch.zeros((B, H, L), device=dev)
    q = torch.randn((steps, B, G, w.d_k), generator=gen, device=dev).to(torch.bfloat16)
    k = torch.randn((steps, B, G, w.d_k), generator=gen, device=dev).to(torch.bfloat16)
    v = torch.randn((steps, B, H, w.d_v), generator=gen, device=dev).to(torch.bfloat16)
    a = torch.rand((steps, B, H), generator=gen, device=dev) * 0.5 + 0.5
    lam = torch.rand((steps, B, H, L), generator=gen, device=dev)
    return st, lsc, q, k, v, a, lam


def decode_bytes(w, pos: int) -> int:
    """Algorithmic bytes of one decode step at position pos: every live state read once,
    the merged state written once, the token's inputs read and its output written."""
    B, H, G, L = w.batch, w.heads, w.groups, w.levels
    state = w.d_k * w.d_v * 4
    tok_io = B * (2 * G * w.d_k * 2 + H * w.d_v * 2 * 2 + H * 4 + H * L * 4)
    return B * H * (bin(pos).count("1") * state + state) + tok_io


def decode_measure(sml, torch, dev, hbm_peak, steps=1024):
    """Decode workload timing: B=64, H=48, positions 32768..33791."""
    from structured_mask_linear_gb300.inputs import workload

    w = workload("decode")
    B, H, L = w.batch, w.heads, w.levels
    st, lsc, q, k, v, a, lam = decode_inputs(torch, w, dev, steps)
    o = torch.empty((B, H, w.d_v), dtype=torch.bfloat16, device=dev)
    for i in range(5):
        sml.loglinear_decode_step(w.T + i, q[i], k[i], v[i], a[i], lam[i], st, lsc, o_t=o)
    lsc.zero_()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(steps):
        sml.loglinear_decode_step(w.T + i, q[i], k[i], v[i], a[i], lam[i], st, lsc, o_t=o)
    e1.record()
    torch.cuda.synchronize()
    ms_eager = e0.elapsed_time(e1) / steps
    # The same steps captured once in a CUDA graph and replayed: one launch per step without
    # the host's per-call work between them (the positions, hence the live levels and the
    # work, are those of the eager loop; the state values do not change the work).
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graph, stream=cap):
            for i in range(steps):
                sml.loglinear_decode_step(w.T + i, q[i], k[i], v[i], a[i], lam[i], st, lsc, o_t=o)
    torch.cuda.current_stream().wait_stream(cap)
    graph.replay()
    torch.cuda.synchronize()
    e0.record()
    graph.replay()
    e1.record()
    torch.cuda.synchronize()
    if sml.loglinear_check_status() != 0:
        raise RuntimeError("decode: device status set")
    ms = e0.elapsed_time(e1) / steps
    del graph
    nbytes = sum(decode_bytes(w, w.T + i) for i in range(steps)) / steps
    res = {"workload": f"decode: B={B} H={H} d_k={w.d_k} d_v={w.d_v}, positions "
                       f"{w.T}..{w.T + steps - 1}, {L} fp32 state levels",
           "value": B / (ms / 1e3), "unit": "tokens/s", "us_per_step": 1e3 * ms,
           "launch": "the steps replayed from one CUDA graph",
           "us_per_step_eager_loop": 1e3 * ms_eager,
           "achieved_gbs": nbytes / (ms / 1e3) / 1e9, "frac": nbytes / (ms / 1e3) / 1e9 / hbm_peak,
           "algorithmic_bytes_per_step": int(nbytes),
           "roofline": {"bound": "hbm", "kernel": "decode_step_kernel",
                        "achieved": nbytes / (ms / 1e3) / 1e9, "peak": hbm_peak, "unit": "GB/s",
                        "frac": nbytes / (ms / 1e3) / 1e9 / hbm_peak,
                        "traffic": traffic_for("decode_step_kernel", w, key="decode_step_kernel:decode",
                                               algorithmic=nbytes),
                        "algorithmic_bytes_per_launch": int(nbytes)}}
    del st, lsc, q, k, v, a, lam, o
    torch.cuda.empty_cache()
    # the oracle's recurrent form over the prefix and the decode positions (0..33791), one
    # token at a time as a decode loop runs it; a token = one step of one stream, all heads
    cb = cpu_baseline_sampled(w, T=w.T + steps)
    cb["sample"] += (" (positions 0..%d: the prefix and the decode positions, token by token)"
                     % (w.T + steps - 1))
    res["cpu_baseline"] = cb
    return res


if __name__ == "__main__":
    main()
