#!/usr/bin/env python3
"""Benchmark: sampled-token logprobs/sec of the bit-consistent engine on one GB300.

One step = one pass of the whole hot path over one batch: the lm_head GEMM with its
leaf tree and vocabulary-tile log-sum-exp, the combine and sampled-token gather
(``lp_logprobs``), then the importance weights and D3 against a rollout logprob from
a lagged weight copy (``lp_importance_weights``).  Inputs are seeded synthetic data
already resident in HBM; W alone is larger than L2, so every step streams it from HBM.
The default workload is the largest single-GPU one: the importance-weight batch of 512
responses (about 2.07 M tokens, H 4096, V 151936); the same line then carries decode
sub-records (H 7168, V 129280, batches 1 and 256), each with its own roofline.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Prints ONE JSON line (rank 0).  ``--impl reference`` times the fp64 CPU oracle on the
host cores on a bounded row sample of the same workload.  With N > 1 (torchrun) every
rank runs an independent replica of the workload (weak scaling, no collective on the
data path; the ranks only meet at the timing barriers).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sampled-token logprobs/sec (prefill & decode) at diff=0; % of roofline"
UNIT = "tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
# Sources that decide the dominant kernel's code and launch (the recorded DRAM traffic is
# dropped when they change): the leaf GEMM, and from the host library only the functions
# that encode its tensor maps, pick its launch shape and its scheduling band; plus the FP8
# kernel and its launch for --fp8.
KERNEL_SOURCES = ["bit_consistent_logprob_gb300/csrc/kernels.cuh",
                  "bit_consistent_logprob_gb300/csrc/numerics.cuh",
                  "bit_consistent_logprob_gb300/csrc/ptx.cuh"]
HOST_LAUNCH = ("bit_consistent_logprob_gb300/csrc/lp_api.cu",
               ["encode_kmajor", "scheduling_band", "x_box_rows", "pick_band", "launch_gemm_variant",
                "launch_leaf_gemm"])
FP8_SOURCES = ["bit_consistent_logprob_gb300/csrc/fp8_kernels.cuh"]
FP8_HOST_LAUNCH = ["quantize_x_chunk", "launch_fp8_gemm", "quantize_weights"]


def _function_text(src: str, name: str) -> str:
    """The definition of the first function called `name` (signature through its closing brace)."""
    m = re.search(r"^[^\n;{}]*\b" + re.escape(name) + r"\([^;{]*\{", src, flags=re.M)
    if m is None:
        raise KeyError(name)
    depth, i = 0, m.end() - 1
    while True:
        depth += {"{": 1, "}": -1}.get(src[i], 0)
        i += 1
        if depth == 0:
            return src[m.start():i]


# ----------------------------------------------------------------------------- setup
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
        pg = dist
    return world, rank, local, pg


def barrier(pg, device=None):
    if pg is not None:
        if device is not None:
            pg.barrier(device_ids=[device.index])
        else:
            pg.barrier()


def max_over_ranks(pg, value: float, device) -> float:
    if pg is None:
        return value
    import torch

    t = torch.tensor([value], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash(fp8: bool = False) -> str:
    """SHA-256 (first 16 hex digits) of the kernel and launch sources with comments and
    whitespace removed, so that a recorded traffic figure survives edits to comments only."""
    def strip_comments(src):
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        return re.sub(r"//[^\n]*", " ", src)

    def canon(src):
        return " ".join(src.split()).encode()

    h = hashlib.sha256()
    for rel in KERNEL_SOURCES + (FP8_SOURCES if fp8 else []):
        with open(os.path.join(ROOT, rel)) as f:
            h.update(canon(strip_comments(f.read())))
    with open(os.path.join(ROOT, HOST_LAUNCH[0])) as f:
        host = strip_comments(f.read())
    for name in HOST_LAUNCH[1] + (FP8_HOST_LAUNCH if fp8 else []):
        h.update(canon(_function_text(host, name)))
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch of the dominant kernel from the committed ncu summary, if it
    was taken on the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(workload)
    if not e or e.get("kernel_source_sha") != kernel_source_hash(fp8=workload.endswith("_fp8")):
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    def __init__(self, index: int, period_ms: int = 100):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(period_ms), "-i", str(index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=10)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "power_w_max": max(power), "samples": len(sm), "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------- workloads
def first_rows(lengths, rows: int):
    """The sequence lengths of the first `rows` tokens of a packed batch (the last one cut)."""
    kept, left = [], rows
    for L in lengths:
        if left == 0:
            break
        kept.append(min(L, left))
        left -= kept[-1]
    return kept


def make_workload(name: str, device, seed_offset: int = 0, batch: int = 128, rows: int = 0):
    """The named workload's inputs; rows > 0 keeps only its first `rows` tokens (a small case
    of the same shapes, for profiler captures)."""
    import torch

    from bit_consistent_logprob_gb300 import inputs

    wl = inputs.WORKLOADS[name]
    seed = wl.seed + seed_offset
    if name in ("qwen_prefill", "is_d3"):
        lengths = inputs.packed_lengths(wl.n_seqs, wl.len_lo, wl.len_hi, wl.seed)
        T = sum(lengths)
    elif name == "ds_decode":
        lengths = [1] * batch
        T = batch
    else:
        T = wl.T
        lengths = [T]
    if 0 < rows < T:
        lengths, T = first_rows(lengths, rows), rows
    X = inputs.hidden_states(T, wl.H, seed, device=device)
    W = inputs.lm_head(wl.V, wl.H, seed, device=device)
    ids = inputs.uniform_ids(T, wl.V, seed, device=device)
    return wl, lengths, X, W, ids


def rollout_logprobs(W, X, ids, wl, seed, max_tokens):
    """The rollout side's logprob mu, from a weight copy a few updates behind (data prep)."""
    from bit_consistent_logprob_gb300 import Engine, inputs

    W_lag = inputs.lagged_lm_head(W, seed)
    with Engine(W_lag, n_leaves=wl.n_leaves, max_tokens=max_tokens) as eng:
        mu = eng.logprobs(X, ids)
        eng.check()
    del W_lag
    return mu


# ----------------------------------------------------------------------------- RL epilogues
RL_BYTES_PER_TOKEN = {"stats": 9, "reinforce_zero": 17}  # reads a, b, mask; + writes w_hat, grad


def rl_inputs(device, seed_offset: int = 0):
    """The importance-weight workload's token stream: 512 responses of U[128, 8192] tokens in
    groups of 8, learner / rollout logprobs, response mask, 0/1 rewards."""
    from bit_consistent_logprob_gb300 import inputs

    wl = inputs.WORKLOADS["is_d3"]
    offs, rewards = inputs.response_batch(wl.n_seqs // 8, 8, wl.len_lo, wl.len_hi, wl.seed)
    T = int(offs[-1])
    lp, lm, mask = inputs.synthetic_is_inputs(T, seed=wl.seed + seed_offset, device=device)
    return wl, offs, rewards, lp, lm, mask


def run_rl_epilogue(args, world, rank, local, pg):
    import torch

    from bit_consistent_logprob_gb300 import Engine, inputs

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wl, offs_h, rewards_h, lp, lm, mask = rl_inputs(dev, seed_offset=rank)
    T, B = lp.shape[0], rewards_h.shape[0]
    offs, rewards = offs_h.to(dev), rewards_h.to(dev)
    W = inputs.lm_head(1024, 256, wl.seed, device=dev)  # the handle's workspace only
    eng = Engine(W, n_leaves=4, max_tokens=128)
    stats = torch.empty(5, dtype=torch.float64, device=dev)
    w_hat = torch.empty(T, dtype=torch.float32, device=dev)
    grad = torch.empty(T, dtype=torch.float32, device=dev)
    adv = torch.empty(B, dtype=torch.float64, device=dev)
    stream = torch.cuda.current_stream()
    launches = [0]
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    timing = [False]

    def step(k=None):
        eng.acceptance_stats(lp, lm, mask, out=stats)
        launches[0] += eng.last_launch_count
        if k is not None:
            ev[k][0].record(stream)
        loss = eng.reinforce_zero(lp, lm, offs, rewards, 8, mask=mask, out_w_hat=w_hat,
                                  out_grad=grad, out_adv=adv)[0]
        if k is not None:
            ev[k][1].record(stream)
        launches[0] += eng.last_launch_count
        return loss

    for _ in range(args.warmup):
        step()
    eng.check()
    torch.cuda.synchronize()
    launches[0] = 0
    sampler = ClockSampler(local)
    time.sleep(0.3)
    barrier(pg, dev)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for k in range(args.steps):
        step(k)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(pg, dev)
    clocks = sampler.stop()
    eng.check()
    ms = e0.elapsed_time(e1) / args.steps
    ms_max = max_over_ranks(pg, ms, dev)
    rz_ms = sum(a.elapsed_time(b) for a, b in ev) / args.steps

    e2e = None
    if not args.no_e2e:
        lph, lmh, mh = (t.cpu().pin_memory() for t in (lp, lm, mask))
        offh, rwh = offs_h.pin_memory(), rewards_h.pin_memory()
        res = torch.empty(6, dtype=torch.float64).pin_memory()

        def step_e2e():
            a, b, m = (t.to(dev, non_blocking=True) for t in (lph, lmh, mh))
            o, r = offh.to(dev, non_blocking=True), rwh.to(dev, non_blocking=True)
            eng.acceptance_stats(a, b, m, out=stats)
            loss = eng.reinforce_zero(a, b, o, r, 8, mask=m, out_w_hat=w_hat, out_grad=grad,
                                      out_adv=adv)[0]
            res[:5].copy_(stats, non_blocking=True)
            res[5:].copy_(loss, non_blocking=True)
            torch.cuda.current_stream().synchronize()

        for _ in range(max(1, args.warmup)):
            step_e2e()
        barrier(pg, dev)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            step_e2e()
        t1 = time.perf_counter()
        barrier(pg, dev)
        e2e_ms = max_over_ranks(pg, (t1 - t0) * 1000.0 / args.steps, dev)
        e2e = {"value": world * T / (e2e_ms / 1000.0), "unit": UNIT, "ms_per_step": e2e_ms,
               "h2d_bytes_per_step": T * 9 + offh.numel() * 8 + B * 4,
               "d2h_bytes_per_step": 48}

    peaks, peak_src = load_peaks()
    algo = RL_BYTES_PER_TOKEN["reinforce_zero"] * T
    achieved = algo / (rz_ms / 1000.0) / 1e9
    peak = float(peaks["hbm_gbs"])
    roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": achieved / peak, "peak_source": f"{peak_src} hbm_gbs",
            "traffic": None, "kernel": "lp_reinforce_zero (rz_seq_kernel)",
            "kernel_ms": rz_ms, "algorithmic_per_launch": algo}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle

        oracle.build()
        a, b, m = lp.cpu().numpy(), lm.cpu().numpy(), mask.cpu().numpy()
        t0 = time.perf_counter()
        oracle.acceptance_stats(a, b, m)
        oracle.reinforce_zero(a, b, offs_h.numpy(), rewards_h.numpy(), 8, mask=m)
        dt = time.perf_counter() - t0
        cpu = {"value": T / dt, "unit": UNIT, "cores": 1, "kind": "oracle", "seconds": dt,
               "sample": f"the whole {T}-token stream: acceptance statistics + REINFORCE Zero"}
    eng.close()
    if rank != 0:
        return None
    return {
        "metric": "RL-epilogue tokens/sec (acceptance statistics + REINFORCE Zero loss)",
        "value": world * T / (ms_max / 1000.0), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32/f64",
        "data": "synthetic",
        "config": {"workload": "rl_epilogue", "T": T, "responses": B, "group_size": 8,
                   "l2": "inputs smaller than L2 (19 MB); each step re-reads them",
                   "step": "lp_acceptance_stats + lp_reinforce_zero"},
        "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches[0],
        "clocks": clocks,
    }


# ----------------------------------------------------------------------------- backward
def run_backward(args, world, rank, local, pg):
    """The logprob backward over the workload's batch: dl = g (onehot - p) from the forward's
    logits (the leaf GEMM's gradient epilogue), then dX = dl W and dW = dl^T X (the library's
    own tcgen05 GEMMs)."""
    import torch

    from bit_consistent_logprob_gb300 import Engine

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wl, lengths, X, W, ids = make_workload(args.workload, dev, seed_offset=rank, batch=args.batch,
                                           rows=args.rows)
    T, H, V, N = X.shape[0], wl.H, wl.V, wl.n_leaves
    eng = Engine(W, n_leaves=N, max_tokens=min(T, args.max_tokens))
    _, logZ = eng.logprobs(X, ids, return_logZ=True)
    g = torch.randn(T, generator=torch.Generator().manual_seed(wl.seed), dtype=torch.float32).to(dev)
    chunk = min(T, 4096)
    eng.backward_reserve(chunk)
    dX = torch.empty(T, H, dtype=torch.float32, device=dev)
    dW = torch.empty(V, H, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    launches = [0]

    def step():
        eng.logprobs_backward(X, ids, logZ, g, dX=dX, dW=dW)
        launches[0] += eng.last_launch_count

    for _ in range(args.warmup):
        step()
    eng.check()
    torch.cuda.synchronize()
    launches[0] = 0
    eng.profile_enable(True)
    sampler = ClockSampler(local)
    time.sleep(0.3)
    barrier(pg, dev)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(pg, dev)
    clocks = sampler.stop()
    from bit_consistent_logprob_gb300._native import LP_PROFILE_GRAD_DW, LP_PROFILE_GRAD_DX

    dx_ms, dx_n = eng.profile_read_kind(LP_PROFILE_GRAD_DX)
    dw_ms, dw_n = eng.profile_read_kind(LP_PROFILE_GRAD_DW)
    gemm_ms, gemm_n = eng.profile_read()
    eng.profile_enable(False)
    eng.check()
    ms = max_over_ranks(pg, e0.elapsed_time(e1) / args.steps, dev)
    peaks, peak_src = load_peaks()
    grad_ms = gemm_ms / max(1, gemm_n)
    per_launch = 2.0 * T * H * V / (gemm_n / max(1, args.steps))
    achieved = per_launch / (grad_ms / 1000.0) / 1e12
    peak, src = tensor_peak(peaks, peak_src, ms * args.steps / 1000.0, False)
    # the two GEMMs of the backward, each 2 * T * H * V flop per step, against the same peak
    grad_gemms = {}
    for name, tot, cnt in (("dX = dl W (grad_gemm_kernel, K split summed)", dx_ms, dx_n),
                           ("dW += dl^T X (grad_gemm_kernel)", dw_ms, dw_n)):
        step_ms = tot / max(1, args.steps)
        tf = 2.0 * T * H * V / (step_ms / 1000.0) / 1e12 if step_ms > 0 else None
        grad_gemms[name] = {"ms_per_step": step_ms, "launches_per_step": cnt / max(1, args.steps),
                            "achieved": tf, "unit": "TFLOP/s", "peak": peak,
                            "frac": tf / peak if tf else None}
    roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
            "frac": achieved / peak, "peak_source": src,
            "traffic": None, "kernel": "leaf_gemm_kernel<gradient epilogue>",
            "kernel_ms": grad_ms, "algorithmic_per_launch": per_launch}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import numpy as np

        import oracle

        oracle.build()
        rows = np.array([0, T // 2, T - 1])
        t0 = time.perf_counter()
        oracle.logprob_grad(X[rows].cpu(), W.cpu(), ids.cpu().numpy()[rows],
                            g.cpu().double().numpy()[rows])
        dt = time.perf_counter() - t0
        cpu = {"value": len(rows) / dt, "unit": UNIT, "cores": oracle.num_threads(),
               "kind": "oracle", "seconds": dt,
               "sample": f"{len(rows)} rows of the {wl.name} batch: their dX and dW terms"}
    eng.close()
    if rank != 0:
        return None
    return {
        "metric": "logprob-backward tokens/sec (dX and dW)", "value": world * T / (ms / 1000.0),
        "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 (dl bf16, fp32 accumulation)", "data": "synthetic",
        "config": {"workload": wl.name + "+backward", "T": T, "H": H, "V": V, "n_leaves": N,
                   "row_chunk": chunk, "step": "lp_logprobs_backward (dX and dW)",
                   "step_tflops": 3 * 2.0 * T * H * V / (ms / 1000.0) / 1e12},
        "roofline": roof, "grad_gemms": grad_gemms, "cpu_baseline": cpu, "e2e": None,
        "gpu_launches": launches[0], "clocks": clocks,
    }


# ----------------------------------------------------------------------------- our arm
BURST_SECONDS = 1.0  # a timed region shorter than this is a burst: the burst bf16 peak applies
IS_BYTES_PER_TOKEN = 12  # lp_importance_weights: reads log pi and log mu, writes w (fp32)


def tensor_peak(peaks, peak_src, timed_s: float, fp8: bool):
    """The bf16 (x 2 for fp8) tensor peak that matches the timed region: the burst figure for
    a region under BURST_SECONDS, the sustained (power-capped) figure for a longer one."""
    key = "bf16_tflops_sustained" if timed_s >= BURST_SECONDS else "bf16_tflops"
    peak = float(peaks[key])
    src = f"{peak_src} {key} (timed region {timed_s:.2f} s)"
    if fp8:  # dense fp8 = 2 x bf16 (nominal 4.5 / 2.25 PFLOP/s)
        peak *= 2.0
        src += " x 2, the nominal fp8/bf16 ratio"
    return peak, src


def forward_roofline(workload, fp8, T, H, V, gemm_avg_ms, launches_per_step, timed_s):
    """Roofline record of the dominant kernel (the fused leaf GEMM) of one forward step."""
    peaks, peak_src = load_peaks()
    if workload == "ds_decode":
        # HBM-bound: W streamed once per step plus X and the per-tile partials.
        nb = (V + 63) // 64  # (max, sum-exp) partial per 64-column tile
        wbytes = H * V + 4 * ((V + 127) // 128) * (H // 128) if fp8 else 2 * H * V
        xbytes = T * H + 4 * T * (H // 128) if fp8 else 2 * T * H
        algo = (wbytes + xbytes + 8 * T * nb + 8 * T) / launches_per_step
        achieved = algo / (gemm_avg_ms / 1000.0) / 1e9
        peak = float(peaks["hbm_gbs"])
        return {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "peak_source": f"{peak_src} hbm_gbs",
                "algorithmic_per_launch": algo, "kernel_ms": gemm_avg_ms}
    algo = 2.0 * T * H * V / launches_per_step
    achieved = algo / (gemm_avg_ms / 1000.0) / 1e12
    peak, src = tensor_peak(peaks, peak_src, timed_s, fp8)
    return {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
            "frac": achieved / peak, "peak_source": src, "algorithmic_per_launch": algo,
            "kernel_ms": gemm_avg_ms}


def time_forward(eng, X, ids, mu, phase, steps, warmup, entropy, dev, local, pg):
    """Warm up, then time `steps` forward steps (logprobs [+ entropy] + importance weights)
    with CUDA events on the launching stream, the leaf GEMM bracketed by the library's
    profiling events and the importance-weight call by events of its own."""
    import torch

    T = X.shape[0]
    logp = torch.empty(T, dtype=torch.float32, device=dev)
    w = torch.empty(T, dtype=torch.float32, device=dev)
    d3 = torch.empty(1, dtype=torch.float64, device=dev)
    nv = torch.empty(1, dtype=torch.int64, device=dev)
    ent = torch.empty(T, dtype=torch.float32, device=dev) if entropy else None
    logz = torch.empty(T, dtype=torch.float32, device=dev) if entropy else None
    stream = torch.cuda.current_stream()
    launches = [0]
    is_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(steps)]

    def step(k=None):
        if entropy:
            eng.logprobs_entropy(X, ids, out=logp, out_logZ=logz, out_entropy=ent, phase=phase)
        else:
            eng.logprobs(X, ids, out=logp, phase=phase)
        launches[0] += eng.last_launch_count
        if k is not None:
            is_ev[k][0].record(stream)
        eng.importance_weights(logp, mu, out_w=w, out_d3=d3, out_nvalid=nv)
        if k is not None:
            is_ev[k][1].record(stream)
        launches[0] += eng.last_launch_count

    for _ in range(warmup):
        step()
    eng.check()
    torch.cuda.synchronize()
    launches[0] = 0
    eng.profile_enable(True)
    sampler = ClockSampler(local)
    time.sleep(0.3)
    barrier(pg, dev)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for k in range(steps):
        step(k)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(pg, dev)
    clocks = sampler.stop()
    gemm_ms, gemm_n = eng.profile_read()
    eng.profile_enable(False)
    eng.check()
    ms = e0.elapsed_time(e1) / steps
    is_ms = sum(a.elapsed_time(b) for a, b in is_ev) / steps
    return {"ms": ms, "ms_max": max_over_ranks(pg, ms, dev), "gemm_ms": gemm_ms,
            "gemm_n": gemm_n, "is_ms": is_ms, "launches": launches[0], "clocks": clocks}


def decode_subrecord(args, batch, rank, dev, local, pg):
    """One decode batch of the DeepSeek-like shape (H 7168, V 129280, N 8), timed like the
    main line: its tokens/s and the leaf GEMM's HBM roofline."""
    from bit_consistent_logprob_gb300 import Engine, LP_PHASE_DECODE

    wl, _, X, W, ids = make_workload("ds_decode", dev, seed_offset=rank, batch=batch)
    mu = rollout_logprobs(W, X, ids, wl, wl.seed + rank, batch)
    steps = max(args.steps, 500)  # a decode step is ~0.3 ms: enough steps for clock samples
    with Engine(W, n_leaves=wl.n_leaves, max_tokens=batch) as eng:
        r = time_forward(eng, X, ids, mu, LP_PHASE_DECODE, steps, args.warmup, False, dev,
                         local, pg)
    gemm_avg = r["gemm_ms"] / max(1, r["gemm_n"])
    roof = forward_roofline("ds_decode", False, batch, wl.H, wl.V, gemm_avg,
                            r["gemm_n"] / steps, r["ms"] * steps / 1000.0)
    roof["traffic"] = recorded_traffic(f"ds_decode_b{batch}")
    roof["kernel"] = "leaf_gemm_kernel<fused>"
    return {"workload": "ds_decode", "batch": batch, "H": wl.H, "V": wl.V,
            "n_leaves": wl.n_leaves, "steps": steps,
            "value": batch / (r["ms_max"] / 1000.0), "unit": UNIT, "ms_per_step": r["ms_max"],
            "roofline": roof, "gpu_launches": r["launches"], "clocks": r["clocks"]}


def run_ours(args, world, rank, local, pg):
    import torch

    from bit_consistent_logprob_gb300 import Engine, LP_PHASE_DECODE, LP_PHASE_PREFILL

    assert torch.cuda.is_available(), "bench.py needs a CUDA device"
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wl, lengths, X, W, ids = make_workload(args.workload, dev, seed_offset=rank, batch=args.batch,
                                           rows=args.rows)
    T, H, V, N = X.shape[0], wl.H, wl.V, wl.n_leaves
    max_tokens = min(T, args.max_tokens)
    mu = rollout_logprobs(W, X, ids, wl, wl.seed + rank, max_tokens)
    eng = Engine(W, n_leaves=N, max_tokens=max_tokens, fp8=args.fp8)
    phase = LP_PHASE_DECODE if args.workload == "ds_decode" else LP_PHASE_PREFILL
    r = time_forward(eng, X, ids, mu, phase, args.steps, args.warmup, args.entropy, dev, local,
                     pg)
    ms_max = r["ms_max"]

    # end to end through the public API with host buffers (pinned), copies in the region
    e2e = None
    if not args.no_e2e and not args.entropy:
        # pinned host copies made directly (no pageable intermediate: 17 GB per rank at is_d3)
        Xh = torch.empty(X.shape, dtype=X.dtype, pin_memory=True)
        Xh.copy_(X)
        idsh = ids.cpu().pin_memory()
        muh = mu.cpu().pin_memory()
        logph = torch.empty(T, dtype=torch.float32).pin_memory()
        wh = torch.empty(T, dtype=torch.float32).pin_memory()

        def step_e2e():
            eng.logprobs_host(Xh, idsh, out=logph)
            return eng.importance_weights_host(logph, muh, out_w=wh)

        for _ in range(max(1, args.warmup)):
            step_e2e()
        torch.cuda.synchronize()
        barrier(pg, dev)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            step_e2e()
        t1 = time.perf_counter()
        barrier(pg, dev)
        e2e_ms = max_over_ranks(pg, (t1 - t0) * 1000.0 / args.steps, dev)
        bi = T * H * 2 + T * 4 + T * 4 + T * 4
        bo = T * 4 + T * 4 + 16
        e2e = {"value": world * T / (e2e_ms / 1000.0), "unit": UNIT, "ms_per_step": e2e_ms,
               "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo}
        del Xh

    gemm_avg_ms = r["gemm_ms"] / max(1, r["gemm_n"])
    timed_s = r["ms"] * args.steps / 1000.0
    roof = forward_roofline(args.workload, args.fp8, T, H, V, gemm_avg_ms,
                            r["gemm_n"] / max(1, args.steps), timed_s)
    key = args.workload + ("_fp8" if args.fp8 else "") + ("_entropy" if args.entropy else "")
    if args.workload == "ds_decode":
        key += f"_b{args.batch}"
    # the recorded traffic is for a full-size launch; a --rows case has none
    roof["traffic"] = recorded_traffic(key) if not args.rows else None
    roof["kernel"] = ("leaf_gemm_fp8_kernel" if args.fp8 else
                      "leaf_gemm_kernel<fused, entropy>" if args.entropy else "leaf_gemm_kernel<fused>")
    roof["timed_region_s"] = timed_s
    roof["launches_per_step"] = r["gemm_n"] / max(1, args.steps)

    # the importance-weight epilogue's own bandwidth: 12 bytes per token against HBM
    peaks, peak_src = load_peaks()
    is_algo = IS_BYTES_PER_TOKEN * T + 16
    is_gbs = is_algo / (r["is_ms"] / 1000.0) / 1e9
    epilogue = {"kernel": "lp_importance_weights (is_fused_kernel)",
                "bound": "hbm", "achieved": is_gbs, "peak": float(peaks["hbm_gbs"]),
                "unit": "GB/s", "frac": is_gbs / float(peaks["hbm_gbs"]),
                "peak_source": f"{peak_src} hbm_gbs", "kernel_ms": r["is_ms"],
                "algorithmic_per_launch": is_algo,
                "note": f"{is_algo / 1e6:.1f} MB per call; log pi was just written by the "
                        "combine, so part of the stream may come from L2 (129 MB)"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not args.fp8:
        cpu = cpu_baseline(X, W, ids, mu, wl, rows=args.cpu_rows)
    eng.close()
    del X, W, ids, mu
    torch.cuda.empty_cache()

    decode = None
    if args.decode_batches and not args.fp8 and not args.entropy and args.workload != "ds_decode":
        decode = [decode_subrecord(args, int(b), rank, dev, local, pg)
                  for b in args.decode_batches.split(",")]

    if rank != 0:
        return None
    value = world * T / (ms_max / 1000.0)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3 block-FP8" if args.fp8 else "bf16",
        "data": "synthetic",
        "config": {"workload": wl.name + ("+fp8" if args.fp8 else ""), "T": T, "H": H, "V": V, "n_leaves": N,
                   "n_seqs": len(lengths), "phase": "decode" if phase == LP_PHASE_DECODE else "prefill",
                   "parallelism": f"replicas{world}" if world > 1 else "single-gpu",
                   "row_chunk": max_tokens,
                   **({"rows_kept": args.rows} if args.rows else {}),
                   "l2": f"inputs larger than L2 (W {2 * H * V / 1e6:.0f} MB streamed every step)",
                   "step": ("lp_logprobs_entropy" if args.entropy else "lp_logprobs")
                           + " + lp_importance_weights"},
        "roofline": roof, "epilogue": epilogue, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": r["launches"], "clocks": r["clocks"],
    }
    if decode is not None:
        line["decode"] = decode
    return line


def cpu_baseline(X, W, ids, mu, wl, rows: int):
    """The fp64 oracle, as it stands, on a seeded row sample of the same workload."""
    import numpy as np
    import torch

    import oracle

    T = X.shape[0]
    rng = np.random.default_rng(wl.seed)
    sample = np.sort(rng.choice(T, size=min(rows, T), replace=False))
    idx = torch.as_tensor(sample, device=X.device)
    Xh, Wh = X[idx].cpu(), W.cpu()        # only the sampled rows travel to the host
    idsh = ids[idx].cpu().numpy()
    oracle.build()
    t0 = time.perf_counter()
    logp, _ = oracle.logprobs(Xh, Wh, idsh)
    oracle.importance_weights(logp.astype(np.float32), mu[idx].cpu().numpy())
    dt = time.perf_counter() - t0
    del torch
    return {"value": len(sample) / dt, "unit": UNIT, "cores": oracle.num_threads(),
            "kind": "oracle", "seconds": dt,
            "sample": f"{len(sample)} seeded rows of the {wl.name} batch (full vocabulary each), "
                      f"logprob + importance weight"}


# ----------------------------------------------------------------------------- reference arm
def run_reference_rl(args, world):
    """The oracle's acceptance statistics + REINFORCE Zero loss over the whole token stream."""
    import oracle

    wl, offs, rewards, lp, lm, mask = rl_inputs("cpu")
    a, b, m = lp.numpy(), lm.numpy(), mask.numpy()
    T = a.shape[0]
    oracle.build()

    def step():
        oracle.acceptance_stats(a, b, m)
        oracle.reinforce_zero(a, b, offs.numpy(), rewards.numpy(), 8, mask=m)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    value = T / dt
    return {
        "impl": "reference", "metric": "RL-epilogue tokens/sec (acceptance statistics + "
        "REINFORCE Zero loss)", "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1000.0,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": "rl_epilogue", "T": T, "responses": int(rewards.numel()),
                   "group_size": 8},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"the whole {T}-token stream per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_reference(args, world, rank):
    """The CPU oracle as the reference implementation, on a bounded row sample per step."""
    if rank != 0:
        return None
    if args.workload == "rl_epilogue":
        return run_reference_rl(args, world)
    import numpy as np

    import oracle
    from bit_consistent_logprob_gb300 import inputs

    wl = inputs.WORKLOADS[args.workload]
    if args.workload in ("qwen_prefill", "is_d3"):
        T = sum(inputs.packed_lengths(wl.n_seqs, wl.len_lo, wl.len_hi, wl.seed))
    elif args.workload == "ds_decode":
        T = args.batch
    else:
        T = wl.T
    oracle.build()
    # Rows generated on the host are a stand-in sample of the batch: the oracle cost per
    # row is H * V fp64 products whatever the row holds.
    W = inputs.lm_head(wl.V, wl.H, wl.seed)
    rng = np.random.default_rng(wl.seed)
    threads = oracle.num_threads()
    # calibrate on one row per thread (the oracle spreads rows over its OpenMP threads)
    Xp = inputs.hidden_states(threads, wl.H, wl.seed)
    idsp = inputs.uniform_ids(threads, wl.V, wl.seed)
    oracle.logprobs(Xp[:1], W, idsp[:1].numpy())  # start the thread pool
    t0 = time.perf_counter()
    oracle.logprobs(Xp, W, idsp.numpy())
    per_round = time.perf_counter() - t0
    rounds = max(1, round(args.ref_step_seconds / max(per_round, 1e-9)))
    rows = int(min(T, rounds * threads))
    Xs = inputs.hidden_states(rows, wl.H, wl.seed + 1)
    idss = inputs.uniform_ids(rows, wl.V, wl.seed + 1).numpy()
    mus = rng.standard_normal(rows).astype(np.float32) - 5.0

    def step():
        lp, _ = oracle.logprobs(Xs, W, idss)
        oracle.importance_weights(lp.astype(np.float32), mus)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    value = rows / dt
    sample = (f"{rows} rows per step of the {wl.name} workload (H={wl.H}, V={wl.V}), full "
              f"vocabulary per row, fp64 oracle")
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1000.0,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": wl.name, "T": T, "H": wl.H, "V": wl.V, "n_leaves": wl.n_leaves,
                   "sample_rows_per_step": rows},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="is_d3",
                    choices=("tiny", "qwen_prefill", "ds_prefill", "ds_decode", "is_d3",
                             "rl_epilogue"))
    ap.add_argument("--batch", type=int, default=128, help="rows of the decode workload")
    ap.add_argument("--rows", type=int, default=0,
                    help="keep only the workload's first ROWS tokens (a small case for profiler "
                         "captures; 0 = the whole workload)")
    ap.add_argument("--max-tokens", type=int, default=32768, help="row chunk of the engine")
    ap.add_argument("--cpu-rows", type=int, default=128, help="rows of the CPU-baseline sample")
    ap.add_argument("--ref-step-seconds", type=float, default=1.5)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--decode-batches", default="1,256",
                    help="decode batches (DeepSeek-like shape) timed after a prefill workload "
                         "and reported in the same line; empty to skip")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--entropy", action="store_true",
                    help="the step also forms each row's softmax entropy (lp_logprobs_entropy)")
    ap.add_argument("--backward", action="store_true",
                    help="time the logprob backward (dX, dW) instead of the forward step")
    ap.add_argument("--fp8", action="store_true",
                    help="block-FP8 (W8A8) handle: 1x128 activation, 128x128 weight blocks")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    return args


def main(argv=None):
    args = parse_args(argv)
    world, rank, local, pg = dist_setup()
    if args.gpus != world and world > 1:
        raise SystemExit(f"--gpus {args.gpus} but WORLD_SIZE={world}")
    if args.impl == "reference":
        line = run_reference(args, world, rank)
    elif args.workload == "rl_epilogue":
        line = run_rl_epilogue(args, world, rank, local, pg)
    elif args.backward:
        line = run_backward(args, world, rank, local, pg)
    else:
        line = run_ours(args, world, rank, local, pg)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
