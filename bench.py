#!/usr/bin/env python
"""Benchmark of the fused blockwise attention + FFN layer (forward + recompute
backward) on GB300, through the C ABI.

One step = bpt_layer_fwd + bpt_layer_bwd of one layer on one batch of seeded
synthetic input, everything resident in HBM.  Default workload: the GPT-3B
shaped layer at s = 32768 (h 2560, 32 heads x 80, FFN 10240, GeLU, LayerNorm,
causal) -- the configuration the headline metric is quoted on.

Prints ONE JSON line (rank 0).  --impl reference times the fp64 CPU oracle
instead, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused BPT layer fwd+bwd TFLOP/s and tokens/s at s=32K; % of bf16 tensor peak"
L2_BYTES = 129 * 1024 * 1024


# ----------------------------------------------------------------- FLOP count

def flop_counts(c) -> dict:
    """Algorithmic FLOPs (multiply-add = 2) of one layer, causal pairs exact.

    F_linear = 2 s h (H + 2 H_kv) d + 2 s H d h + 2 s h f n_mat
    F_attn   = 4 d H * (number of unmasked query/key pairs)   (~ 2 s^2 H d)
    forward  = F_linear + F_attn
    executed (fwd + recompute bwd) = forward + (forward - fc2) + 2 F_linear + 2.5 F_attn,
               less the Q/K/V projection (save policy 1) and also the attention
               forward (policy 2) that the backward then does not rebuild
    model    = 3 * forward"""
    s, h, H, Hk, d, f, b = c.s, c.h, c.n_heads, c.n_kv_heads, c.head_dim, c.ffn_dim, c.b
    n_mat = 3 if c.act == 2 else 2
    lin = b * (2 * s * h * (H + 2 * Hk) * d + 2 * s * H * d * h + 2 * s * h * f * n_mat)
    fc2 = b * 2 * s * f * h
    pairs = s * (s + 1) / 2 if c.causal else s * s
    attn = b * 4.0 * d * H * pairs
    fwd = lin + attn
    if not c.backward:
        return {"forward": fwd, "executed": fwd, "model": fwd, "linear": lin, "attn": attn}
    executed = fwd + (fwd - fc2) + 2 * lin + 2.5 * attn
    qkv = b * 2 * s * h * (H + 2 * Hk) * d
    save = getattr(c, "save_policy", 0)
    if c.head_chunk and c.head_chunk < H and save == 0:
        # Q/K/V of every stage is projected once more for the attention backward
        executed += qkv
    if save >= 1:
        executed -= qkv   # the backward takes the projections the forward kept
    if save >= 2:
        executed -= attn  # and the attention output
    return {"forward": fwd, "executed": executed, "model": 3 * fwd, "linear": lin, "attn": attn}


def vanilla_activation_bytes(c) -> int:
    """Activation bytes a vanilla (materialised, non-checkpointed) GPT layer
    keeps: 34 sbh + 5 a s^2 b ("Training memory: model states, activations and
    checkpointing", section 3)."""
    return 34 * c.s * c.b * c.h + 5 * c.n_heads * c.s * c.s * c.b


def vanilla_layer_bytes(c, inp, dev):
    """Device bytes of the plain materialised layer, for the memory
    comparison only (never for results): the layer written with PyTorch ops
    on the GPU in bf16, Q K^T and the probabilities materialised per head,
    every activation kept by autograd for a backward.  Returns the peak
    during the forward and the bytes still held after it, both above the
    inputs and weights."""
    import torch
    import torch.nn.functional as F

    W = {k: (None if v is None else v.detach().clone().requires_grad_(True)) for k, v in inp["weights"].items()}
    x = inp["x"].detach().clone().requires_grad_(True)
    b, s, h, H, Hk, d = c.b, c.s, c.h, c.n_heads, c.n_kv_heads, c.head_dim

    def norm(t, w, bias):
        if c.norm == 0:
            return F.layer_norm(t, (h,), w, bias, 1e-5)
        return t * torch.rsqrt(t.float().pow(2).mean(-1, keepdim=True) + 1e-5).to(t.dtype) * w

    def lin(t, w, bias=None):
        return F.linear(t, W[w], W[bias] if bias and W.get(bias) is not None else None)

    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats(dev)
    base = torch.cuda.memory_allocated(dev)
    xn = norm(x, W["ln1_w"], W.get("ln1_b"))
    q = lin(xn, "wq", "bq").view(b, s, H, d).transpose(1, 2)
    k = lin(xn, "wk", "bk").view(b, s, Hk, d).transpose(1, 2).repeat_interleave(H // Hk, dim=1)
    v = lin(xn, "wv", "bv").view(b, s, Hk, d).transpose(1, 2).repeat_interleave(H // Hk, dim=1)
    sc = (q @ k.transpose(-1, -2)) * (1.0 / d ** 0.5)
    if c.causal:
        sc = sc.masked_fill(torch.ones(s, s, dtype=torch.bool, device=dev).triu(1), float("-inf"))
    o = (torch.softmax(sc, dim=-1) @ v).transpose(1, 2).reshape(b, s, H * d)
    x1 = x + lin(o, "wo", "bo")
    x1n = norm(x1, W["ln2_w"], W.get("ln2_b"))
    if c.act == 2:
        a = F.silu(lin(x1n, "w1")) * lin(x1n, "w3")
    else:
        a = F.gelu(lin(x1n, "w1", "b1"), approximate="tanh" if c.act == 1 else "none")
    y = x1 + lin(a, "w2", "b2")
    torch.cuda.synchronize()
    peak = torch.cuda.max_memory_allocated(dev) - base
    held = torch.cuda.memory_allocated(dev) - base
    del y, a, x1n, x1, o, sc, q, k, v, xn
    torch.cuda.synchronize()
    return {"peak_bytes": int(peak), "held_after_forward_bytes": int(held),
            "what": "plain PyTorch bf16 layer on the GPU, scores and probabilities materialised, "
                    "activations kept for a backward (memory comparison only)"}


# ----------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampled every 200 ms while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self):
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        idx = vis.split(",")[0] if vis and vis.split(",")[0].isdigit() else None
        if idx is not None and any(r[0] == idx for r in rows):
            rows = [r for r in rows if r[0] == idx]
        else:
            first = rows[0][0] if rows else None
            rows = [r for r in rows if r[0] == first]

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        power = [num(r[3]) for r in rows if num(r[3]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows), "power_w_max": max(power) if power else None}


# ----------------------------------------------------------------- helpers

def load_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d.get("hbm_gbs", 6800.0), "bf16": d.get("bf16_tflops", 1872.7),
                "bf16_sustained": d.get("bf16_tflops_sustained", 1702.7), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16": 1900.0, "bf16_sustained": 1700.0, "source": "fallback"}


def load_traffic() -> dict:
    """Per-launch DRAM bytes of the dominant kernel from the committed ncu
    summary (null until a capture of the current kernel exists)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(p):
        try:
            return json.load(open(p))
        except ValueError:
            return {}
    return {}


# A rank that dies (or never arrives) must not leave the others waiting in a
# collective forever: every collective of the bench's process group gives up
# after this many seconds and raises.
PG_TIMEOUT_S = 600


def init_group(backend: str, timeout_s: float = PG_TIMEOUT_S):
    import datetime

    import torch.distributed as tdist
    tdist.init_process_group(backend, timeout=datetime.timedelta(seconds=timeout_s))


def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# Multi-rank host logic (one process per GPU, each a full replica of the layer
# step on its own seeded batch: the step shards by batch with no exchange).

def rank_seed(c, rank: int) -> int:
    """Seed of this rank's synthetic batch: every replica gets different data."""
    return c.seed + 101 * rank


def reports(rank: int) -> bool:
    """Only rank 0 prints the JSON line (and runs the reference arm)."""
    return rank == 0


def max_over_ranks(x: float, world: int, device="cpu") -> float:
    """The slowest rank's time: the job is done when every replica is."""
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as tdist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(flops_per_rank_step: float, world: int, ms: float) -> float:
    """Whole-job TFLOP/s: the work of all ranks over the slowest rank's time."""
    return flops_per_rank_step * world / (ms * 1e-3) / 1e12


def describe(c) -> dict:
    return {"workload": c.name, "b": c.b, "s": c.s, "h": c.h, "n_heads": c.n_heads,
            "n_kv_heads": c.n_kv_heads, "head_dim": c.head_dim, "ffn_dim": c.ffn_dim,
            "act": ["gelu-erf", "gelu-tanh", "swiglu"][c.act], "norm": ["layernorm", "rmsnorm"][c.norm],
            "causal": bool(c.causal), "q_block": c.q_block, "kv_block": c.kv_block,
            "ffn_block": c.ffn_block, "head_chunk": c.head_chunk or c.n_heads,
            "pass": "fwd+bwd" if c.backward else "fwd", "seed": c.seed,
            "l2": "no flush: every step streams inputs and buffers far larger than the 129 MB L2",
            **({"rope_base": c.rope_base} if c.rope_base else {}),
            **({"stage_order": ["contiguous", "interleaved"][c.stage_order]} if c.stage_order else {}),
            **({"save_policy": ["log-sum-exp", "+ Q/K/V", "+ Q/K/V and O"][c.save_policy]} if c.save_policy else {})}


# ----------------------------------------------------------------- CPU oracle leg

def oracle_sample(c, rows: int):
    """The fp64 CPU oracle on the first `rows` positions of the workload
    (same width, heads and FFN; a bounded sample)."""
    import numpy as np

    from blockwise_attention_ffn_gb300.synth import make_layer_inputs
    from oracle import ref
    sc = c.with_(s=rows)
    inp = make_layer_inputs(sc, seed=c.seed, device="cpu", with_dy=c.backward)
    W = {k: v.float().double().numpy() for k, v in inp["weights"].items() if v is not None}
    x = inp["x"].float().double().numpy()
    oc = ref.LayerCfg(s=rows, h=c.h, n_heads=c.n_heads, n_kv_heads=c.n_kv_heads, head_dim=c.head_dim,
                      ffn_dim=c.ffn_dim, b=c.b, causal=bool(c.causal), norm=c.norm, act=c.act,
                      has_bias=bool(c.has_bias), norm_eps=c.norm_eps, rope_base=float(c.rope_base))
    t0 = time.perf_counter()
    ref.layer_forward(x, W, oc)
    if c.backward:
        ref.layer_backward(x, W, inp["dy"].float().double().numpy(), oc)
    dt = time.perf_counter() - t0
    fl = flop_counts(sc)["executed"]
    del np
    return dt, fl, sc


def blas_threads() -> int:
    """Threads the oracle's BLAS runs on: what the BLAS library reports when
    threadpoolctl is installed, else the usual environment limits, else every
    host core."""
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n and n[0]:
            return int(n[0])
    except Exception:  # noqa: BLE001 - fall back to the environment
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        v = os.environ.get(var, "")
        if v.isdigit() and int(v) > 0:
            return min(int(v), os.cpu_count() or int(v))
    return os.cpu_count() or 1


def cpu_baseline(c, rows: int) -> dict:
    dt, fl, sc = oracle_sample(c, rows)
    return {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle",
            "seconds": dt,
            "sample": f"fp64 NumPy oracle, {'forward + backward' if c.backward else 'forward'} of the first {rows} positions of the "
                      f"workload (same layer shape), {fl / 1e12:.3f} TFLOP of the same FLOP "
                      f"definition; cores = the BLAS threads"}


def run_reference(args, c):
    ws, rank, _ = dist_setup()
    if not reports(rank):
        return 0
    times, fl = [], None
    for i in range(args.warmup + args.steps):
        dt, f, _ = oracle_sample(c, args.ref_rows)
        fl = f
        if i >= args.warmup:
            times.append(dt)
    t = sum(times) / len(times)
    val = fl / t / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": t * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic", "config": describe(c),
            "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle",
                             "sample": f"first {args.ref_rows} positions of the workload per step"},
            "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------- GPU leg

def run_gpu(args, c):
    import torch
    import torch.distributed as tdist

    import blockwise_attention_ffn_gb300 as bpt
    from blockwise_attention_ffn_gb300.synth import make_layer_inputs

    world, rank, local = dist_setup()
    if world > 1:
        init_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    bpt.lib()

    inp = make_layer_inputs(c, seed=rank_seed(c, rank), device=dev, with_dy=c.backward)
    W = inp["weights"]
    x = inp["x"]
    dy = inp.get("dy")
    y = torch.empty_like(x)
    saved = bpt.alloc_bytes(bpt.bpt_saved_bytes(c), dev)
    ws_bytes = bpt.bpt_workspace_bytes(c, bpt.BPT_PASS_FWD)
    if c.backward:
        ws_bytes = max(ws_bytes, bpt.bpt_workspace_bytes(c, bpt.BPT_PASS_BWD))
    torch.cuda.synchronize()
    base_mem = torch.cuda.memory_allocated(dev)
    ws = bpt.alloc_bytes(ws_bytes, dev)
    dx = torch.empty_like(x)
    grads = bpt.alloc_grads(W, dev) if c.backward else None
    stream = torch.cuda.current_stream(dev)

    def step(cfg=c):
        bpt.bpt_layer_fwd(cfg, W, x, y, saved, ws, stream)
        if cfg.backward:
            bpt.bpt_layer_bwd(cfg, W, x, saved, dy, dx, grads, ws, stream)

    torch.cuda.reset_peak_memory_stats(dev)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    st_, site = bpt.bpt_last_device_error(stream)
    if st_ != bpt.BPT_OK:
        raise RuntimeError(f"device error {st_} at wait site {site}")
    peak_mem = torch.cuda.max_memory_allocated(dev)

    clocks = ClockSampler()
    if rank == 0:
        clocks.start()
    if world > 1:
        tdist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        tdist.barrier()
    ms = e0.elapsed_time(e1) / args.steps
    clk = clocks.stop() if rank == 0 else None
    ms = max_over_ranks(ms, world, dev)
    st_, site = bpt.bpt_last_device_error(stream)
    if st_ != bpt.BPT_OK:
        raise RuntimeError(f"device error {st_} at wait site {site}")

    fl = flop_counts(c)
    value = job_throughput(fl["executed"], world, ms)
    peaks = load_peaks()

    # the two passes timed on their own, the same way (forward: K forward
    # calls; backward: K backward calls on the log-sum-exp the last forward
    # saved).  Supplementary: a failure here is reported, not raised.
    passes = None
    if c.backward:
        try:
            p0, p1, p2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
            torch.cuda.synchronize()
            p0.record(stream)
            for _ in range(args.steps):
                bpt.bpt_layer_fwd(c, W, x, y, saved, ws, stream)
            p1.record(stream)
            for _ in range(args.steps):
                bpt.bpt_layer_bwd(c, W, x, saved, dy, dx, grads, ws, stream)
            p2.record(stream)
            torch.cuda.synchronize()
            fwd_ms = max_over_ranks(p0.elapsed_time(p1) / args.steps, world, dev)
            bwd_ms = max_over_ranks(p1.elapsed_time(p2) / args.steps, world, dev)
            passes = {"fwd_ms": fwd_ms, "bwd_ms": bwd_ms,
                      "fwd_tflops": job_throughput(fl["forward"], world, fwd_ms),
                      "bwd_tflops": job_throughput(fl["executed"] - fl["forward"], world, bwd_ms),
                      "note": "each pass timed alone over the same K calls; the step above runs both"}
        except Exception as e:  # noqa: BLE001 - reported in the line
            passes = {"error": repr(e)}

    # per-kernel breakdown of the same step (separate profiled steps).  These
    # run every kernel on one stream, so that no event span also covers
    # weight-gradient work overlapping on the backward's second stream.
    one = c.with_(flags=c.flags | bpt.BPT_FLAG_ONE_STREAM)
    bpt.bpt_profile_enable(True)
    nprof = max(1, min(args.steps, 3))
    for _ in range(nprof):
        step(one)
    torch.cuda.synchronize()
    prof = bpt.bpt_profile_collect()
    bpt.bpt_profile_enable(False)
    launches_per_step = sum(v["launches"] for v in prof.values()) / nprof
    tot_ms = sum(v["ms"] for v in prof.values())
    kernels = {}
    for k, v in prof.items():
        if v["launches"]:
            kernels[k] = {"launches_per_step": v["launches"] / nprof, "ms_per_step": v["ms"] / nprof,
                          "share": v["ms"] / tot_ms if tot_ms else None,
                          "tflops": (v["flops"] / (v["ms"] * 1e-3) / 1e12) if v["flops"] else None,
                          "gbs": (v["bytes"] / (v["ms"] * 1e-3) / 1e9) if v["bytes"] else None}
    dom = max(prof, key=lambda k: prof[k]["ms"])
    dv = prof[dom]
    traffic = load_traffic().get(dom)
    if dv["flops"]:
        ach = dv["flops"] / (dv["ms"] * 1e-3) / 1e12
        roof = {"kernel": dom, "bound": "tensor", "achieved": ach, "peak": peaks["bf16_sustained"],
                "unit": "TFLOP/s", "frac": ach / peaks["bf16_sustained"],
                "frac_of_burst_peak": ach / peaks["bf16"],
                "peak_note": f"{peaks['source']} bf16 sustained (kernel timed inside the long step)",
                "per_launch_flops": dv["flops"] / dv["launches"],
                "avg_launch_ms": dv["ms"] / dv["launches"], "traffic": traffic}
    else:
        ach = dv["bytes"] / (dv["ms"] * 1e-3) / 1e9
        roof = {"kernel": dom, "bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": ach / peaks["hbm_gbs"], "peak_note": f"{peaks['source']} HBM copy bandwidth",
                "per_launch_bytes": dv["bytes"] / dv["launches"],
                "avg_launch_ms": dv["ms"] / dv["launches"], "traffic": traffic}

    # end to end through the C ABI from pinned host buffers.  Every step
    # copies its x and dy in and its dx out inside the timed region, the way
    # a training loop prefetches its next batch: x alternates between two
    # device buffers, and the next step's x comes in on a copy stream while
    # this step's backward runs; dy comes in on that stream while the forward
    # runs (after the previous backward has read it), and dx goes out on a
    # third stream while the next step's forward runs (the next backward,
    # which overwrites dx, waits for it).
    xh = x.cpu().pin_memory()
    dyh = dy.cpu().pin_memory() if c.backward else None
    outh = torch.empty_like(xh).pin_memory()
    xs = [x, torch.empty_like(x)] if c.backward else [x]
    h2d_st, d2h_st = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_x = [torch.cuda.Event() for _ in xs]
    ev_dy, ev_bwd, ev_out = (torch.cuda.Event() for _ in range(3))
    n_e2e = [0]

    def step_e2e():
        if not c.backward:
            x.copy_(xh, non_blocking=True)
            bpt.bpt_layer_fwd(c, W, x, y, saved, ws, stream)
            outh.copy_(y, non_blocking=True)
            return
        k = n_e2e[0]
        xk = xs[k % 2]
        if k == 0:
            with torch.cuda.stream(h2d_st):
                xk.copy_(xh, non_blocking=True)
                ev_x[0].record(h2d_st)
        stream.wait_event(ev_x[k % 2])
        bpt.bpt_layer_fwd(c, W, xk, y, saved, ws, stream)
        if k:
            h2d_st.wait_event(ev_bwd)  # the previous backward has read dy and the other x
        with torch.cuda.stream(h2d_st):
            dy.copy_(dyh, non_blocking=True)
            ev_dy.record(h2d_st)
            xs[(k + 1) % 2].copy_(xh, non_blocking=True)  # the next step's x
            ev_x[(k + 1) % 2].record(h2d_st)
        stream.wait_event(ev_dy)
        if k:
            stream.wait_event(ev_out)  # the previous dx has been copied out
        bpt.bpt_layer_bwd(c, W, xk, saved, dy, dx, grads, ws, stream)
        ev_bwd.record(stream)
        d2h_st.wait_event(ev_bwd)
        with torch.cuda.stream(d2h_st):
            outh.copy_(dx, non_blocking=True)
            ev_out.record(d2h_st)
        n_e2e[0] += 1

    for _ in range(max(1, args.warmup // 2)):
        step_e2e()
    torch.cuda.synchronize()
    if world > 1:
        tdist.barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step_e2e()
    torch.cuda.synchronize()
    e2e_ms = (time.perf_counter() - t0) * 1e3 / args.steps
    e2e_ms = max_over_ranks(e2e_ms, world, dev)
    h2d = xh.numel() * xh.element_size() + (dyh.numel() * dyh.element_size() if c.backward else 0)
    d2h = outh.numel() * outh.element_size()

    if reports(rank):
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) inputs, N(0,0.02) weights)",
            "config": describe(c),
            "flops_per_step": {"executed": fl["executed"], "model": fl["model"], "forward": fl["forward"]},
            "tokens_per_s": c.b * c.s * world / (ms * 1e-3),
            "model_tflops": fl["model"] * world / (ms * 1e-3) / 1e12,
            "pct_of_bf16_peak": 100 * value / (peaks["bf16"] * world),
            "pct_of_bf16_peak_sustained": 100 * value / (peaks["bf16_sustained"] * world),
            "peak_source": peaks["source"],
            "clocks": clk,
            "e2e": {"value": job_throughput(fl["executed"], world, e2e_ms), "unit": "TFLOP/s", "ms_per_step": e2e_ms,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "what": "pinned host x (and dy) copied in, fwd+bwd through the C ABI, dx copied out; the next "
                            "step's x comes in during this step's backward, into the other of two device buffers"},
            "gpu_launches": int(round(launches_per_step * args.steps)),
            "roofline": roof, "kernels": kernels, "passes": passes,
            "memory": {"peak_device_bytes": peak_mem, "inputs_weights_grads_bytes": base_mem,
                       "workspace_bytes": ws_bytes, "saved_bytes": bpt.bpt_saved_bytes(c),
                       "vanilla_layer_activation_bytes_analytic": vanilla_activation_bytes(c)},
        }
        # the materialised layer where it fits comfortably (the analytic
        # estimate under 32 GB: the forward-only workloads)
        if vanilla_activation_bytes(c) < 32 * 2 ** 30:
            try:
                line["memory"]["vanilla_layer_measured"] = vanilla_layer_bytes(c, inp, dev)
            except Exception as e:  # noqa: BLE001 - reported in the line
                line["memory"]["vanilla_layer_measured"] = {"error": repr(e)}
        if not args.no_cpu_baseline and world == 1:
            # a reported baseline, not the measurement: a failure here must not
            # cost the line
            try:
                line["cpu_baseline"] = cpu_baseline(c, min(args.cpu_rows, c.s))
            except Exception as e:  # noqa: BLE001 - reported in the line
                line["cpu_baseline"] = {"error": repr(e), "kind": "oracle"}
        print(json.dumps(line), flush=True)
    if world > 1:
        tdist.barrier()
        tdist.destroy_process_group()
    return 0


def lm_flops(c) -> dict:
    """Algorithmic FLOPs of the language-model loss step: the logits 2 n h V
    in the forward; the backward rebuilds them and forms dx = dz W and
    dW = dz^T x, 2 n h V each."""
    f = 2.0 * c.n * c.h * c.vocab
    return {"forward": f, "executed": 4 * f, "model": 3 * f}


def describe_lm(c) -> dict:
    return {"workload": c.name, "n": c.n, "h": c.h, "vocab": c.vocab,
            "vocab_block": c.vocab_block or min(8192, (c.vocab + 255) // 256 * 256), "pass": "fwd+bwd",
            "seed": c.seed, "l2": "no flush: x, W and dW alone are 0.9 GB, far larger than the 129 MB L2"}


def cpu_baseline_lm(c, rows: int) -> dict:
    import numpy as np  # noqa: F401

    from blockwise_attention_ffn_gb300.synth import make_lm_inputs
    from oracle import lm_loss
    sc = c.with_(n=rows)
    inp = make_lm_inputs(sc, seed=c.seed)
    x, w, t = inp["x"].double().numpy(), inp["w"].double().numpy(), inp["targets"].numpy()
    t0 = time.perf_counter()
    lm_loss.lm_loss(x, w, t)
    lm_loss.lm_loss_backward(x, w, t)
    dt = time.perf_counter() - t0
    fl = lm_flops(sc)["executed"]
    return {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle", "seconds": dt,
            "sample": f"fp64 NumPy oracle, loss and gradients of the first {rows} positions (same h and V), "
                      f"{fl / 1e12:.3f} TFLOP of the same FLOP definition; cores = the BLAS threads"}


def run_gpu_lm(args, c):
    """One step = bpt_lm_loss_fwd + bpt_lm_loss_bwd of the loss workload."""
    import torch
    import torch.distributed as tdist

    import blockwise_attention_ffn_gb300 as bpt
    from blockwise_attention_ffn_gb300.synth import make_lm_inputs

    world, rank, local = dist_setup()
    if world > 1:
        init_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    bpt.lib()
    inp = make_lm_inputs(c, seed=rank_seed(c, rank), device=dev)
    x, w, t = inp["x"], inp["w"], inp["targets"]
    loss = torch.empty(1, device=dev)
    lse = torch.empty(c.n, device=dev)
    dx = torch.empty_like(x)
    dw = torch.empty(c.vocab, c.h, device=dev)
    torch.cuda.synchronize()
    base_mem = torch.cuda.memory_allocated(dev)
    ws_bytes = max(bpt.bpt_lm_workspace_bytes(c, bpt.BPT_PASS_FWD), bpt.bpt_lm_workspace_bytes(c, bpt.BPT_PASS_BWD))
    ws = bpt.alloc_bytes(ws_bytes, dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        bpt.bpt_lm_loss_fwd(c, x, w, t, loss, lse, ws, stream)
        bpt.bpt_lm_loss_bwd(c, x, w, t, lse, 1.0, dx, dw, ws, stream)

    torch.cuda.reset_peak_memory_stats(dev)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if bpt.bpt_last_device_error(stream)[0] != bpt.BPT_OK:
        raise RuntimeError("device error in the warm-up")
    peak_mem = torch.cuda.max_memory_allocated(dev)
    clocks = ClockSampler()
    if rank == 0:
        clocks.start()
    if world > 1:
        tdist.barrier()
    torch.cuda.synchronize()
    e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        tdist.barrier()
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, dev)
    clk = clocks.stop() if rank == 0 else None
    # the forward alone
    e0.record(stream)
    for _ in range(args.steps):
        bpt.bpt_lm_loss_fwd(c, x, w, t, loss, lse, ws, stream)
    e2.record(stream)
    torch.cuda.synchronize()
    fwd_ms = max_over_ranks(e0.elapsed_time(e2) / args.steps, world, dev)
    fl = lm_flops(c)
    value = job_throughput(fl["executed"], world, ms)
    peaks = load_peaks()
    bpt.bpt_profile_enable(True)
    nprof = max(1, min(args.steps, 3))
    for _ in range(nprof):
        step()
    torch.cuda.synchronize()
    prof = bpt.bpt_profile_collect()
    bpt.bpt_profile_enable(False)
    tot_ms = sum(v["ms"] for v in prof.values())
    kernels = {k: {"launches_per_step": v["launches"] / nprof, "ms_per_step": v["ms"] / nprof,
                   "share": v["ms"] / tot_ms if tot_ms else None,
                   "tflops": (v["flops"] / (v["ms"] * 1e-3) / 1e12) if v["flops"] else None,
                   "gbs": (v["bytes"] / (v["ms"] * 1e-3) / 1e9) if v["bytes"] else None}
               for k, v in prof.items() if v["launches"]}
    g = prof["gemm"]
    ach = g["flops"] / (g["ms"] * 1e-3) / 1e12
    roof = {"kernel": "gemm", "bound": "tensor", "achieved": ach, "peak": peaks["bf16_sustained"], "unit": "TFLOP/s",
            "frac": ach / peaks["bf16_sustained"], "frac_of_burst_peak": ach / peaks["bf16"],
            "peak_note": f"{peaks['source']} bf16 sustained (kernel timed inside the long step)",
            "per_launch_flops": g["flops"] / g["launches"], "avg_launch_ms": g["ms"] / g["launches"],
            "traffic": load_traffic().get("lm_gemm")}
    launches = sum(v["launches"] for v in prof.values()) / nprof
    # end to end: x and the targets in from pinned host memory, dx and the
    # loss back
    # dx leaves on a second stream while the next step's copies in and
    # forward run; the next backward, which overwrites dx, waits for it
    xh, th = x.cpu().pin_memory(), t.cpu().pin_memory()
    dxh, lh = torch.empty_like(xh).pin_memory(), torch.empty(1).pin_memory()
    copy_st = torch.cuda.Stream(dev)
    ev_used, ev_out = torch.cuda.Event(), torch.cuda.Event()
    n_e2e = [0]

    def step_e2e():
        x.copy_(xh, non_blocking=True)
        t.copy_(th, non_blocking=True)
        bpt.bpt_lm_loss_fwd(c, x, w, t, loss, lse, ws, stream)
        if n_e2e[0]:
            stream.wait_event(ev_out)
        bpt.bpt_lm_loss_bwd(c, x, w, t, lse, 1.0, dx, dw, ws, stream)
        lh.copy_(loss, non_blocking=True)  # on this stream: the next forward rewrites it
        ev_used.record(stream)
        copy_st.wait_event(ev_used)
        with torch.cuda.stream(copy_st):
            dxh.copy_(dx, non_blocking=True)
            ev_out.record(copy_st)
        n_e2e[0] += 1

    for _ in range(max(1, args.warmup // 2)):
        step_e2e()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step_e2e()
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks((time.perf_counter() - t0) * 1e3 / args.steps, world, dev)
    if reports(rank):
        line = {
            "metric": "blockwise LM loss (vocabulary projection + cross-entropy) fwd+bwd TFLOP/s and tokens/s",
            "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) x, N(0,0.02) W, uniform targets)", "config": describe_lm(c),
            "flops_per_step": fl, "tokens_per_s": c.n * world / (ms * 1e-3),
            "pct_of_bf16_peak": 100 * value / (peaks["bf16"] * world),
            "pct_of_bf16_peak_sustained": 100 * value / (peaks["bf16_sustained"] * world),
            "peak_source": peaks["source"], "clocks": clk,
            "passes": {"fwd_ms": fwd_ms, "fwd_tflops": job_throughput(fl["forward"], world, fwd_ms)},
            "e2e": {"value": job_throughput(fl["executed"], world, e2e_ms), "unit": "TFLOP/s", "ms_per_step": e2e_ms,
                    "h2d_bytes_per_step": xh.numel() * 2 + th.numel() * 4,
                    "d2h_bytes_per_step": dxh.numel() * 2 + 4,
                    "what": "pinned host x and targets copied in, loss fwd+bwd through the C ABI, dx and the loss out"},
            "gpu_launches": int(round(launches * args.steps)), "roofline": roof, "kernels": kernels,
            "memory": {"peak_device_bytes": peak_mem, "inputs_weights_grads_bytes": base_mem,
                       "workspace_bytes": ws_bytes, "logits_bytes_bf16_not_held": 2 * c.n * c.vocab},
        }
        if not args.no_cpu_baseline and world == 1:
            try:
                line["cpu_baseline"] = cpu_baseline_lm(c, min(args.cpu_rows, c.n))
            except Exception as e:  # noqa: BLE001 - reported in the line
                line["cpu_baseline"] = {"error": repr(e), "kind": "oracle"}
        print(json.dumps(line), flush=True)
    if world > 1:
        tdist.barrier()
        tdist.destroy_process_group()
    return 0


def run_one_kernel(args, c):
    """One launch of one component at the workload's shape with a shorter
    sequence (--seq), for profiler captures of a small case."""
    import torch

    import blockwise_attention_ffn_gb300 as bpt
    sc = c.with_(s=args.seq)
    H, Hk, d, s = sc.n_heads, sc.n_kv_heads, sc.head_dim, sc.s
    g = torch.Generator(device="cuda").manual_seed(0)
    qkv = torch.randn(sc.b * s, (H + 2 * Hk) * d, generator=g, device="cuda").to(torch.bfloat16)
    o = torch.empty(sc.b * s, H * d, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(sc.b, H, bpt.s_pad(sc), dtype=torch.float32, device="cuda")
    bpt.bpt_attention_fwd(sc, qkv, o, lse)
    if args.profile_kernel == "attn_bwd":
        dout = torch.randn(sc.b * s, H * d, generator=g, device="cuda").to(torch.bfloat16)
        dqkv = torch.empty_like(qkv)
        ws = bpt.alloc_bytes(bpt.bpt_attention_bwd_workspace_bytes(sc))
        bpt.bpt_attention_bwd(sc, qkv, o, lse, dout, dqkv, ws)
    elif args.profile_kernel == "layer":
        from blockwise_attention_ffn_gb300.synth import make_layer_inputs
        inp = make_layer_inputs(sc, seed=0, device="cuda", with_dy=True)
        y = torch.empty_like(inp["x"])
        saved = bpt.alloc_bytes(bpt.bpt_saved_bytes(sc))
        ws = bpt.alloc_bytes(max(bpt.bpt_workspace_bytes(sc, 0), bpt.bpt_workspace_bytes(sc, 1)))
        bpt.bpt_layer_fwd(sc, inp["weights"], inp["x"], y, saved, ws)
        dx = torch.empty_like(inp["x"])
        bpt.bpt_layer_bwd(sc, inp["weights"], inp["x"], saved, inp["dy"], dx, bpt.alloc_grads(inp["weights"]), ws)
    torch.cuda.synchronize()
    st_, site = bpt.bpt_last_device_error()
    print(json.dumps({"profile_kernel": args.profile_kernel, "seq": args.seq, "status": st_}))
    return 0 if st_ == bpt.BPT_OK else 1


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="c3",
                    help="c1..c5 (default c3, the s=32K workload); lm3: the language-model loss after it")
    ap.add_argument("--ref-rows", type=int, default=1024,
                    help="positions of the workload the CPU oracle runs per step of --impl reference")
    ap.add_argument("--cpu-rows", type=int, default=4096,
                    help="positions of the workload (at most s) in the cpu_baseline sample of the "
                         "GPU run: about 10-15 s of fp64 work on 16 host cores at the s=32K workload")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--rope-base", type=float, default=0.0,
                    help="rotary position embedding base for the layer (0: none, the workloads' setting)")
    ap.add_argument("--head-chunk", type=int, default=None,
                    help="query heads per stage U (the workload's own by default)")
    ap.add_argument("--stage-order", type=int, default=0, choices=[0, 1],
                    help="head-chunk stage order: 0 contiguous, 1 interleaved over the key/value groups")
    ap.add_argument("--ffn-block", type=int, default=None,
                    help="rows per FFN block c_f (the workload's own by default)")
    ap.add_argument("--save-policy", type=int, default=0, choices=[0, 1, 2],
                    help="kept for the backward: 0 the log-sum-exp, 1 + Q/K/V, 2 + the attention output")
    ap.add_argument("--profile-kernel", choices=["attn_fwd", "attn_bwd", "layer"], default=None,
                    help="run one launch of this component (small case for profiler captures)")
    ap.add_argument("--seq", type=int, default=4096, help="sequence length for --profile-kernel")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    from blockwise_attention_ffn_gb300.presets import LM3, PRESETS
    if args.config == "lm3":
        if args.impl == "reference":
            ws, rank, _ = dist_setup()
            if reports(rank):
                cb = cpu_baseline_lm(LM3, args.cpu_rows)
                print(json.dumps({"impl": "reference", "metric": "blockwise LM loss fwd+bwd TFLOP/s",
                                  "value": cb["value"], "unit": "TFLOP/s", "n_gpus": args.gpus,
                                  "steps": 1, "warmup": 0, "ms_per_step": cb["seconds"] * 1e3,
                                  "higher_is_better": True, "dtype": "f64", "config": describe_lm(LM3),
                                  "cpu_baseline": cb}), flush=True)
            return 0
        return run_gpu_lm(args, LM3)
    c = PRESETS[args.config]
    if args.rope_base:
        c = c.with_(rope_base=args.rope_base)
    if args.head_chunk is not None:
        c = c.with_(head_chunk=args.head_chunk)
    if args.ffn_block is not None:
        c = c.with_(ffn_block=args.ffn_block)
    if args.stage_order or args.save_policy:
        c = c.with_(stage_order=args.stage_order, save_policy=args.save_policy)
    if args.profile_kernel:
        return run_one_kernel(args, c)
    if args.impl == "reference":
        return run_reference(args, c)
    return run_gpu(args, c)


if __name__ == "__main__":
    sys.exit(main())
