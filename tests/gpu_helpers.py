"""Shared pieces of the GPU parity tests: the acceptance check, device input
creation and the calls into the library."""
from __future__ import annotations

import numpy as np
import torch

import blockwise_attention_ffn_gb300 as bpt
from blockwise_attention_ffn_gb300.synth import make_layer_inputs

# Acceptance for bf16-in / fp32-accumulate results against the fp64 oracle.
MAX_ABS = 2e-2
REL_FRO = 5e-3


def errors(got, want):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert got.shape == want.shape, (got.shape, want.shape)
    diff = got - want
    max_abs = float(np.max(np.abs(diff))) if diff.size else 0.0
    den = float(np.linalg.norm(want))
    rel = float(np.linalg.norm(diff) / den) if den > 0 else float(np.linalg.norm(diff))
    return max_abs, rel


def assert_close(got, want, what, max_abs=MAX_ABS, rel_fro=REL_FRO):
    ma, rf = errors(got, want)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    assert ma <= max_abs and rf <= rel_fro, f"{what}: max_abs={ma:.3e} rel_fro={rf:.3e}"
    return ma, rf


def assert_close_grad(got, want, what):
    """Weight gradients: fp32 results, relative Frobenius over the whole
    tensor, max abs error measured in units of the tensor's RMS when that RMS
    exceeds 1 (a gradient summed over thousands of rows has entries far
    above 1, where an absolute 2e-2 would demand more than fp32 sums of bf16
    products carry)."""
    want = np.asarray(want, np.float64)
    rms = float(np.sqrt(np.mean(want * want))) if want.size else 0.0
    return assert_close(got, want, what, max_abs=MAX_ABS * max(1.0, rms))


def to64(t):
    return t.detach().float().cpu().double().numpy()


def device_inputs(cfg, seed, with_dy=True):
    """Seeded inputs generated on the CPU (so the oracle sees exactly the same
    values) and copied to the GPU."""
    inp = make_layer_inputs(cfg, seed, device="cpu", with_dy=with_dy)
    dev = {"x": inp["x"].cuda(), "weights": {k: (None if v is None else v.cuda())
                                             for k, v in inp["weights"].items()}}
    if with_dy:
        dev["dy"] = inp["dy"].cuda()
    return inp, dev


def run_fwd(cfg, dev):
    x = dev["x"]
    y = torch.empty_like(x)
    saved = bpt.alloc_bytes(bpt.bpt_saved_bytes(cfg))
    ws = bpt.alloc_bytes(bpt.bpt_workspace_bytes(cfg, bpt.BPT_PASS_FWD))
    bpt.bpt_layer_fwd(cfg, dev["weights"], x, y, saved, ws)
    torch.cuda.synchronize()
    st, detail = bpt.bpt_last_device_error()
    assert st == bpt.BPT_OK, f"device error {st} at wait site {detail}"
    return y, saved


def run_bwd(cfg, dev, saved, dy=None):
    x = dev["x"]
    dy = dev["dy"] if dy is None else dy
    dx = torch.empty_like(x)
    grads = bpt.alloc_grads(dev["weights"])
    ws = bpt.alloc_bytes(bpt.bpt_workspace_bytes(cfg, bpt.BPT_PASS_BWD))
    bpt.bpt_layer_bwd(cfg, dev["weights"], x, saved, dy, dx, grads, ws)
    torch.cuda.synchronize()
    st, detail = bpt.bpt_last_device_error()
    assert st == bpt.BPT_OK, f"device error {st} at wait site {detail}"
    return dx, grads
