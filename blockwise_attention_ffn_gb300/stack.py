"""A stack of L layers trained with a checkpoint every k layers.

"Training memory: model states, activations and checkpointing", section 3
("Checkpoint every k layers"): the forward pass keeps the input of every k-th
layer; the backward pass takes the segments last first, re-runs each one's
forward from its checkpoint, keeping the inputs of the segment's layers, and
back-propagates through the segment layer by layer before moving on.

Each layer call of this library is already fully checkpointed inside: its
backward rebuilds everything from the layer input and the log-sum-exp the
forward saved.  So a layer's cache here is its input alone, and the stack
holds at most ceil(L/k) + k - 1 layer inputs of b*s*h bf16 at once (the
checkpoints still to be used, plus the rebuilt inputs of one segment; the
segment's first input is its checkpoint), plus one log-sum-exp per layer.
With k = 1 every layer input is a checkpoint and no forward is re-run at the
stack level; with k = L only x is kept and every layer but the last runs its
forward twice.  Both hold L inputs at the peak; k near sqrt(L) holds about
2 sqrt(L), the same trade-off as the page's M(k) = (L/k) c + k A with the
cache A of a layer equal to its checkpoint c.

This module only schedules: every step of every layer runs in the library's
kernels through bpt_layer_fwd / bpt_layer_bwd.  ``ops`` replaces those two
calls and the allocations around them (the tests drive the same schedule with
another implementation of the layer on the CPU).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field


def held_inputs(L: int, k: int) -> int:
    """The most layer inputs the backward pass holds at once: ceil(L/k)
    checkpoints while the last segment is rebuilt, plus that segment's other
    inputs; later segments hold one checkpoint fewer.  (The forward pass holds
    the checkpoints plus the running layer's input and output.)"""
    n = math.ceil(L / k)
    last = L - (n - 1) * k
    peak = n + last - 1
    if n > 1:
        peak = max(peak, n - 1 + k - 1)
    return max(peak, 1)


class LibOps:
    """The library's layer calls on the tensors' CUDA device and a stream."""

    def __init__(self, stream=None):
        self.stream = stream

    def workspace(self, cfg, like):
        from . import BPT_PASS_BWD, BPT_PASS_FWD, alloc_bytes, bpt_workspace_bytes
        return alloc_bytes(max(bpt_workspace_bytes(cfg, BPT_PASS_FWD), bpt_workspace_bytes(cfg, BPT_PASS_BWD)),
                           device=like.device)

    def saved(self, cfg, like):
        from . import alloc_bytes, bpt_saved_bytes
        return alloc_bytes(bpt_saved_bytes(cfg), device=like.device)

    def empty_like(self, t):
        import torch
        return torch.empty_like(t)

    def grads(self, W, like):
        from . import alloc_grads
        return alloc_grads(W, device=like.device)

    def layer_fwd(self, cfg, W, x, y, saved, ws):
        from . import bpt_layer_fwd
        bpt_layer_fwd(cfg, W, x, y, saved, ws, self.stream)

    def layer_bwd(self, cfg, W, x, saved, dy, dx, grads, ws):
        from . import bpt_layer_bwd
        bpt_layer_bwd(cfg, W, x, saved, dy, dx, grads, ws, self.stream)


@dataclass
class StackState:
    """What the forward pass keeps for the backward pass: the inputs of
    layers 0, k, 2k, ... and every layer's log-sum-exp.  The backward pass
    consumes it (each checkpoint is released once its segment is done)."""
    k: int
    n_layers: int
    ckpt: dict = field(default_factory=dict)
    saved: list = field(default_factory=list)
    peak_held: int = 0  # most layer inputs the backward pass held at once


def stack_fwd(cfg, weights: list, x, k: int, ws=None, ops=None):
    """y = layer_{L-1}(... layer_0(x)), keeping a checkpoint every k layers.
    weights: one weight dict per layer (the layer call's layout).  Returns
    (y, state) for stack_bwd."""
    L = len(weights)
    if not 1 <= k <= L:
        raise ValueError(f"checkpoint interval k={k} must be in [1, {L}]")
    ops = ops or LibOps()
    ws = ops.workspace(cfg, x) if ws is None else ws
    st = StackState(k=k, n_layers=L)
    h = x
    for i, W in enumerate(weights):
        if i % k == 0:
            st.ckpt[i] = h
        y = ops.empty_like(h)
        sv = ops.saved(cfg, h)
        ops.layer_fwd(cfg, W, h, y, sv, ws)
        st.saved.append(sv)
        h = y
    return h, st


def stack_bwd(cfg, weights: list, state: StackState, dy, ws=None, ops=None, grads=None):
    """Gradients of the stack given dy.  Returns (dx, grads) with one
    gradient dict per layer (fp32, overwritten, or those passed in)."""
    L = len(weights)
    if L != state.n_layers:
        raise ValueError("weights do not match the forward pass")
    ops = ops or LibOps()
    ws = ops.workspace(cfg, dy) if ws is None else ws
    grads = [ops.grads(W, dy) for W in weights] if grads is None else grads
    k = state.k
    rebuilt_saved = None  # log-sum-exp of re-run forwards (already kept in state.saved)
    g = dy
    for s0 in sorted(state.ckpt, reverse=True):
        s1 = min(L, s0 + k)
        seg_in = [state.ckpt[s0]]
        for i in range(s0, s1 - 1):
            if rebuilt_saved is None:
                rebuilt_saved = ops.saved(cfg, dy)
            y = ops.empty_like(seg_in[-1])
            ops.layer_fwd(cfg, weights[i], seg_in[-1], y, rebuilt_saved, ws)
            seg_in.append(y)
        state.peak_held = max(state.peak_held, len(state.ckpt) + len(seg_in) - 1)
        for i in range(s1 - 1, s0 - 1, -1):
            dx = ops.empty_like(g)
            ops.layer_bwd(cfg, weights[i], seg_in[i - s0], state.saved[i], g, dx, grads[i], ws)
            g = dx
        del seg_in
        del state.ckpt[s0]
    return g, grads
