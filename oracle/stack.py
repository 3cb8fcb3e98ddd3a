"""fp64 oracle of a stack of layers trained with checkpoints every k layers.

TEST INFRASTRUCTURE ONLY, like the rest of :mod:`oracle`.

"Training memory: model states, activations and checkpointing", section 3
("Checkpoint every k layers"): the forward pass keeps only the input of every
k-th layer; the backward pass re-runs the forward of one segment of k layers
from its checkpoint, keeping that segment's activations, and back-propagates
through it before moving to the previous segment.  Peak activation memory is
then about (L/k) c + k A, with c the bytes of one checkpoint and A the
activation bytes of one layer.  The same page's full checkpointing (k = 1
with the layer input only) is what one call of the library's recompute
backward does for one layer.

The stack applies :func:`oracle.ref.layer_forward` L times with each layer's
own weights.  The checkpointed backward must equal the plain chain rule
exactly: it repeats the same operations on the same values.  It also counts
what it holds (checkpoints and live per-layer caches), so that the schedule
can be pinned against the page's M(k).
"""
from __future__ import annotations

import numpy as np

from .ref import LayerCfg, layer_backward, layer_forward


def stack_forward(x, Ws, cfg: LayerCfg):
    """y = layer_{L-1}( ... layer_0(x)): Ws is one weight dict per layer."""
    h = np.asarray(x, np.float64)
    for W in Ws:
        h = layer_forward(h, W, cfg)
    return h


def stack_backward(x, Ws, dy, cfg: LayerCfg):
    """Plain chain rule, every layer input kept.  Returns (dx, [grads per
    layer])."""
    inputs = [np.asarray(x, np.float64)]
    for W in Ws[:-1]:
        inputs.append(layer_forward(inputs[-1], W, cfg))
    g = np.asarray(dy, np.float64)
    grads = [None] * len(Ws)
    for i in range(len(Ws) - 1, -1, -1):
        g, grads[i] = layer_backward(inputs[i], Ws[i], g, cfg)
    return g, grads


def stack_backward_checkpointed(x, Ws, dy, cfg: LayerCfg, k: int):
    """Checkpoints every k layers; per segment (last first) re-run its
    forward from the checkpoint keeping each layer's cache, then back through
    it.  Returns (dx, grads, held): held lists (checkpoints, live layer
    caches) at every point where the schedule holds the most, one entry per
    segment; :func:`peak_units` turns it into M = max(n_ckpt c + n_cache A)."""
    L = len(Ws)
    assert 1 <= k <= L
    # forward: keep the input of layers 0, k, 2k, ...
    ckpt = {}
    h = np.asarray(x, np.float64)
    for i, W in enumerate(Ws):
        if i % k == 0:
            ckpt[i] = h
        h = layer_forward(h, W, cfg)
    held = []
    g = np.asarray(dy, np.float64)
    grads = [None] * L
    for s0 in sorted(ckpt, reverse=True):
        s1 = min(L, s0 + k)
        # re-run the segment's forward, keeping every layer's input (its
        # cache: the layer's backward rebuilds the rest from it)
        seg_in = [ckpt[s0]]
        for i in range(s0, s1 - 1):
            seg_in.append(layer_forward(seg_in[-1], Ws[i], cfg))
        held.append((len(ckpt), len(seg_in)))
        for i in range(s1 - 1, s0 - 1, -1):
            g, grads[i] = layer_backward(seg_in[i - s0], Ws[i], g, cfg)
        del ckpt[s0]
    return g, grads, held


def peak_units(held, c, A):
    """Largest n_ckpt * c + n_cache * A over the schedule's snapshots."""
    return max(n * c + m * A for n, m in held)
