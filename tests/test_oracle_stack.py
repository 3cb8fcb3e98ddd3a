"""Pins of the layer-stack oracle with checkpoints every k layers (the
multi-layer row that comes next).  A checkpointed backward that dropped or
reordered a segment, or used a stale input, would not equal the plain chain
rule; one that kept every input would exceed the page's M(k)."""
import json
import os

import numpy as np
import pytest

from oracle import accounting, stack
from oracle.ref import LayerCfg
from tests.oracle_helpers import rand_layer

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_numbers.json")))
CFG = LayerCfg(s=9, h=16, n_heads=2, n_kv_heads=1, head_dim=8, ffn_dim=24)


def _stack(L, seed=40):
    x, W0, dy = rand_layer(CFG, seed=seed)
    Ws = [W0] + [rand_layer(CFG, seed=seed + 1 + i)[1] for i in range(L - 1)]
    return x, Ws, dy


@pytest.mark.parametrize("L,k", [(1, 1), (4, 1), (4, 2), (5, 2), (6, 3), (5, 5)])
def test_checkpointed_backward_equals_chain_rule(L, k):
    x, Ws, dy = _stack(L)
    dx0, g0 = stack.stack_backward(x, Ws, dy, CFG)
    dx1, g1, _ = stack.stack_backward_checkpointed(x, Ws, dy, CFG, k)
    assert np.array_equal(dx0, dx1)
    for a, b in zip(g0, g1):
        for name in a:
            assert np.array_equal(a[name], b[name]), name


def test_stack_gradient_matches_finite_differences():
    x, Ws, dy = _stack(2, seed=50)
    dx, grads = stack.stack_backward(x, Ws, dy, CFG)

    def loss(xx, WW):
        return float(np.sum(stack.stack_forward(xx, WW, CFG) * dy))

    eps = 1e-5
    fdx = np.zeros_like(x)
    for idx in np.ndindex(x.shape):
        xp = x.copy(); xp[idx] += eps
        xm = x.copy(); xm[idx] -= eps
        fdx[idx] = (loss(xp, Ws) - loss(xm, Ws)) / (2 * eps)
    assert np.linalg.norm(fdx - dx) <= 1e-6 * np.linalg.norm(dx)
    # the first layer's query weights: the path through both layers
    w = Ws[0]["wq"]
    fd = np.zeros_like(w)
    for idx in np.ndindex(w.shape):
        Wp = [dict(Ws[0]), Ws[1]]; Wp[0]["wq"] = w.copy(); Wp[0]["wq"][idx] += eps
        Wm = [dict(Ws[0]), Ws[1]]; Wm[0]["wq"] = w.copy(); Wm[0]["wq"][idx] -= eps
        fd[idx] = (loss(x, Wp) - loss(x, Wm)) / (2 * eps)
    assert np.linalg.norm(fd - grads[0]["wq"]) <= 1e-6 * np.linalg.norm(grads[0]["wq"])


@pytest.mark.parametrize("L,k", [(8, 1), (8, 2), (8, 4), (9, 3), (6, 6)])
def test_schedule_holds_the_pages_m_of_k(L, k):
    """The schedule's largest hold, in checkpoints of c and layer caches of
    A, is the page's M(k) = (L/k) c + k A."""
    x, Ws, dy = _stack(L, seed=60)
    _, _, held = stack.stack_backward_checkpointed(x, Ws, dy, CFG, k)
    g = GOLD["checkpoint_every_k"]
    c, A = g["c_sbh"], g["A_sbh"]
    assert stack.peak_units(held, c, A) == accounting.checkpoint_every_k(L, k, c, A)
