"""The layer-stack schedule (checkpoint every k layers) driven on the CPU with
the fp64 oracle standing in for the library's layer calls.  It must give
exactly the oracle's stack (same layer operations on the same values), hold
no more layer inputs than ceil(L/k) + k - 1, and release what it consumed."""
import numpy as np
import pytest
import torch

from blockwise_attention_ffn_gb300 import stack
from oracle import ref
from oracle import stack as ostack
from oracle.ref import LayerCfg
from tests.oracle_helpers import rand_layer

CFG = LayerCfg(s=9, h=16, n_heads=2, n_kv_heads=1, head_dim=8, ffn_dim=24)


class OracleOps:
    """The layer calls' contract (write y; write dx and every gradient) on
    CPU fp64 tensors, computed by the oracle."""

    def __init__(self):
        self.fwd_calls, self.bwd_calls = [], []

    def workspace(self, cfg, like):
        return None

    def saved(self, cfg, like):
        return torch.empty(0)

    def empty_like(self, t):
        return torch.empty_like(t)

    def grads(self, W, like):
        return {k: (None if v is None else torch.empty(np.shape(v), dtype=torch.float64)) for k, v in W.items()}

    def layer_fwd(self, cfg, W, x, y, saved, ws):
        self.fwd_calls.append(id(W))
        y.copy_(torch.from_numpy(ref.layer_forward(x.numpy(), W, cfg)))

    def layer_bwd(self, cfg, W, x, saved, dy, dx, grads, ws):
        self.bwd_calls.append(id(W))
        d, g = ref.layer_backward(x.numpy(), W, dy.numpy(), cfg)
        dx.copy_(torch.from_numpy(d))
        for k, v in g.items():
            grads[k].copy_(torch.from_numpy(v))


def _stack(L, seed=90):
    x, W0, dy = rand_layer(CFG, seed=seed)
    Ws = [W0] + [rand_layer(CFG, seed=seed + 1 + i)[1] for i in range(L - 1)]
    return x, Ws, dy


@pytest.mark.parametrize("L,k", [(1, 1), (3, 1), (3, 2), (3, 3), (5, 2), (6, 3), (7, 3)])
def test_schedule_equals_the_oracle_stack(L, k):
    x, Ws, dy = _stack(L)
    ops = OracleOps()
    y, st = stack.stack_fwd(CFG, Ws, torch.from_numpy(x), k, ops=ops)
    assert np.array_equal(y.numpy(), ostack.stack_forward(x, Ws, CFG))
    dx, grads = stack.stack_bwd(CFG, Ws, st, torch.from_numpy(dy), ops=ops)
    dx_ref, g_ref = ostack.stack_backward(x, Ws, dy, CFG)
    assert np.array_equal(dx.numpy(), dx_ref)
    for i in range(L):
        for name, v in g_ref[i].items():
            assert np.array_equal(grads[i][name].numpy(), v), (i, name)
    # every layer's backward ran once, last layer first; the forward re-ran
    # every layer that is not the last of its segment, once
    assert ops.bwd_calls == [id(W) for W in reversed(Ws)]
    rerun = [i for i in range(L) if i % k != k - 1 and i != L - 1]
    assert len(ops.fwd_calls) == L + len(rerun)
    # the checkpoints were consumed, and the hold matches the closed form
    assert st.ckpt == {}
    assert st.peak_held == stack.held_inputs(L, k)


@pytest.mark.parametrize("L", [1, 2, 5, 8, 80])
def test_held_inputs_closed_form(L):
    for k in range(1, L + 1):
        n = -(-L // k)
        assert stack.held_inputs(L, k) <= n + k - 1
        # equal to the page's M(k) count less the checkpoint counted twice
        # whenever k divides L (c = A: a layer's cache is its input)
        if L % k == 0:
            assert stack.held_inputs(L, k) == L // k + k - 1
    # both ends hold every input; the best k is near sqrt(L)
    assert stack.held_inputs(L, 1) == L and stack.held_inputs(L, L) == L
    best = min(range(1, L + 1), key=lambda k: stack.held_inputs(L, k))
    assert abs(best - L ** 0.5) <= 1 + L ** 0.5 / 2


def test_interval_is_checked():
    x, Ws, _ = _stack(2)
    with pytest.raises(ValueError):
        stack.stack_fwd(CFG, Ws, torch.from_numpy(x), 3, ops=OracleOps())
    with pytest.raises(ValueError):
        stack.stack_fwd(CFG, Ws, torch.from_numpy(x), 0, ops=OracleOps())
