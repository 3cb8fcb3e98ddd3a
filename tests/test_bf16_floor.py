"""The error floor of a bf16-in / fp32-accumulate layer, emulated on the CPU.

Any tensor-core implementation of the layer must round to bf16 the operands of
its products: the normalised input xn of the Q/K/V projection, Q, K and V
themselves, the attention output O, the gradients dx1, dO, dS and dQ/dK/dV,
and P.  This test emulates exactly those roundings around the exact fp64
layer, plus one the kernels here add (dS is formed from the bf16 copy of P
that also feeds dV), and measures the relative Frobenius error of the
attention-projection weight gradients against the fp64 oracle.

It shows two things the GPU parity tests rely on:
* the floor for dWq / dWk at the GPT-3B and Llama-8B layer shapes is above the
  5e-3 relative Frobenius bound, so no bf16-in implementation can meet that
  bound for the gradients upstream of the attention; and
* it stays below ATTN_GRAD_REL_FRO (1.2e-2), the derived bound the GPU tests
  apply to exactly those tensors (dWq, dbq, dWk, dbk, dWv, dbv, dWo, dbo and
  the N1 scale/shift), with a margin of at least 1.5x.
"""
from math import sqrt

import numpy as np
import pytest
import torch

from blockwise_attention_ffn_gb300.presets import PRESETS
from blockwise_attention_ffn_gb300.synth import make_layer_inputs
from oracle import ref
from tests.gpu_helpers import ATTN_GRAD_REL_FRO, REL_FRO
from tests.oracle_helpers import inputs_to_oracle, oracle_cfg


def _bf(a):
    return torch.tensor(a).to(torch.bfloat16).double().numpy()


def emulated_attention_grads(cfg, seed=3):
    """dWq, dWk, dWv of the bf16-operand pipeline and of the exact oracle."""
    inp = make_layer_inputs(cfg, seed=seed, device="cpu")
    o = inputs_to_oracle(inp)
    W, x, dy = o["W"], o["x"][0], o["dy"][0]
    oc = oracle_cfg(cfg)
    _, g_ref = ref.layer_backward(o["x"], W, o["dy"], oc)
    s, H, Hk, d = cfg.s, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim
    G = H // Hk

    def lin(a, w, b=None):
        return a @ W[w].T + (W[b] if (b and b in W) else 0.0)

    xn, _, _ = ref.norm_forward(x, W["ln1_w"], W.get("ln1_b"), oc)
    xn = _bf(xn)
    q = _bf(lin(xn, "wq", "bq")).reshape(s, H, d)
    k = _bf(lin(xn, "wk", "bk")).reshape(s, Hk, d)
    v = _bf(lin(xn, "wv", "bv")).reshape(s, Hk, d)
    O = np.zeros((s, H, d))
    P = {}
    for n in range(H):
        S = q[:, n] @ k[:, n // G].T / sqrt(d)
        S = np.where(np.arange(s)[None, :] > np.arange(s)[:, None], -np.inf, S)
        E = np.exp(S - S.max(1, keepdims=True))
        P[n] = E / E.sum(1, keepdims=True)
        O[:, n] = P[n] @ v[:, n // G]
    Of = _bf(O.reshape(s, H * d))
    x1 = x + lin(Of, "wo", "bo")
    x1n, xhat2, rstd2 = ref.norm_forward(x1, W["ln2_w"], W.get("ln2_b"), oc)
    if cfg.act == 2:
        g_, u_ = x1n @ W["w1"].T, x1n @ W["w3"].T
        da = dy @ W["w2"]
        dx1n = (da * u_ * ref.silu_grad(g_)) @ W["w1"] + (da * ref.silu(g_)) @ W["w3"]
    else:
        z = lin(x1n, "w1", "b1")
        dx1n = ((dy @ W["w2"]) * ref.gelu_grad(z, cfg.act)) @ W["w1"]
    dx1_n, _, _ = ref.norm_backward(dx1n, xhat2, rstd2, W["ln2_w"], oc)
    dx1 = _bf(dy + dx1_n)
    do = _bf(dx1 @ W["wo"]).reshape(s, H, d)
    dq, dk, dv = np.zeros((s, H, d)), np.zeros((s, Hk, d)), np.zeros((s, Hk, d))
    for n in range(H):
        gk = n // G
        Dn = (do[:, n] * O[:, n]).sum(1, keepdims=True)
        dS = _bf(_bf(P[n]) * (do[:, n] @ v[:, gk].T - Dn))
        dv[:, gk] += _bf(P[n]).T @ do[:, n]
        dq[:, n] = dS @ k[:, gk] / sqrt(d)
        dk[:, gk] += dS.T @ q[:, n] / sqrt(d)
    got = {"wq": _bf(dq.reshape(s, -1)).T @ xn, "wk": _bf(dk.reshape(s, -1)).T @ xn,
           "wv": _bf(dv.reshape(s, -1)).T @ xn}
    return got, g_ref


@pytest.mark.slow
@pytest.mark.parametrize("name,s", [("c3", 384), ("c5", 256)])
def test_bf16_operand_floor_sets_the_attention_gradient_bound(name, s):
    cfg = PRESETS[name].with_(s=s)
    got, want = emulated_attention_grads(cfg)
    rel = {k: np.linalg.norm(got[k] - want[k]) / np.linalg.norm(want[k]) for k in got}
    # the floor exceeds the generic bound for the query/key projections ...
    assert rel["wq"] > REL_FRO and rel["wk"] > REL_FRO, rel
    # ... and the derived bound leaves a 1.5x margin above it
    assert max(rel.values()) * 1.5 <= ATTN_GRAD_REL_FRO, rel
