"""The layer's forward and backward with exactly the bf16 roundings the
kernels make, everything else in fp64: the error floor of a bf16-storage,
fp32-accumulation implementation of this schedule, against which the GPU
parity tests' per-tensor bounds are derived.

Test infrastructure: built from the oracle's fp64 primitives plus one
rounding helper; it shares nothing with the CUDA path.  The rounding points,
in the order the kernels meet them:

forward   xn = bf(N1(x)); q, k, v = bf(xn W^T + b) (rotary embedding: rotated
          and rounded again); per head P~ = bf(exp(S - rowmax)), l = sum P~
          (fp32 sum of the rounded values; of the unrounded ones at d = 128),
          O = bf(P~ V / l), LSE = rowmax + ln l; x1 = x + O Wo^T + bo (fp32);
          x1n = bf(N2(x1)); GeLU: a = bf(gelu(z)), gelu'(z) kept as bf16;
          SwiGLU: g, u kept as bf16, a = bf(silu(g) u) from the fp32 sums;
          y = bf(x1 + a W2^T + b2)
backward  dz = bf(dA gelu'(z)) (SwiGLU: bf(dA u silu'(g)), bf(dA silu(g)) from
          the bf16 g, u); dx1n = bf(dz W1); dx1 = dy + N2^T(dx1n), kept fp32
          and as bf(.); dO = bf(dx1 Wo); per head P = exp(S - LSE),
          dS = bf(P (dO V^T - D)) with D = rowsum(dO O), dV = sum bf(P)^T dO,
          dK = sum dS^T q / sqrt(d), dQ = dS k / sqrt(d), each rounded once;
          rotary embedding turned back and rounded; dxn = dQKV Wqkv (fp32);
          dx = bf(dx1 + N1^T(dxn)); weight gradients fp32 from the bf16
          operands; bias gradients fp32 column sums of the bf16 gradients.
"""
from __future__ import annotations

from math import sqrt

import numpy as np
import torch

from oracle import ref


def bf(a):
    """Round to the nearest bf16 (ties to even), back in fp64."""
    return torch.from_numpy(np.ascontiguousarray(a, np.float64)).to(torch.bfloat16).double().numpy()


def _lin(a, W, w, b=None):
    return a @ W[w].T + (W[b] if (b is not None and W.get(b) is not None) else 0.0)


def layer_grads_bf16(x, W, dy, cfg: ref.LayerCfg):
    """(y, dx, grads) of one sequence (x, dy: [s, h]) through the bf16-operand
    pipeline described in the module docstring."""
    s, H, Hk, d, G = x.shape[0], cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.group
    sc = 1.0 / sqrt(d)
    hb = cfg.has_bias
    # ---------------- forward
    xn_f, xhat1, rstd1 = ref.norm_forward(x, W["ln1_w"], W.get("ln1_b"), cfg)
    xn = bf(xn_f)
    q = bf(_lin(xn, W, "wq", "bq")).reshape(s, H, d)
    k = bf(_lin(xn, W, "wk", "bk")).reshape(s, Hk, d)
    v = bf(_lin(xn, W, "wv", "bv")).reshape(s, Hk, d)
    if cfg.rope_base:
        q = bf(ref.rope(q, cfg.rope_base))
        k = bf(ref.rope(k, cfg.rope_base))
    mask = np.arange(s)[None, :] > np.arange(s)[:, None] if cfg.causal else np.zeros((s, s), bool)
    O = np.empty((s, H, d))
    lse = np.empty((H, s))
    for n in range(H):
        S = np.where(mask, -np.inf, q[:, n] @ k[:, n // G].T * sc)
        m = S.max(1, keepdims=True)
        E = np.exp(S - m)
        Pt = bf(E)
        l_ = (E if d == 128 else Pt).sum(1, keepdims=True)
        O[:, n] = bf(Pt @ v[:, n // G] / l_)
        lse[n] = (m + np.log(l_))[:, 0]
    Of = O.reshape(s, H * d)
    x1 = x + _lin(Of, W, "wo", "bo")
    x1n_f, xhat2, rstd2 = ref.norm_forward(x1, W["ln2_w"], W.get("ln2_b"), cfg)
    x1n = bf(x1n_f)
    if cfg.act == ref.ACT_SWIGLU:
        g_f, u_f = x1n @ W["w1"].T, x1n @ W["w3"].T
        a = bf(ref.silu(g_f) * u_f)
        g_b, u_b = bf(g_f), bf(u_f)
    else:
        z = _lin(x1n, W, "w1", "b1")
        a = bf(ref.gelu(z, cfg.act))
        gd = bf(ref.gelu_grad(z, cfg.act))
    y = bf(x1 + _lin(a, W, "w2", "b2"))
    # ---------------- backward
    gr = {}
    gr["w2"] = dy.T @ a
    if hb:
        gr["b2"] = dy.sum(0)
    dA = dy @ W["w2"]
    if cfg.act == ref.ACT_SWIGLU:
        dg = bf(dA * u_b * ref.silu_grad(g_b))
        du = bf(dA * ref.silu(g_b))
        gr["w1"] = dg.T @ x1n
        gr["w3"] = du.T @ x1n
        dx1n = bf(dg @ W["w1"] + du @ W["w3"])
    else:
        dz = bf(dA * gd)
        gr["w1"] = dz.T @ x1n
        if hb:
            gr["b1"] = dz.sum(0)
        dx1n = bf(dz @ W["w1"])
    dx1_n, gr["ln2_w"], db2 = ref.norm_backward(dx1n, xhat2, rstd2, W["ln2_w"], cfg)
    if db2 is not None:
        gr["ln2_b"] = db2
    dx1f = dy + dx1_n
    dx1 = bf(dx1f)
    gr["wo"] = dx1.T @ Of
    if hb:
        gr["bo"] = dx1.sum(0)
    do = bf(dx1 @ W["wo"]).reshape(s, H, d)
    dq = np.empty((s, H, d))
    dk = np.zeros((s, Hk, d))
    dv = np.zeros((s, Hk, d))
    for n in range(H):
        gk = n // G
        S = np.where(mask, -np.inf, q[:, n] @ k[:, gk].T * sc)
        P = np.exp(S - lse[n][:, None])
        D = (do[:, n] * O[:, n]).sum(1, keepdims=True)
        dS = bf(P * (do[:, n] @ v[:, gk].T - D))
        dv[:, gk] += bf(P).T @ do[:, n]
        dk[:, gk] += dS.T @ q[:, n] * sc
        dq[:, n] = dS @ k[:, gk] * sc
    dq, dk, dv = bf(dq), bf(dk), bf(dv)
    if cfg.rope_base:
        dq = bf(ref.rope(dq, cfg.rope_base, inverse=True))
        dk = bf(ref.rope(dk, cfg.rope_base, inverse=True))
    dq, dk, dv = dq.reshape(s, -1), dk.reshape(s, -1), dv.reshape(s, -1)
    gr["wq"], gr["wk"], gr["wv"] = dq.T @ xn, dk.T @ xn, dv.T @ xn
    if hb:
        gr["bq"], gr["bv"] = dq.sum(0), dv.sum(0)
        # the key bias cancels in the softmax without a rotation after it
        gr["bk"] = dk.sum(0) if cfg.rope_base else np.zeros(Hk * d)
    dxn = dq @ W["wq"] + dk @ W["wk"] + dv @ W["wv"]
    dx_n, gr["ln1_w"], db1 = ref.norm_backward(dxn, xhat1, rstd1, W["ln1_w"], cfg)
    if db1 is not None:
        gr["ln1_b"] = db1
    dx = bf(dx1f + dx_n)
    return y, dx, gr


def floor_errors(cfg, seed=3, sparse_rows=None):
    """Per tensor (y, dx and every weight gradient): (relative Frobenius
    error, max-abs error in units of the tensor's largest entry or 1) of the
    bf16-operand pipeline against the exact fp64 oracle, on the seeded
    inputs of ``cfg`` (batch 1).  sparse_rows: the upstream gradient is kept
    on those rows only (the full-size parity tests' sparse-gradient run)."""
    from blockwise_attention_ffn_gb300.synth import make_layer_inputs
    from tests.oracle_helpers import inputs_to_oracle, oracle_cfg
    inp = make_layer_inputs(cfg, seed=seed, device="cpu")
    o = inputs_to_oracle(inp)
    oc = oracle_cfg(cfg)
    W = {k: np.asarray(v, np.float64) for k, v in o["W"].items()}
    x, dy = o["x"][0], o["dy"][0].copy()
    if sparse_rows is not None:
        keep = np.zeros(x.shape[0], bool)
        keep[sparse_rows] = True
        dy[~keep] = 0.0
    y_e, dx_e, g_e = layer_grads_bf16(x, W, dy, oc)
    y_r = ref.layer_forward(x[None], W, oc)[0]
    dx_r, g_r = ref.layer_backward(x[None], W, dy[None], oc)
    out = {}

    def err(got, want):
        den = np.linalg.norm(want)
        rel = np.linalg.norm(got - want) / den if den > 0 else np.linalg.norm(got - want)
        return float(rel), float(np.max(np.abs(got - want)) / max(1.0, np.max(np.abs(want))))
    out["y"] = err(y_e, y_r)
    out["dx"] = err(dx_e, dx_r[0])
    for k, v in g_r.items():
        out[k] = err(g_e[k], v)
    return out
