"""Row-sampled forward and sparse-upstream-gradient backward (fp64).

TEST INFRASTRUCTURE ONLY.  For sequence lengths where the dense oracle would
take too long, two exact reductions of the same definition as
:mod:`oracle.ref`:

* Forward at sampled rows.  Output row i of a causal layer depends on key and
  value rows 0..i only (every other step is position-wise), so y[i] is
  computed from K and V of all rows and Q of row i alone.  This is the row
  independence the BPT page relies on ("Why fusion is now possible": the
  attention output of query block i does not depend on any other query block,
  and the FFN is position-wise).
* Backward with an upstream gradient that is nonzero on a few rows R only.
  Then dx1, dO and dQ are nonzero only on R; dK, dV need the softmax rows of R
  only; and every weight gradient and dx follow exactly from those sparse
  pieces.  Nothing is approximated: the result equals the dense analytic
  backward of :func:`oracle.ref.layer_backward` for that dy.

With ``rope_base`` set, query rows are rotated at their own positions and
key rows at theirs, as :func:`oracle.ref.rope` defines, and the gradients go
back through the transposed rotation.
"""
from __future__ import annotations

from math import sqrt

import numpy as np

from .ref import (ACT_SWIGLU, F64, LayerCfg, _as64, _lin, ffn_forward, gelu_grad, norm_backward,
                  norm_forward, rope, silu, silu_grad)


def _proj(xn, W, name, bias):
    return _lin(xn, W[name], W.get(bias))


def _attn_rows(qr, rows, k, v, causal, s_):
    """Attention of the query rows ``rows`` (one head) against k, v."""
    d = qr.shape[1]
    S = (qr @ k.T) / sqrt(d)
    if causal:
        S = np.where(np.arange(s_)[None, :] > np.asarray(rows)[:, None], -np.inf, S)
    m = S.max(1, keepdims=True)
    E = np.exp(S - m)
    P = E / E.sum(1, keepdims=True)
    return P @ v, P


def forward_rows(x, W, cfg: LayerCfg, rows, batch=0):
    """y[batch, rows] of the layer (exact)."""
    W = _as64(W)
    xb = np.asarray(x[batch], F64)
    H, Hk, d, G = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.group
    s_ = xb.shape[0]
    rows = np.asarray(rows)
    xn, _, _ = norm_forward(xb, W["ln1_w"], W.get("ln1_b"), cfg)
    k = _proj(xn, W, "wk", "bk").reshape(s_, Hk, d)
    v = _proj(xn, W, "wv", "bv").reshape(s_, Hk, d)
    q = _proj(xn[rows], W, "wq", "bq").reshape(len(rows), H, d)
    if cfg.rope_base:
        k = rope(k, cfg.rope_base)
        q = rope(q, cfg.rope_base, positions=rows)
    o = np.empty((len(rows), H, d), F64)
    for n in range(H):
        o[:, n], _ = _attn_rows(q[:, n], rows, k[:, n // G], v[:, n // G], cfg.causal, s_)
    x1 = xb[rows] + _lin(o.reshape(len(rows), H * d), W["wo"], W.get("bo"))
    x1n, _, _ = norm_forward(x1, W["ln2_w"], W.get("ln2_b"), cfg)
    f, _ = ffn_forward(x1n, W, cfg)
    return x1 + f


def backward_sparse_dy(x, W, dy_rows, rows, cfg: LayerCfg, batch=0):
    """dx (all rows) and every weight gradient for an upstream gradient that
    equals ``dy_rows`` on ``rows`` of sequence ``batch`` and zero elsewhere
    (b must be 1 or the other sequences carry zero gradient)."""
    W64 = _as64(W)
    xb = np.asarray(x[batch], F64)
    dyr = np.asarray(dy_rows, F64)
    rows = np.asarray(rows)
    assert len(np.unique(rows)) == len(rows), "sampled rows must be distinct"
    H, Hk, d, G = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.group
    s_ = xb.shape[0]
    R = len(rows)
    grads = {k_: np.zeros(np.shape(v_), F64) for k_, v_ in W64.items() if v_ is not None}

    xn, xhat1, rstd1 = norm_forward(xb, W64["ln1_w"], W64.get("ln1_b"), cfg)
    k = _proj(xn, W64, "wk", "bk").reshape(s_, Hk, d)
    v = _proj(xn, W64, "wv", "bv").reshape(s_, Hk, d)
    q = _proj(xn[rows], W64, "wq", "bq").reshape(R, H, d)
    if cfg.rope_base:
        k = rope(k, cfg.rope_base)
        q = rope(q, cfg.rope_base, positions=rows)
    o = np.empty((R, H, d), F64)
    P = [None] * H
    for n in range(H):
        o[:, n], P[n] = _attn_rows(q[:, n], rows, k[:, n // G], v[:, n // G], cfg.causal, s_)
    of = o.reshape(R, H * d)
    x1 = xb[rows] + _lin(of, W64["wo"], W64.get("bo"))
    x1n, xhat2, rstd2 = norm_forward(x1, W64["ln2_w"], W64.get("ln2_b"), cfg)

    # FFN branch on the sampled rows
    if cfg.act == ACT_SWIGLU:
        g = _lin(x1n, W64["w1"])
        u = _lin(x1n, W64["w3"])
        a = silu(g) * u
        grads["w2"] += dyr.T @ a
        da = dyr @ W64["w2"]
        dg = da * u * silu_grad(g)
        du = da * silu(g)
        grads["w1"] += dg.T @ x1n
        grads["w3"] += du.T @ x1n
        dx1n = dg @ W64["w1"] + du @ W64["w3"]
    else:
        z = _lin(x1n, W64["w1"], W64.get("b1"))
        _, fc = ffn_forward(x1n, W64, cfg)
        a = fc["a"]
        grads["w2"] += dyr.T @ a
        da = dyr @ W64["w2"]
        dz = da * gelu_grad(z, cfg.act)
        grads["w1"] += dz.T @ x1n
        dx1n = dz @ W64["w1"]
        if cfg.has_bias:
            grads["b1"] += dz.sum(0)
    if cfg.has_bias:
        grads["b2"] += dyr.sum(0)
    dx1_n, dw, db = norm_backward(dx1n, xhat2, rstd2, W64["ln2_w"], cfg)
    grads["ln2_w"] += dw
    if db is not None:
        grads["ln2_b"] += db
    dx1 = dyr + dx1_n

    grads["wo"] += dx1.T @ of
    if cfg.has_bias:
        grads["bo"] += dx1.sum(0)
    do = (dx1 @ W64["wo"]).reshape(R, H, d)

    dq = np.zeros((R, H, d), F64)
    dk = np.zeros((s_, Hk, d), F64)
    dv = np.zeros((s_, Hk, d), F64)
    for n in range(H):
        gk = n // G
        Pn = P[n]
        dP = do[:, n] @ v[:, gk].T
        dS = Pn * (dP - (Pn * dP).sum(1, keepdims=True))
        dv[:, gk] += Pn.T @ do[:, n]
        dq[:, n] = dS @ k[:, gk] / sqrt(d)
        dk[:, gk] += dS.T @ q[:, n] / sqrt(d)
    if cfg.rope_base:
        dq = rope(dq, cfg.rope_base, inverse=True, positions=rows)
        dk = rope(dk, cfg.rope_base, inverse=True)
    dqf = dq.reshape(R, H * d)
    dkf = dk.reshape(s_, Hk * d)
    dvf = dv.reshape(s_, Hk * d)
    grads["wq"] += dqf.T @ xn[rows]
    grads["wk"] += dkf.T @ xn
    grads["wv"] += dvf.T @ xn
    if cfg.has_bias:
        grads["bq"] += dqf.sum(0)
        grads["bk"] += dkf.sum(0)
        grads["bv"] += dvf.sum(0)
    dxn = dkf @ W64["wk"] + dvf @ W64["wv"]
    dxn[rows] += dqf @ W64["wq"]
    dx_n, dw, db = norm_backward(dxn, xhat1, rstd1, W64["ln1_w"], cfg)
    grads["ln1_w"] += dw
    if db is not None:
        grads["ln1_b"] += db
    dx = dx_n
    dx[rows] += dx1
    return dx, grads
