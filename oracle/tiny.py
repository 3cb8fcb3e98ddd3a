"""Scalar-loop forward of the layer, for tiny shapes only.

TEST INFRASTRUCTURE ONLY.  A second, independent restatement of the same
definition as :mod:`oracle.ref` (pre-norm layer, softmax attention with the
causal mask and 1/sqrt(head_dim) scale, GeLU or SwiGLU FFN), written with
Python floats and explicit loops so that no array broadcasting, reshaping or
library call is shared with the NumPy version.  Sources: "Training memory:
model states, activations and checkpointing", section 3 (the layer and its
parameters); "Blockwise Parallel Transformer for Long Context Large Models",
section 3.4 (scaled dot-product attention, causal bias).  With a nonzero
``rope_base`` the query and key heads are rotated as :func:`oracle.ref.rope`
describes, pair by pair with ``math.cos`` / ``math.sin``.
"""
from __future__ import annotations

import math


def _norm_row(row, w, b, kind, eps):
    n = len(row)
    if kind == 0:
        mu = sum(row) / n
        var = sum((t - mu) * (t - mu) for t in row) / n
        r = 1.0 / math.sqrt(var + eps)
        return [(row[i] - mu) * r * w[i] + b[i] for i in range(n)]
    ms = sum(t * t for t in row) / n
    r = 1.0 / math.sqrt(ms + eps)
    return [row[i] * r * w[i] for i in range(n)]


def _matvec(W, v, bias=None):
    out = []
    for o in range(len(W)):
        acc = 0.0
        for i in range(len(v)):
            acc += W[o][i] * v[i]
        if bias is not None:
            acc += bias[o]
        out.append(acc)
    return out


def _gelu(z, act):
    if act == 0:
        return 0.5 * z * (1.0 + math.erf(z / math.sqrt(2.0)))
    c = math.sqrt(2.0 / math.pi)
    return 0.5 * z * (1.0 + math.tanh(c * (z + 0.044715 * z ** 3)))


def _silu(z):
    return z / (1.0 + math.exp(-z))


def _rope_row(row, pos, nheads, d, base):
    """Rotate element i of every head with element i + d/2 by pos * base^(-2i/d)."""
    out = list(row)
    half = d // 2
    for n in range(nheads):
        for i in range(half):
            ang = pos * math.pow(base, -2.0 * i / d)
            a, b = row[n * d + i], row[n * d + half + i]
            out[n * d + i] = a * math.cos(ang) - b * math.sin(ang)
            out[n * d + half + i] = a * math.sin(ang) + b * math.cos(ang)
    return out


def layer_forward(x, W, cfg):
    """x: nested list [b][s][h]; W: dict of nested lists (nn.Linear [out][in]);
    cfg: object with the oracle.ref.LayerCfg fields.  Returns nested list y."""
    H, Hk, d = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim
    G = H // Hk
    out = []
    for xb in x:
        s = len(xb)
        xn = [_norm_row(xb[t], W["ln1_w"], W.get("ln1_b"), cfg.norm, cfg.norm_eps) for t in range(s)]
        q = [_matvec(W["wq"], xn[t], W.get("bq")) for t in range(s)]
        k = [_matvec(W["wk"], xn[t], W.get("bk")) for t in range(s)]
        v = [_matvec(W["wv"], xn[t], W.get("bv")) for t in range(s)]
        base = getattr(cfg, "rope_base", 0.0)
        if base:
            q = [_rope_row(q[t], t, H, d, base) for t in range(s)]
            k = [_rope_row(k[t], t, Hk, d, base) for t in range(s)]
        yb = []
        for i in range(s):
            o = [0.0] * (H * d)
            for n in range(H):
                g = n // G
                keys = range(i + 1) if cfg.causal else range(s)
                sc = []
                for j in keys:
                    dot = 0.0
                    for c in range(d):
                        dot += q[i][n * d + c] * k[j][g * d + c]
                    sc.append(dot / math.sqrt(d))
                m = max(sc)
                e = [math.exp(t - m) for t in sc]
                tot = sum(e)
                for idx, j in enumerate(keys):
                    p = e[idx] / tot
                    for c in range(d):
                        o[n * d + c] += p * v[j][g * d + c]
            proj = _matvec(W["wo"], o, W.get("bo"))
            x1 = [xb[i][c] + proj[c] for c in range(len(proj))]
            x1n = _norm_row(x1, W["ln2_w"], W.get("ln2_b"), cfg.norm, cfg.norm_eps)
            if cfg.act == 2:
                gt = _matvec(W["w1"], x1n)
                up = _matvec(W["w3"], x1n)
                a = [_silu(gt[c]) * up[c] for c in range(len(gt))]
            else:
                z = _matvec(W["w1"], x1n, W.get("b1"))
                a = [_gelu(t, cfg.act) for t in z]
            f = _matvec(W["w2"], a, W.get("b2"))
            yb.append([x1[c] + f[c] for c in range(len(f))])
        out.append(yb)
    return out
