"""fp64 NumPy oracle: the pre-norm transformer layer, materialised, forward and backward.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Plain, slow and meant to
be checked by eye against the pages:

* Layer structure (pre-LN GPT layer: LN1 -> QKV -> attention -> output
  projection -> +residual; LN2 -> fc1 -> GeLU -> fc2 -> +residual, every linear
  with a bias): "Training memory: model states, activations and checkpointing",
  section 3, "Activations" (the pre-LN layer of Korthikanti et al.) and
  "Parameters: 12h^2 + 13h per layer"; the same page's section 5 code uses
  ``nn.LayerNorm`` (eps 1e-5) and the erf form of ``F.gelu``.
* Llama-style variant (RMSNorm, SwiGLU with three matrices, no biases, grouped
  query attention): same page, "Parameters" (Llama-style paragraph) and
  "Untied Ulysses", section 4.1 "The GQA Scheduling Algorithm" (query head i
  uses key/value head floor(i/G)).
* Attention: softmax(Q K^T / sqrt(d) + M) V with d the head dimension and
  M_ij = -inf where key j > query i (causal): "Blockwise Parallel Transformer
  for Long Context Large Models", section 3.4, "Blockwise Self-Attention with
  Online Softmax" (scaled dot-product attention) and "The Nested-Loop Algorithm
  in Detail (Algorithm 1)" (the causal bias is -inf where the key index exceeds
  the query index).
* Backward rules (linear keeps its input, GeLU keeps its input, softmax
  gradient p * (pbar - <p, pbar>), LayerNorm needs the normalised input):
  "Training memory ...", section 2, "The rule: every operation keeps what its
  backward pass needs".
* The blockwise variant (:func:`blockwise_attention`, :func:`bpt_layer_forward`)
  follows Algorithm 1 and the carry state of Figure 3 as the BPT page describes
  them (numerator, denominator, running max, correction factor
  exp(prev_max - new_max), final numerator / denominator, then the FFN with its
  residual applied to the finished query block).  It exists only so that the
  tests can pin the materialised definition against the method's claim that
  the blockwise schedule computes the same function.

Everything is float64.  Inputs are the bf16 values the GPU receives, upcast
exactly.  Nothing here emulates bf16 rounding.

Readings of points the pages leave open (each is listed with its reason in the
design notes): GeLU defaults to the erf form (act=0) with the tanh form as
act=1 and SwiGLU as act=2; the score scale is 1/sqrt(head_dim); the causal mask
keeps the diagonal; RMSNorm eps defaults to 1e-5 like LayerNorm; variance is
the biased 1/h form; no dropout (p = 0); no positional encoding unless
``rope_base`` is set.

Rotary position embedding (``rope_base`` > 0, off by default): "Untied
Ulysses: Memory-Efficient Context Parallelism via Headwise Chunking" lists
fused RoPE among the per-layer kernels of its Llama runs and notes the fp32
cast it needs, without giving the rotation.  Reading: the standard rotary
embedding in the half-split layout Llama checkpoints use -- element i of a
query or key head is paired with element i + d/2, and the pair at sequence
position p is rotated by the angle p * base^(-2i/d) -- applied to Q and K
after their projection (and bias), before the scores.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from math import sqrt

import numpy as np
from scipy.special import erf as _erf

F64 = np.float64

NORM_LAYER = 0
NORM_RMS = 1
ACT_GELU_ERF = 0
ACT_GELU_TANH = 1
ACT_SWIGLU = 2


@dataclass(frozen=True)
class LayerCfg:
    """Shape and variant of one layer (mirrors the fields the library takes)."""

    s: int
    h: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn_dim: int
    b: int = 1
    causal: bool = True
    norm: int = NORM_LAYER
    act: int = ACT_GELU_ERF
    has_bias: bool = True
    norm_eps: float = 1e-5
    rope_base: float = 0.0  # 0: no positional encoding

    @property
    def group(self) -> int:
        assert self.n_heads % self.n_kv_heads == 0
        return self.n_heads // self.n_kv_heads


def weight_shapes(cfg: LayerCfg) -> dict:
    """nn.Linear convention [out, in] for every matrix; None = absent."""
    h, H, Hk, d, f = cfg.h, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.ffn_dim
    shp = {
        "ln1_w": (h,), "wq": (H * d, h), "wk": (Hk * d, h), "wv": (Hk * d, h),
        "wo": (h, H * d), "ln2_w": (h,), "w1": (f, h), "w2": (h, f),
    }
    if cfg.norm == NORM_LAYER:
        shp["ln1_b"] = (h,)
        shp["ln2_b"] = (h,)
    if cfg.has_bias:
        shp.update({"bq": (H * d,), "bk": (Hk * d,), "bv": (Hk * d,), "bo": (h,),
                    "b1": (f,), "b2": (h,)})
    if cfg.act == ACT_SWIGLU:
        shp["w3"] = (f, h)
    return shp


# ----------------------------------------------------------------------------
# elementwise pieces
# ----------------------------------------------------------------------------

def gelu(z, act):
    if act == ACT_GELU_ERF:
        return 0.5 * z * (1.0 + _erf(z / sqrt(2.0)))
    c = sqrt(2.0 / np.pi)
    return 0.5 * z * (1.0 + np.tanh(c * (z + 0.044715 * z ** 3)))


def gelu_grad(z, act):
    if act == ACT_GELU_ERF:
        phi = np.exp(-0.5 * z * z) / sqrt(2.0 * np.pi)
        return 0.5 * (1.0 + _erf(z / sqrt(2.0))) + z * phi
    c = sqrt(2.0 / np.pi)
    t = np.tanh(c * (z + 0.044715 * z ** 3))
    return 0.5 * (1.0 + t) + 0.5 * z * (1.0 - t * t) * c * (1.0 + 3 * 0.044715 * z * z)


def sigmoid(z):
    return 1.0 / (1.0 + np.exp(-z))


def silu(z):
    return z * sigmoid(z)


def silu_grad(z):
    sg = sigmoid(z)
    return sg * (1.0 + z * (1.0 - sg))


def norm_forward(x, w, b, cfg: LayerCfg):
    """Row-wise LayerNorm (biased variance) or RMSNorm over the last axis.

    Returns (y, xhat, rstd) where y = xhat * w (+ b)."""
    if cfg.norm == NORM_LAYER:
        mu = x.mean(-1, keepdims=True)
        var = ((x - mu) ** 2).mean(-1, keepdims=True)
        rstd = 1.0 / np.sqrt(var + cfg.norm_eps)
        xhat = (x - mu) * rstd
        return xhat * w + b, xhat, rstd
    ms = (x * x).mean(-1, keepdims=True)
    rstd = 1.0 / np.sqrt(ms + cfg.norm_eps)
    xhat = x * rstd
    return xhat * w, xhat, rstd


def norm_backward(dy, xhat, rstd, w, cfg: LayerCfg):
    """Gradient of norm_forward w.r.t. its input, scale and shift."""
    red = tuple(range(dy.ndim - 1))
    dw = (dy * xhat).sum(red)
    db = dy.sum(red) if cfg.norm == NORM_LAYER else None
    g = dy * w
    if cfg.norm == NORM_LAYER:
        dx = rstd * (g - g.mean(-1, keepdims=True) - xhat * (g * xhat).mean(-1, keepdims=True))
    else:
        dx = rstd * (g - xhat * (g * xhat).mean(-1, keepdims=True))
    return dx, dw, db


# ----------------------------------------------------------------------------
# rotary position embedding
# ----------------------------------------------------------------------------

def rope_freqs(d, base):
    """Angular frequency of pair i (elements i and i + d/2): base^(-2i/d)."""
    return base ** (-2.0 * np.arange(d // 2, dtype=F64) / d)


def rope(x, base, inverse=False, positions=None):
    """Rotate every (i, i + d/2) pair of x [s, n, d] by the angle
    p * base^(-2i/d), p the row's position (row index, or ``positions``);
    inverse=True rotates by the negated angle, which is the transpose of the
    rotation and so also its gradient."""
    s_, _, d = x.shape
    p = np.arange(s_, dtype=F64) if positions is None else np.asarray(positions, F64)
    ang = p[:, None] * rope_freqs(d, base)[None, :]
    c = np.cos(ang)[:, None, :]
    sn = np.sin(ang)[:, None, :]
    if inverse:
        sn = -sn
    a, b = x[..., : d // 2], x[..., d // 2:]
    return np.concatenate([a * c - b * sn, a * sn + b * c], axis=-1)


# ----------------------------------------------------------------------------
# attention, materialised per head (rows processed in chunks so that an s x s
# matrix for the whole sequence is never held at once; every chunk is the full
# textbook softmax over its rows)
# ----------------------------------------------------------------------------

_ROW_CHUNK = 2048


def _scores(q_rows, k, r0, causal, scale):
    S = (q_rows @ k.T) * scale
    if causal:
        i = np.arange(r0, r0 + q_rows.shape[0])[:, None]
        j = np.arange(k.shape[0])[None, :]
        S = np.where(j > i, -np.inf, S)
    return S


def attention_head(q, k, v, causal=True):
    """softmax(q k^T / sqrt(d) + M) v for one head; also the natural-log
    log-sum-exp of every row of the scaled, masked scores."""
    s_, d = q.shape
    scale = 1.0 / sqrt(d)
    o = np.empty((s_, v.shape[1]), F64)
    lse = np.empty(s_, F64)
    for r0 in range(0, s_, _ROW_CHUNK):
        r1 = min(s_, r0 + _ROW_CHUNK)
        S = _scores(q[r0:r1], k, r0, causal, scale)
        m = S.max(1, keepdims=True)
        E = np.exp(S - m)
        l = E.sum(1, keepdims=True)
        o[r0:r1] = (E / l) @ v
        lse[r0:r1] = (m + np.log(l))[:, 0]
    return o, lse


def attention_head_backward(q, k, v, do, causal=True):
    """Gradients of attention_head w.r.t. q, k, v given the upstream do.

    Softmax rule: dS = P * (dP - rowsum(P * dP)) with dP = do v^T."""
    s_, d = q.shape
    scale = 1.0 / sqrt(d)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for r0 in range(0, s_, _ROW_CHUNK):
        r1 = min(s_, r0 + _ROW_CHUNK)
        S = _scores(q[r0:r1], k, r0, causal, scale)
        m = S.max(1, keepdims=True)
        E = np.exp(S - m)
        P = E / E.sum(1, keepdims=True)
        dP = do[r0:r1] @ v.T
        dS = P * (dP - (P * dP).sum(1, keepdims=True))
        dv += P.T @ do[r0:r1]
        dq[r0:r1] = (dS @ k) * scale
        dk += (dS.T @ q[r0:r1]) * scale
    return dq, dk, dv


# ----------------------------------------------------------------------------
# the layer
# ----------------------------------------------------------------------------

def _lin(x, w, b=None):
    y = x @ w.T
    return y if b is None else y + b


def _split_heads(t, n, d):
    return t.reshape(t.shape[0], n, d)


def _as64(W):
    return {k: (None if v is None else np.asarray(v, F64)) for k, v in W.items()}


def attention_block(xn, W, cfg: LayerCfg):
    """Q, K, V projections and attention for one sequence xn [s, h].
    Returns (o [s, H*d], lse [H, s], q, k, v)."""
    H, Hk, d, G = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.group
    q = _split_heads(_lin(xn, W["wq"], W.get("bq")), H, d)
    k = _split_heads(_lin(xn, W["wk"], W.get("bk")), Hk, d)
    v = _split_heads(_lin(xn, W["wv"], W.get("bv")), Hk, d)
    if cfg.rope_base:
        q = rope(q, cfg.rope_base)
        k = rope(k, cfg.rope_base)
    o = np.empty_like(q)
    lse = np.empty((H, xn.shape[0]), F64)
    for n in range(H):
        g = n // G
        o[:, n, :], lse[n] = attention_head(q[:, n, :], k[:, g, :], v[:, g, :], cfg.causal)
    return o.reshape(xn.shape[0], H * d), lse, q, k, v


def ffn_forward(x1n, W, cfg: LayerCfg):
    """FFN(x1n): GeLU MLP with biases, or SwiGLU (w1 gate, w3 up, w2 down)."""
    if cfg.act == ACT_SWIGLU:
        g = _lin(x1n, W["w1"])
        u = _lin(x1n, W["w3"])
        a = silu(g) * u
        return _lin(a, W["w2"], W.get("b2")), {"g": g, "u": u, "a": a}
    z = _lin(x1n, W["w1"], W.get("b1"))
    a = gelu(z, cfg.act)
    return _lin(a, W["w2"], W.get("b2")), {"z": z, "a": a}


def layer_forward(x, W, cfg: LayerCfg, keep=False):
    """y = x1 + FFN(N2(x1)),  x1 = x + Attn(N1(x)) Wo^T + bo.

    x: [b, s, h].  Returns y (and a cache of intermediates when keep=True)."""
    W = _as64(W)
    x = np.asarray(x, F64)
    ys, caches = [], []
    for bi in range(x.shape[0]):
        xb = x[bi]
        xn, xhat1, rstd1 = norm_forward(xb, W["ln1_w"], W.get("ln1_b"), cfg)
        o, lse, q, k, v = attention_block(xn, W, cfg)
        x1 = xb + _lin(o, W["wo"], W.get("bo"))
        x1n, xhat2, rstd2 = norm_forward(x1, W["ln2_w"], W.get("ln2_b"), cfg)
        f, fc = ffn_forward(x1n, W, cfg)
        ys.append(x1 + f)
        if keep:
            caches.append(dict(xn=xn, xhat1=xhat1, rstd1=rstd1, o=o, lse=lse, q=q, k=k, v=v,
                               x1=x1, x1n=x1n, xhat2=xhat2, rstd2=rstd2, **fc))
    y = np.stack(ys)
    return (y, caches) if keep else y


def layer_backward(x, W, dy, cfg: LayerCfg):
    """Analytic gradient of layer_forward.  Returns (dx, grads) with grads keyed
    like the weights."""
    W64 = _as64(W)
    dy = np.asarray(dy, F64)
    _, caches = layer_forward(x, W, cfg, keep=True)
    H, Hk, d, G = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.group
    grads = {k: np.zeros(np.shape(v), F64) for k, v in W64.items() if v is not None}
    dxs = []
    for bi, c in enumerate(caches):
        g_ = dy[bi]
        # FFN branch
        if cfg.act == ACT_SWIGLU:
            grads["w2"] += g_.T @ c["a"]
            da = g_ @ W64["w2"]
            dg = da * c["u"] * silu_grad(c["g"])
            du = da * silu(c["g"])
            grads["w1"] += dg.T @ c["x1n"]
            grads["w3"] += du.T @ c["x1n"]
            dx1n = dg @ W64["w1"] + du @ W64["w3"]
        else:
            grads["w2"] += g_.T @ c["a"]
            da = g_ @ W64["w2"]
            dz = da * gelu_grad(c["z"], cfg.act)
            grads["w1"] += dz.T @ c["x1n"]
            dx1n = dz @ W64["w1"]
            if cfg.has_bias:
                grads["b1"] += dz.sum(0)
        if cfg.has_bias:
            grads["b2"] += g_.sum(0)
        dx1_n, dw, db = norm_backward(dx1n, c["xhat2"], c["rstd2"], W64["ln2_w"], cfg)
        grads["ln2_w"] += dw
        if db is not None:
            grads["ln2_b"] += db
        dx1 = g_ + dx1_n
        # attention branch
        grads["wo"] += dx1.T @ c["o"]
        if cfg.has_bias:
            grads["bo"] += dx1.sum(0)
        do = _split_heads(dx1 @ W64["wo"], H, d)
        dq = np.zeros_like(c["q"])
        dk = np.zeros_like(c["k"])
        dv = np.zeros_like(c["v"])
        for n in range(H):
            gk = n // G
            a_, b_, c_ = attention_head_backward(c["q"][:, n], c["k"][:, gk], c["v"][:, gk],
                                                 do[:, n], cfg.causal)
            dq[:, n] += a_
            dk[:, gk] += b_
            dv[:, gk] += c_
        if cfg.rope_base:
            # back through the rotation (the cache holds the rotated q, k)
            dq = rope(dq, cfg.rope_base, inverse=True)
            dk = rope(dk, cfg.rope_base, inverse=True)
        dq = dq.reshape(dq.shape[0], -1)
        dk = dk.reshape(dk.shape[0], -1)
        dv = dv.reshape(dv.shape[0], -1)
        xn = c["xn"]
        grads["wq"] += dq.T @ xn
        grads["wk"] += dk.T @ xn
        grads["wv"] += dv.T @ xn
        if cfg.has_bias:
            grads["bq"] += dq.sum(0)
            grads["bk"] += dk.sum(0)
            grads["bv"] += dv.sum(0)
        dxn = dq @ W64["wq"] + dk @ W64["wk"] + dv @ W64["wv"]
        dx_n, dw, db = norm_backward(dxn, c["xhat1"], c["rstd1"], W64["ln1_w"], cfg)
        grads["ln1_w"] += dw
        if db is not None:
            grads["ln1_b"] += db
        dxs.append(dx1 + dx_n)
    return np.stack(dxs), grads


# ----------------------------------------------------------------------------
# blockwise variant (Algorithm 1 / Figure 3 of the BPT page), for pinning only
# ----------------------------------------------------------------------------

def blockwise_attention(q, k, v, causal, c_q, c_kv, kv_order=None):
    """Online-softmax attention for one head, query block by query block.

    For each query block a carry (numerator, denominator, running max) is
    threaded over the key/value blocks in ``kv_order`` (default: natural
    order).  Each step: scores with the block's causal bias, new max = max(old
    max, block max), correction = exp(old max - new max), numerator and
    denominator rescaled by the correction plus the block's exp(scores - new
    max) terms.  The output is numerator / denominator."""
    s_, d = q.shape
    scale = 1.0 / sqrt(d)
    nkv = -(-s_ // c_kv)
    order = list(range(nkv)) if kv_order is None else list(kv_order)
    out = np.empty((s_, v.shape[1]), F64)
    for q0 in range(0, s_, c_q):
        q1 = min(s_, q0 + c_q)
        out[q0:q1] = _query_block_attention(q[q0:q1], k, v, q0, causal, c_kv, order)
    return out


def bpt_layer_forward(x, W, cfg: LayerCfg, c_q, c_kv):
    """The BPT schedule: projections for the whole sequence, then for each
    query block the blockwise attention of all heads, the output projection
    with residual, and the FFN with residual on that block alone."""
    W = _as64(W)
    x = np.asarray(x, F64)
    H, Hk, d, G = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.group
    out = np.empty_like(x)
    for bi in range(x.shape[0]):
        xb = x[bi]
        xn, _, _ = norm_forward(xb, W["ln1_w"], W.get("ln1_b"), cfg)
        q = _split_heads(_lin(xn, W["wq"], W.get("bq")), H, d)
        k = _split_heads(_lin(xn, W["wk"], W.get("bk")), Hk, d)
        v = _split_heads(_lin(xn, W["wv"], W.get("bv")), Hk, d)
        if cfg.rope_base:
            q = rope(q, cfg.rope_base)
            k = rope(k, cfg.rope_base)
        s_ = xb.shape[0]
        for q0 in range(0, s_, c_q):
            q1 = min(s_, q0 + c_q)
            kv_end = q1 if cfg.causal else s_
            a = np.empty((q1 - q0, H, d), F64)
            for n in range(H):
                g = n // G
                # attention of this query block against keys [0, kv_end)
                a[:, n] = _query_block_attention(q[q0:q1, n], k[:kv_end, g], v[:kv_end, g],
                                                 q0, cfg.causal, c_kv)
            x1 = xb[q0:q1] + _lin(a.reshape(q1 - q0, H * d), W["wo"], W.get("bo"))
            x1n, _, _ = norm_forward(x1, W["ln2_w"], W.get("ln2_b"), cfg)
            f, _ = ffn_forward(x1n, W, cfg)
            out[bi, q0:q1] = x1 + f
    return out


def _query_block_attention(qb, k, v, q0, causal, c_kv, order=None):
    """Algorithm 1's inner loop for one query block starting at row q0:
    the carry (numerator, denominator, running max) is threaded over the
    key/value blocks, in ``order`` if given."""
    d = qb.shape[1]
    scale = 1.0 / sqrt(d)
    num = np.zeros((qb.shape[0], v.shape[1]), F64)
    den = np.zeros((qb.shape[0], 1), F64)
    mx = np.full((qb.shape[0], 1), -np.inf)
    nkv = -(-k.shape[0] // c_kv)
    for jb in (range(nkv) if order is None else order):
        k0, k1 = jb * c_kv, min(k.shape[0], (jb + 1) * c_kv)
        S = (qb @ k[k0:k1].T) * scale
        if causal:
            i = np.arange(q0, q0 + qb.shape[0])[:, None]
            j = np.arange(k0, k1)[None, :]
            S = np.where(j > i, -np.inf, S)
        new_mx = np.maximum(mx, S.max(1, keepdims=True))
        corr = np.exp(mx - new_mx)
        E = np.exp(S - new_mx)
        num = num * corr + E @ v[k0:k1]
        den = den * corr + E.sum(1, keepdims=True)
        mx = new_mx
    return num / den
