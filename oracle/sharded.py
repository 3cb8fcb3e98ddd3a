"""fp64 oracle of one layer sharded by sequence position over P ranks.

TEST INFRASTRUCTURE ONLY, like the rest of :mod:`oracle`.  The library runs
on one GPU; this module states, and lets the tests check on CPU ranks, how the
same layer splits across devices and which exchanges it needs:

* Norms, projections and the FFN are position-wise, so each rank computes them
  for its own rows alone.
* A query row attends to the keys and values of every position at or before
  it, so each rank needs K and V of the whole sequence: one all-gather of K
  and V per layer.  "Untied Ulysses: Memory-Efficient Context Parallelism via
  Headwise Chunking" ("Where Prior Approaches Fall Short", the Ring Attention
  paragraph) passes the same K/V shards around a ring of devices instead;
  every rank ends up attending to the full sequence either way, and the
  result is the same.
* In the backward pass a rank's queries give gradients for the keys and
  values of every position: those partial dK and dV are summed over ranks
  and each rank keeps its own rows (a reduce-scatter).  Weight gradients are
  sums over positions, so they are summed over ranks (an all-reduce).
* Rows go to ranks in the zigzag order the same page's baselines use for
  causal load balance (its "Baselines" list, USP-Ring and native PyTorch
  ring).  Reading, since the page names the order without defining it: the
  sequence is cut into 2P equal chunks and rank r takes chunks r and
  2P - 1 - r, so every rank holds one early and one late chunk and the same
  number of unmasked (query, key) pairs.

Collectives are passed in (``comm``), so the arithmetic here has no
dependence on how ranks talk: the tests use torch.distributed over gloo.
The layer definition is :mod:`oracle.ref`'s; only attention over rows at
arbitrary positions is written out again here.
"""
from __future__ import annotations

from math import sqrt

import numpy as np

from .ref import (ACT_SWIGLU, F64, LayerCfg, _as64, _lin, ffn_forward, gelu_grad, norm_backward,
                  norm_forward, rope, silu, silu_grad)


def zigzag_rows(s: int, P: int, r: int) -> np.ndarray:
    """Global positions held by rank r of P: chunks r and 2P-1-r of 2P."""
    assert s % (2 * P) == 0, "the zigzag split wants s divisible by 2P"
    c = s // (2 * P)
    return np.concatenate([np.arange(r * c, (r + 1) * c), np.arange((2 * P - 1 - r) * c, (2 * P - r) * c)])


def causal_pairs(rows) -> int:
    """Unmasked (query, key) pairs of the given query positions: p + 1 each."""
    return int(np.sum(np.asarray(rows) + 1))


def _probs(q, qpos, k, kpos, causal):
    """softmax(q k^T / sqrt(d) + M) over the keys, M = -inf where a key's
    position exceeds the query's."""
    S = (q @ k.T) / sqrt(q.shape[1])
    if causal:
        S = np.where(kpos[None, :] > qpos[:, None], -np.inf, S)
    E = np.exp(S - S.max(1, keepdims=True))
    return E / E.sum(1, keepdims=True)


def _heads(t, n, d):
    return t.reshape(t.shape[0], n, d)


def _local_qkv(xb, pos, W, cfg):
    xn, xhat1, rstd1 = norm_forward(xb, W["ln1_w"], W.get("ln1_b"), cfg)
    H, Hk, d = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim
    q = _heads(_lin(xn, W["wq"], W.get("bq")), H, d)
    k = _heads(_lin(xn, W["wk"], W.get("bk")), Hk, d)
    v = _heads(_lin(xn, W["wv"], W.get("bv")), Hk, d)
    if cfg.rope_base:
        q = rope(q, cfg.rope_base, positions=pos)
        k = rope(k, cfg.rope_base, positions=pos)
    return xn, xhat1, rstd1, q, k, v


def _forward_rows(xb, pos, W, cfg, comm):
    """One sequence's rows on this rank; returns y and what the backward
    needs.  comm.all_gather(a) returns every rank's a, in rank order."""
    xn, xhat1, rstd1, q, k, v = _local_qkv(xb, pos, W, cfg)
    kpos = np.concatenate(comm.all_gather(np.asarray(pos, F64)))
    K = np.concatenate(comm.all_gather(k))   # [s, Hk, d], rows in rank order
    V = np.concatenate(comm.all_gather(v))
    H, d, G = cfg.n_heads, cfg.head_dim, cfg.group
    o = np.empty_like(q)
    probs = []
    for n in range(H):
        Pn = _probs(q[:, n], pos, K[:, n // G], kpos, cfg.causal)
        o[:, n] = Pn @ V[:, n // G]
        probs.append(Pn)
    o = o.reshape(xb.shape[0], H * d)
    x1 = xb + _lin(o, W["wo"], W.get("bo"))
    x1n, xhat2, rstd2 = norm_forward(x1, W["ln2_w"], W.get("ln2_b"), cfg)
    f, fc = ffn_forward(x1n, W, cfg)
    cache = dict(xn=xn, xhat1=xhat1, rstd1=rstd1, q=q, K=K, V=V, probs=probs, o=o, x1n=x1n,
                 xhat2=xhat2, rstd2=rstd2, **fc)
    return x1 + f, cache


def rank_layer_forward(x_r, pos, W, cfg: LayerCfg, comm):
    """y for this rank's rows: x_r [b, rows, h] holds the positions `pos`."""
    W = _as64(W)
    return np.stack([_forward_rows(np.asarray(xb, F64), pos, W, cfg, comm)[0] for xb in x_r])


def rank_layer_backward(x_r, pos, W, dy_r, cfg: LayerCfg, comm):
    """(dx for this rank's rows, weight gradients summed over all ranks).
    comm.all_reduce(a) returns the elementwise sum of every rank's a."""
    W = _as64(W)
    H, Hk, d, G = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.group
    rows = len(pos)
    me = comm.rank
    grads = {k: np.zeros(np.shape(v), F64) for k, v in W.items() if v is not None}
    dxs = []
    for xb, g_ in zip(np.asarray(x_r, F64), np.asarray(dy_r, F64)):
        _, c = _forward_rows(xb, pos, W, cfg, comm)
        # FFN branch and second norm: own rows only
        grads["w2"] += g_.T @ c["a"]
        da = g_ @ W["w2"]
        if cfg.act == ACT_SWIGLU:
            dg = da * c["u"] * silu_grad(c["g"])
            du = da * silu(c["g"])
            grads["w1"] += dg.T @ c["x1n"]
            grads["w3"] += du.T @ c["x1n"]
            dx1n = dg @ W["w1"] + du @ W["w3"]
        else:
            dz = da * gelu_grad(c["z"], cfg.act)
            grads["w1"] += dz.T @ c["x1n"]
            dx1n = dz @ W["w1"]
            if cfg.has_bias:
                grads["b1"] += dz.sum(0)
        if cfg.has_bias:
            grads["b2"] += g_.sum(0)
        dx1_n, dw, db = norm_backward(dx1n, c["xhat2"], c["rstd2"], W["ln2_w"], cfg)
        grads["ln2_w"] += dw
        if db is not None:
            grads["ln2_b"] += db
        dx1 = g_ + dx1_n
        grads["wo"] += dx1.T @ c["o"]
        if cfg.has_bias:
            grads["bo"] += dx1.sum(0)
        do = _heads(dx1 @ W["wo"], H, d)
        # attention: own queries, all keys; partial dK, dV for every position
        scale = 1.0 / sqrt(d)
        dq = np.zeros_like(c["q"])
        dK = np.zeros_like(c["K"])
        dV = np.zeros_like(c["V"])
        for n in range(H):
            Pn, gk = c["probs"][n], n // G
            dP = do[:, n] @ c["V"][:, gk].T
            dS = Pn * (dP - (Pn * dP).sum(1, keepdims=True))
            dV[:, gk] += Pn.T @ do[:, n]
            dq[:, n] = (dS @ c["K"][:, gk]) * scale
            dK[:, gk] += (dS.T @ c["q"][:, n]) * scale
        # reduce-scatter: sum over ranks, keep this rank's rows (rank order)
        dk = comm.all_reduce(dK)[me * rows:(me + 1) * rows]
        dv = comm.all_reduce(dV)[me * rows:(me + 1) * rows]
        if cfg.rope_base:
            dq = rope(dq, cfg.rope_base, inverse=True, positions=pos)
            dk = rope(dk, cfg.rope_base, inverse=True, positions=pos)
        dq, dk, dv = (t.reshape(rows, -1) for t in (dq, dk, dv))
        xn = c["xn"]
        grads["wq"] += dq.T @ xn
        grads["wk"] += dk.T @ xn
        grads["wv"] += dv.T @ xn
        if cfg.has_bias:
            grads["bq"] += dq.sum(0)
            grads["bk"] += dk.sum(0)
            grads["bv"] += dv.sum(0)
        dxn = dq @ W["wq"] + dk @ W["wk"] + dv @ W["wv"]
        dx_n, dw, db = norm_backward(dxn, c["xhat1"], c["rstd1"], W["ln1_w"], cfg)
        grads["ln1_w"] += dw
        if db is not None:
            grads["ln1_b"] += db
        dxs.append(dx1 + dx_n)
    grads = {k: comm.all_reduce(v) for k, v in sorted(grads.items())}
    return np.stack(dxs), grads
