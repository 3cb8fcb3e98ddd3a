"""fp64 oracle of the language-model loss after the last layer (next row).

TEST INFRASTRUCTURE ONLY, like the rest of :mod:`oracle`.

"Blockwise Parallel Transformer for Long Context Large Models", section 3
(the remark before Algorithm 1, "Handling of cross-entropy loss"): the
blockwise schedule applies to the final cross-entropy loss too.  Each block of
positions forms its logits against the whole vocabulary, takes the
log-softmax at its target tokens and adds to the loss, so the s x V logit
matrix never exists.  "Untied Ulysses: Memory-Efficient Context Parallelism
via Headwise Chunking" (the prior-work paragraph on Arctic Long Sequence
Training, with its Table 1) counts that loss among the largest activation
terms (240 S d_model bytes) and adopts a tiled loss for it.

Definition (the plain reading): logits z_i = x_i W^T for positions i < s,
with W the [V, h] output projection (nn.Linear layout, no bias), and
    loss = (1 / s) * sum_i ( logsumexp_v z_iv - z_i,t_i ),
the mean token cross-entropy over the sequence (natural log).  Its gradient
is dz_i = (softmax(z_i) - onehot(t_i)) / s, so dx = dz W and dW = dz^T x.

Two blockwise forms exist only to pin the definition against the claim that
blocking does not change the result: blocks of positions (the page's form),
and blocks of the vocabulary with an online log-sum-exp carry (running max
and rescaled sum, the same bookkeeping as the attention's online softmax),
which is what a kernel that never holds a whole row of V logits needs.
"""
from __future__ import annotations

import numpy as np

F64 = np.float64


def _lse_rows(z):
    m = z.max(1, keepdims=True)
    return (m + np.log(np.exp(z - m).sum(1, keepdims=True)))[:, 0]


def lm_loss(x, W, targets):
    """Mean token cross-entropy of x [s, h] against targets [s] through
    the vocabulary projection W [V, h]."""
    x = np.asarray(x, F64)
    W = np.asarray(W, F64)
    t = np.asarray(targets)
    z = x @ W.T
    return float(np.mean(_lse_rows(z) - z[np.arange(len(t)), t]))


def lm_loss_backward(x, W, targets):
    """(dx, dW) of :func:`lm_loss`."""
    x = np.asarray(x, F64)
    W = np.asarray(W, F64)
    t = np.asarray(targets)
    s_ = x.shape[0]
    z = x @ W.T
    p = np.exp(z - _lse_rows(z)[:, None])
    p[np.arange(s_), t] -= 1.0
    dz = p / s_
    return dz @ W, dz.T @ x


def row_logsumexp(x, W, rows=None, c=1024):
    """log sum_v exp(z_iv) of the logits z = x W^T for the positions in
    ``rows`` (all by default), formed c positions at a time so that a long
    sequence never holds its whole logit matrix: the per-position quantity
    the loss subtracts the target's logit from."""
    x = np.asarray(x, F64)
    W = np.asarray(W, F64)
    idx = np.arange(x.shape[0]) if rows is None else np.asarray(rows)
    out = np.empty(len(idx))
    for r0 in range(0, len(idx), c):
        out[r0:r0 + c] = _lse_rows(x[idx[r0:r0 + c]] @ W.T)
    return out


def lm_loss_and_lse(x, W, targets, c=1024):
    """(loss, per-position log-sum-exp) in one pass over blocks of c
    positions: the loss is the mean of lse_i - z_i,t_i."""
    x = np.asarray(x, F64)
    W = np.asarray(W, F64)
    t = np.asarray(targets)
    lse = np.empty(x.shape[0])
    zt = np.empty(x.shape[0])
    for r0 in range(0, x.shape[0], c):
        z = x[r0:r0 + c] @ W.T
        lse[r0:r0 + c] = _lse_rows(z)
        zt[r0:r0 + c] = z[np.arange(z.shape[0]), t[r0:r0 + c]]
    return float(np.mean(lse - zt)), lse


def lm_dw_rows(x, W, targets, lse, vrows):
    """Rows ``vrows`` of dW = dz^T x, with dz_iv = (exp(z_iv - lse_i) -
    [t_i = v]) / s: only the logits of those vocabulary entries are formed,
    given every position's log-sum-exp (from :func:`lm_loss_and_lse`)."""
    x = np.asarray(x, F64)
    W = np.asarray(W, F64)
    t = np.asarray(targets)
    v = np.asarray(vrows)
    z = x @ W[v].T                                    # [s, len(v)]
    dz = np.exp(z - np.asarray(lse, F64)[:, None]) - (t[:, None] == v[None, :])
    return dz.T @ x / x.shape[0]


def lm_loss_row_blocks(x, W, targets, c):
    """The page's form: positions in blocks of c, each block's logits formed,
    reduced to its loss terms and dropped before the next block."""
    x = np.asarray(x, F64)
    W = np.asarray(W, F64)
    t = np.asarray(targets)
    total = 0.0
    for r0 in range(0, x.shape[0], c):
        z = x[r0:r0 + c] @ W.T
        total += float(np.sum(_lse_rows(z) - z[np.arange(z.shape[0]), t[r0:r0 + c]]))
    return total / x.shape[0]


def lm_loss_vocab_blocks(x, W, targets, c_v):
    """Vocabulary blocks of c_v with an online log-sum-exp per position: for
    each block, new max = max(old max, block max), sum = sum * exp(old max -
    new max) + sum over the block of exp(z - new max); the target's logit is
    picked from the block that holds it."""
    x = np.asarray(x, F64)
    W = np.asarray(W, F64)
    t = np.asarray(targets)
    s_ = x.shape[0]
    mx = np.full(s_, -np.inf)
    sm = np.zeros(s_)
    zt = np.zeros(s_)
    for v0 in range(0, W.shape[0], c_v):
        z = x @ W[v0:v0 + c_v].T
        new = np.maximum(mx, z.max(1))
        sm = sm * np.exp(mx - new) + np.exp(z - new[:, None]).sum(1)
        mx = new
        inb = (t >= v0) & (t < v0 + z.shape[1])
        zt[inb] = z[np.nonzero(inb)[0], t[inb] - v0]
    return float(np.mean(mx + np.log(sm) - zt))
