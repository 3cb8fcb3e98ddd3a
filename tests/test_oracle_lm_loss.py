"""Pins of the language-model loss oracle (the blockwise cross-entropy row).

Each would fail for a plausible mistake: a wrong log-sum-exp or target pick
(uniform closed form, library cross-check), a missing 1/s or a transposed
product in the gradient (finite differences, zero column sums), or broken
online bookkeeping (vocabulary blocks == vanilla)."""
import numpy as np
import pytest
import torch

from oracle import lm_loss as L


def _case(seed, s=23, h=12, V=37, scale=1.0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((s, h)) * scale
    W = rng.standard_normal((V, h)) * scale
    t = rng.integers(0, V, s)
    return x, W, t


def test_zero_projection_gives_log_vocab():
    """All logits equal: every position's loss is ln V exactly, and the
    gradient of W is (1/V - onehot(t))^T x / s."""
    x, W, t = _case(30)
    W0 = np.zeros_like(W)
    V, s = W.shape[0], x.shape[0]
    assert abs(L.lm_loss(x, W0, t) - np.log(V)) < 1e-14
    _, dW = L.lm_loss_backward(x, W0, t)
    want = (np.full((s, V), 1.0 / V) - np.eye(V)[t]).T @ x / s
    assert np.max(np.abs(dW - want)) < 1e-14


def test_matches_torch_cross_entropy():
    x, W, t = _case(31, scale=2.0)
    xt = torch.tensor(x, requires_grad=True)
    Wt = torch.tensor(W, requires_grad=True)
    loss = torch.nn.functional.cross_entropy(xt @ Wt.T, torch.tensor(t))
    loss.backward()
    assert abs(L.lm_loss(x, W, t) - loss.item()) < 1e-12
    dx, dW = L.lm_loss_backward(x, W, t)
    assert np.max(np.abs(dx - xt.grad.numpy())) < 1e-13
    assert np.max(np.abs(dW - Wt.grad.numpy())) < 1e-13


def test_gradient_matches_finite_differences():
    x, W, t = _case(32, s=7, h=5, V=9)
    dx, dW = L.lm_loss_backward(x, W, t)
    eps = 1e-6
    for arr, g, f in ((x, dx, lambda a: L.lm_loss(a, W, t)), (W, dW, lambda a: L.lm_loss(x, a, t))):
        fd = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            p = arr.copy(); p[idx] += eps
            m = arr.copy(); m[idx] -= eps
            fd[idx] = (f(p) - f(m)) / (2 * eps)
        assert np.linalg.norm(fd - g) <= 1e-7 * np.linalg.norm(g)


def test_vocabulary_gradient_columns_sum_to_zero():
    """softmax - onehot sums to zero over the vocabulary in every row, so the
    columns of dW (summed over the vocabulary) vanish."""
    x, W, t = _case(33, scale=3.0)
    _, dW = L.lm_loss_backward(x, W, t)
    assert np.max(np.abs(dW.sum(0))) < 1e-13


@pytest.mark.parametrize("c", [1, 5, 23, 64])
def test_position_blocks_equal_vanilla(c):
    x, W, t = _case(34, scale=2.0)
    assert abs(L.lm_loss_row_blocks(x, W, t, c) - L.lm_loss(x, W, t)) < 1e-13


@pytest.mark.parametrize("c_v", [1, 4, 10, 37, 100])
def test_vocabulary_blocks_with_online_lse_equal_vanilla(c_v):
    x, W, t = _case(35, scale=4.0)   # large logits: the running max must do its job
    assert abs(L.lm_loss_vocab_blocks(x, W, t, c_v) - L.lm_loss(x, W, t)) < 1e-12


def test_row_logsumexp_matches_scipy_and_the_loss():
    """The per-position log-sum-exp equals SciPy's logsumexp of the logits
    (a library routine), for all rows and for a sample in any order, and the
    loss is the mean of it minus the target logits."""
    from scipy.special import logsumexp
    x, W, t = _case(36, scale=3.0)
    z = x @ W.T
    want = logsumexp(z, axis=1)
    for c in (1, 4, 1024):
        assert np.max(np.abs(L.row_logsumexp(x, W, c=c) - want)) < 1e-12
    rows = np.array([5, 0, 22, 7])
    assert np.max(np.abs(L.row_logsumexp(x, W, rows=rows) - want[rows])) < 1e-12
    assert abs(np.mean(want - z[np.arange(len(t)), t]) - L.lm_loss(x, W, t)) < 1e-13


@pytest.mark.parametrize("c", [1, 6, 1024])
def test_one_pass_loss_and_lse_and_sampled_dw_rows(c):
    """The one-pass (loss, lse) equals the vanilla loss and SciPy's
    logsumexp; dW at chosen vocabulary rows, given that lse, equals those rows
    of the full gradient (target rows and others, repeated and unordered)."""
    from scipy.special import logsumexp
    x, W, t = _case(37, scale=2.0)
    loss, lse = L.lm_loss_and_lse(x, W, t, c=c)
    assert abs(loss - L.lm_loss(x, W, t)) < 1e-13
    assert np.max(np.abs(lse - logsumexp(x @ W.T, axis=1))) < 1e-12
    _, dW = L.lm_loss_backward(x, W, t)
    vrows = np.array([t[0], 0, 36, t[3], 5, t[0]])
    assert np.max(np.abs(L.lm_dw_rows(x, W, t, lse, vrows) - dW[vrows])) < 1e-13
