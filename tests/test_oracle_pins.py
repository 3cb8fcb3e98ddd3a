"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Each test would fail for a plausible mistake in the oracle: a dropped
residual, bias or norm term (parameter count, autograd, finite differences,
FFN-zero invariant), a wrong scale or mask (identical keys, library
attention), a wrong sign or transposed operand in the backward (finite
differences, autograd), or broken online-softmax bookkeeping (blockwise ==
vanilla, kv-order permutation), and for the rotary embedding a wrong pairing,
sign or frequency (complex-rotation form, offset-only scores) or a missing
rotation in the backward (finite differences)."""
import json
import os

import numpy as np
import pytest

from oracle import ref, tiny
from oracle.ref import LayerCfg
from tests.oracle_helpers import rand_layer

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_numbers.json")))


def _cfgs_small():
    return [
        LayerCfg(s=37, h=32, n_heads=4, n_kv_heads=4, head_dim=8, ffn_dim=48),
        LayerCfg(s=37, h=32, n_heads=4, n_kv_heads=4, head_dim=8, ffn_dim=48, causal=False),
        LayerCfg(s=29, h=32, n_heads=4, n_kv_heads=2, head_dim=8, ffn_dim=40, norm=1, act=2,
                 has_bias=False),
        LayerCfg(s=21, h=24, n_heads=2, n_kv_heads=1, head_dim=12, ffn_dim=40, act=1, b=2),
        LayerCfg(s=29, h=32, n_heads=4, n_kv_heads=2, head_dim=8, ffn_dim=40, norm=1, act=2,
                 has_bias=False, rope_base=10000.0),
    ]


# -------------------------------------------------- blockwise == vanilla (BPT exactness)

@pytest.mark.parametrize("causal", [True, False])
def test_one_block_equals_vanilla(causal):
    rng = np.random.default_rng(1)
    s, d = 53, 16
    q, k, v = (rng.standard_normal((s, d)) for _ in range(3))
    o, _ = ref.attention_head(q, k, v, causal)
    ob = ref.blockwise_attention(q, k, v, causal, c_q=s, c_kv=s)
    assert np.max(np.abs(o - ob)) < 1e-12


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("cq,ckv", [(16, 16), (7, 13), (64, 5), (1, 53)])
def test_blockwise_any_block_size_equals_vanilla(causal, cq, ckv):
    rng = np.random.default_rng(2)
    s, d = 53, 16
    q, k, v = (rng.standard_normal((s, d)) * 2 for _ in range(3))
    o, _ = ref.attention_head(q, k, v, causal)
    ob = ref.blockwise_attention(q, k, v, causal, c_q=cq, c_kv=ckv)
    assert np.max(np.abs(o - ob)) < 1e-12


@pytest.mark.parametrize("cfg", _cfgs_small())
@pytest.mark.parametrize("cq,ckv", [(8, 8), (5, 16), (64, 64)])
def test_bpt_layer_schedule_equals_vanilla_layer(cfg, cq, ckv):
    x, W, _ = rand_layer(cfg, seed=3)
    y = ref.layer_forward(x, W, cfg)
    yb = ref.bpt_layer_forward(x, W, cfg, c_q=cq, c_kv=ckv)
    assert np.max(np.abs(y - yb)) < 1e-11


def test_kv_block_order_permutation_noncausal():
    rng = np.random.default_rng(4)
    s, d = 64, 8
    q, k, v = (rng.standard_normal((s, d)) * 3 for _ in range(3))
    base = ref.blockwise_attention(q, k, v, False, c_q=16, c_kv=8)
    for seed in range(4):
        order = np.random.default_rng(seed).permutation(8)
        ob = ref.blockwise_attention(q, k, v, False, c_q=16, c_kv=8, kv_order=order)
        assert np.max(np.abs(ob - base)) < 1e-12
    o, _ = ref.attention_head(q, k, v, False)
    assert np.max(np.abs(o - base)) < 1e-12


# -------------------------------------------------- closed forms

@pytest.mark.parametrize("causal", [True, False])
def test_identical_keys_give_mean_of_values(causal):
    rng = np.random.default_rng(5)
    s, d = 40, 8
    q = rng.standard_normal((s, d)) * 4
    k = np.tile(rng.standard_normal((1, d)), (s, 1))
    v = rng.standard_normal((s, d))
    o, lse = ref.attention_head(q, k, v, causal)
    if causal:
        want = np.cumsum(v, 0) / np.arange(1, s + 1)[:, None]
        assert np.array_equal(o[0], v[0])  # row 0 sees key 0 only: exactly V_0
    else:
        want = np.broadcast_to(v.mean(0), v.shape)
    assert np.max(np.abs(o - want)) < 1e-13
    # lse = score + log(number of visible keys)
    sc = (q @ k[0]) / np.sqrt(d)
    cnt = np.arange(1, s + 1) if causal else np.full(s, s)
    assert np.max(np.abs(lse - (sc + np.log(cnt)))) < 1e-12


def test_zero_query_weights_give_uniform_causal_attention():
    cfg = LayerCfg(s=33, h=32, n_heads=4, n_kv_heads=2, head_dim=8, ffn_dim=48)
    x, W, _ = rand_layer(cfg, seed=6)
    W["wq"][:] = 0
    W["bq"][:] = 0
    _, cache = ref.layer_forward(x, W, cfg, keep=True)
    v = cache[0]["v"]
    for n in range(cfg.n_heads):
        want = np.cumsum(v[:, n // cfg.group], 0) / np.arange(1, cfg.s + 1)[:, None]
        got = cache[0]["o"].reshape(cfg.s, cfg.n_heads, cfg.head_dim)[:, n]
        assert np.max(np.abs(got - want)) < 1e-13


def test_zero_fc1_gives_ffn_equal_to_b2():
    cfg = LayerCfg(s=9, h=16, n_heads=2, n_kv_heads=2, head_dim=8, ffn_dim=32)
    x, W, _ = rand_layer(cfg, seed=7)
    W["w1"][:] = 0
    W["b1"][:] = 0
    y, cache = ref.layer_forward(x, W, cfg, keep=True)
    assert np.max(np.abs(y[0] - (cache[0]["x1"] + W["b2"]))) < 1e-14


def test_norms_match_their_definition():
    cfg = LayerCfg(s=9, h=16, n_heads=2, n_kv_heads=2, head_dim=8, ffn_dim=32)
    rng = np.random.default_rng(8)
    x = rng.standard_normal((9, 16)) * 3 + 1
    y, xhat, _ = ref.norm_forward(x, np.ones(16), np.zeros(16), cfg)
    assert np.allclose(y.mean(1), 0, atol=1e-14)
    assert np.allclose((y * y).mean(1), 1 / (1 + 1e-5 / x.var(1)), atol=1e-12)
    rcfg = LayerCfg(s=9, h=16, n_heads=2, n_kv_heads=2, head_dim=8, ffn_dim=32, norm=1)
    y, _, _ = ref.norm_forward(x, np.ones(16), None, rcfg)
    assert np.allclose((y * y).mean(1), (x * x).mean(1) / ((x * x).mean(1) + 1e-5), atol=1e-12)


# -------------------------------------------------- rotary position embedding

@pytest.mark.parametrize("d,base", [(2, 10000.0), (8, 10000.0), (16, 500000.0), (12, 7.0)])
def test_rope_is_a_complex_rotation(d, base):
    """Element i and i + d/2 as the real and imaginary part of one complex
    number, position p multiplies it by exp(j p base^(-2i/d)): position 0 is
    the identity and every pair keeps its length."""
    rng = np.random.default_rng(20)
    s, n = 23, 3
    x = rng.standard_normal((s, n, d))
    z = x[..., : d // 2] + 1j * x[..., d // 2:]
    freq = base ** (-np.arange(0, d, 2) / d)
    w = z * np.exp(1j * np.arange(s)[:, None, None] * freq[None, None, :])
    got = ref.rope(x, base)
    assert np.max(np.abs(got[..., : d // 2] - w.real)) < 1e-12
    assert np.max(np.abs(got[..., d // 2:] - w.imag)) < 1e-12
    assert np.array_equal(got[0], x[0])
    pair_len = np.hypot(got[..., : d // 2], got[..., d // 2:])
    assert np.max(np.abs(pair_len - np.abs(z))) < 1e-12


def test_rope_scores_depend_on_the_offset_only():
    """With the same query and key vector at every position, the rotated
    score q_m . k_n depends on m - n alone (the relative-position property)."""
    rng = np.random.default_rng(21)
    s, d = 19, 8
    q = np.tile(rng.standard_normal((1, 1, d)), (s, 1, 1))
    k = np.tile(rng.standard_normal((1, 1, d)), (s, 1, 1))
    S = ref.rope(q, 100.0)[:, 0] @ ref.rope(k, 100.0)[:, 0].T
    for off in range(-s + 1, s):
        diag = np.diagonal(S, offset=off)
        assert np.max(np.abs(diag - diag[0])) < 1e-12
    assert np.ptp(np.diagonal(S, 0)) < 1e-12 and abs(S[1, 0] - S[0, 0]) > 1e-3


def test_rope_inverse_is_its_transpose():
    rng = np.random.default_rng(22)
    x, y = rng.standard_normal((2, 17, 2, 8))
    assert np.max(np.abs(ref.rope(ref.rope(x, 50.0), 50.0, inverse=True) - x)) < 1e-12
    lhs = np.sum(ref.rope(x, 50.0) * y)
    rhs = np.sum(x * ref.rope(y, 50.0, inverse=True))
    assert abs(lhs - rhs) < 1e-10


# -------------------------------------------------- scalar-loop cross-check

@pytest.mark.parametrize("cfg", [
    LayerCfg(s=5, h=8, n_heads=2, n_kv_heads=2, head_dim=4, ffn_dim=12),
    LayerCfg(s=6, h=8, n_heads=2, n_kv_heads=1, head_dim=4, ffn_dim=12, norm=1, act=2,
             has_bias=False),
    LayerCfg(s=4, h=8, n_heads=2, n_kv_heads=2, head_dim=4, ffn_dim=12, act=1, causal=False, b=2),
    LayerCfg(s=7, h=8, n_heads=2, n_kv_heads=1, head_dim=4, ffn_dim=12, norm=1, act=2,
             has_bias=False, rope_base=10.0),
])
def test_scalar_loop_oracle_matches(cfg):
    x, W, _ = rand_layer(cfg, seed=9)
    y = ref.layer_forward(x, W, cfg)
    Wl = {k: v.tolist() for k, v in W.items()}
    yt = np.array(tiny.layer_forward(x.tolist(), Wl, cfg))
    assert np.max(np.abs(y - yt)) < 1e-12


# -------------------------------------------------- finite differences

def _fd_check(cfg, seed):
    x, W, dy = rand_layer(cfg, seed=seed)
    dx, grads = ref.layer_backward(x, W, dy, cfg)

    def loss(xx, WW):
        return float(np.sum(ref.layer_forward(xx, WW, cfg) * dy))

    eps = 1e-5
    fdx = np.zeros_like(x)
    for idx in np.ndindex(x.shape):
        xp = x.copy(); xp[idx] += eps
        xm = x.copy(); xm[idx] -= eps
        fdx[idx] = (loss(xp, W) - loss(xm, W)) / (2 * eps)
    assert np.linalg.norm(fdx - dx) <= 1e-6 * np.linalg.norm(dx)
    for name, w in W.items():
        fd = np.zeros_like(w)
        for idx in np.ndindex(w.shape):
            Wp = dict(W); Wp[name] = w.copy(); Wp[name][idx] += eps
            Wm = dict(W); Wm[name] = w.copy(); Wm[name][idx] -= eps
            fd[idx] = (loss(x, Wp) - loss(x, Wm)) / (2 * eps)
        assert np.linalg.norm(fd - grads[name]) <= 1e-6 * np.linalg.norm(grads[name]) + 1e-9, name
    if "bk" in grads and not cfg.rope_base:
        # softmax is shift-invariant along a row, so a bias added to every key
        # cannot change the output: its gradient is exactly zero (not so once
        # the rotary embedding turns the bias differently at every position)
        assert np.max(np.abs(grads["bk"])) < 1e-12


@pytest.mark.parametrize("cfg", [
    LayerCfg(s=6, h=8, n_heads=2, n_kv_heads=2, head_dim=4, ffn_dim=12),
    LayerCfg(s=5, h=8, n_heads=2, n_kv_heads=2, head_dim=4, ffn_dim=12, causal=False, act=1),
    LayerCfg(s=6, h=8, n_heads=2, n_kv_heads=1, head_dim=4, ffn_dim=12, norm=1, act=2,
             has_bias=False),
    LayerCfg(s=6, h=8, n_heads=2, n_kv_heads=1, head_dim=4, ffn_dim=12, rope_base=10.0),
])
def test_backward_matches_finite_differences(cfg):
    _fd_check(cfg, seed=10)


# -------------------------------------------------- the pages' printed numbers

def test_param_count_matches_pages():
    from oracle.accounting import gpt_layer_params, param_count
    for e in GOLD["gpt_layer_params"]:
        h = e["h"]
        cfg = LayerCfg(s=8, h=h, n_heads=4, n_kv_heads=4, head_dim=h // 4, ffn_dim=4 * h)
        assert param_count(cfg) == e["value"], e["cite"]
        assert gpt_layer_params(h) == e["value"]


def test_llama_param_count_matches_formula():
    from oracle.accounting import llama_layer_params, param_count
    cfg = LayerCfg(s=8, h=4096, n_heads=32, n_kv_heads=8, head_dim=128, ffn_dim=14336, norm=1,
                   act=2, has_bias=False)
    assert param_count(cfg) == llama_layer_params(4096, 14336, 4)
