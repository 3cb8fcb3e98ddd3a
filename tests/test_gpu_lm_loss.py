"""The blockwise language-model loss (vocabulary projection + mean token
cross-entropy) on the GPU against the fp64 oracle.

Small cases are compared in full: the loss, every row's log-sum-exp, dx and
dW, with the vocabulary ragged against the 256-column tile and against the
backward's vocabulary block, one and several blocks, and the accumulate and
fixed-order flags.  The full-size case (after the GPT-3B-shaped layer,
n = 32768, h = 2560, the GPT-2 vocabulary of 50257 tokens) is compared in
full for the loss and every row's log-sum-exp (one blocked oracle pass), on
64 sampled rows for dx (a row's dx depends on that row alone), and on about
60 sampled vocabulary rows for dW (given the oracle's log-sum-exp of every
row, a vocabulary row of dW needs only its own logits)."""
import numpy as np
import pytest
import torch

import blockwise_attention_ffn_gb300 as bpt
from blockwise_attention_ffn_gb300.presets import LM3, LmConfig
from blockwise_attention_ffn_gb300.synth import make_lm_inputs
from oracle import lm_loss as L
from tests.gpu_helpers import assert_close, assert_close_grad, to64

pytestmark = pytest.mark.gpu

SMALL = [
    LmConfig(n=300, h=256, vocab=1000, vocab_block=512, name="ragged two blocks"),
    LmConfig(n=1000, h=512, vocab=8191, vocab_block=2048, name="four blocks"),
    LmConfig(n=129, h=128, vocab=300, vocab_block=0, name="one block"),
    LmConfig(n=640, h=384, vocab=3000, vocab_block=768, flags=bpt.BPT_FLAG_DETERMINISTIC, name="fixed order"),
]


def run(cfg, inp, dloss=1.0):
    x, w, t = inp["x"].cuda(), inp["w"].cuda(), inp["targets"].cuda()
    loss = torch.full((1,), float("nan"), device="cuda")
    lse = torch.full((cfg.n,), float("nan"), device="cuda")
    ws = bpt.alloc_bytes(max(bpt.bpt_lm_workspace_bytes(cfg, bpt.BPT_PASS_FWD),
                             bpt.bpt_lm_workspace_bytes(cfg, bpt.BPT_PASS_BWD)))
    bpt.bpt_lm_loss_fwd(cfg, x, w, t, loss, lse, ws)
    dx = torch.full_like(x, float("nan"))
    dw = torch.full((cfg.vocab, cfg.h), float("nan"), device="cuda")
    bpt.bpt_lm_loss_bwd(cfg, x, w, t, lse, dloss, dx, dw, ws)
    torch.cuda.synchronize()
    assert bpt.bpt_last_device_error() == (bpt.BPT_OK, 0)
    return float(loss.item()), lse, dx, dw


@pytest.mark.parametrize("cfg", SMALL, ids=lambda c: c.name)
def test_lm_loss_matches_oracle(cfg):
    inp = make_lm_inputs(cfg, seed=50)
    loss, lse, dx, dw = run(cfg, inp)
    x, w = to64(inp["x"]), to64(inp["w"])
    t = inp["targets"].numpy()
    want = L.lm_loss(x, w, t)
    print(f"{cfg.name}: loss {loss:.6f} want {want:.6f}")
    assert abs(loss - want) <= 5e-3 * abs(want)
    assert_close(to64(lse), L.row_logsumexp(x, w), "lse", bf16_out=False)
    dx_ref, dw_ref = L.lm_loss_backward(x, w, t)
    assert_close(to64(dx), dx_ref, "dx", grad=True)
    assert_close_grad(to64(dw), dw_ref, "dW", name="w_vocab")


def test_lm_loss_scaled_and_accumulated():
    """dloss scales both gradients (against the oracle's, scaled: the two
    calls round dz to bf16 independently); BPT_FLAG_ACCUM_GRADS adds dW."""
    cfg = SMALL[0]
    inp = make_lm_inputs(cfg, seed=51)
    _, lse, dx1, dw1 = run(cfg, inp, dloss=1.0)
    _, _, dx3, dw3 = run(cfg, inp, dloss=-3.0)
    dx_ref, dw_ref = L.lm_loss_backward(to64(inp["x"]), to64(inp["w"]), inp["targets"].numpy())
    assert_close(to64(dx3), -3.0 * dx_ref, "dx scaled", grad=True)
    assert_close_grad(to64(dw3), -3.0 * dw_ref, "dW scaled", name="w_vocab")
    acc = cfg.with_(flags=bpt.BPT_FLAG_ACCUM_GRADS)
    x, w, t = inp["x"].cuda(), inp["w"].cuda(), inp["targets"].cuda()
    dw = dw1.clone()
    dx = torch.empty_like(x)
    ws = bpt.alloc_bytes(bpt.bpt_lm_workspace_bytes(acc, bpt.BPT_PASS_BWD))
    bpt.bpt_lm_loss_bwd(acc, x, w, t, lse, 1.0, dx, dw, ws)
    torch.cuda.synchronize()
    assert_close(to64(dw), 2 * to64(dw1), "dW accumulated", bf16_out=False, grad=True, rel_fro=1e-5)


def test_lm_loss_fixed_order_is_bitwise_repeatable():
    cfg = SMALL[3]
    inp = make_lm_inputs(cfg, seed=52)
    l0, lse0, dx0, dw0 = run(cfg, inp)
    l1, lse1, dx1, dw1 = run(cfg, inp)
    assert l0 == l1 and torch.equal(lse0, lse1) and torch.equal(dx0, dx1) and torch.equal(dw0, dw1)


def test_target_outside_the_vocabulary_is_reported():
    """Two targets outside [0, V): the call completes, their rows' terms are
    their log-sum-exp alone, and the error word reports BPT_EINVAL at the
    loss's site; the next call is clean."""
    cfg = SMALL[2]
    inp = make_lm_inputs(cfg, seed=53)
    t = inp["targets"].clone()
    t[5], t[7] = cfg.vocab, -1
    x, w = inp["x"].cuda(), inp["w"].cuda()
    loss = torch.empty(1, device="cuda")
    ws = bpt.alloc_bytes(bpt.bpt_lm_workspace_bytes(cfg, bpt.BPT_PASS_FWD))
    bpt.bpt_lm_loss_fwd(cfg, x, w, t.cuda(), loss, None, ws)
    assert bpt.bpt_last_device_error() == (bpt.BPT_EINVAL, bpt.BPT_LM_BAD_TARGET_SITE)
    assert bpt.bpt_last_device_error() == (bpt.BPT_OK, 0)
    x64, w64 = to64(inp["x"]), to64(inp["w"])
    lse = L.row_logsumexp(x64, w64)
    ok = np.ones(cfg.n, bool)
    ok[[5, 7]] = False
    tv = t.numpy()
    zt = np.einsum("ij,ij->i", x64[ok], w64[tv[ok]])
    want = (np.sum(lse[ok] - zt) + np.sum(lse[~ok])) / cfg.n
    assert abs(float(loss.item()) - want) <= 5e-3 * abs(want)
    bpt.bpt_lm_loss_fwd(cfg, x, w, inp["targets"].cuda(), loss, None, ws)
    assert bpt.bpt_last_device_error() == (bpt.BPT_OK, 0)


def test_lm_loss_full_size_sampled():
    cfg = LM3
    inp = make_lm_inputs(cfg, seed=cfg.seed)
    loss, lse, dx, dw = run(cfg, inp)
    x, w = to64(inp["x"]), to64(inp["w"])
    t = inp["targets"].numpy()
    # one oracle pass over every position: the loss and each row's lse
    want, lse_ref = L.lm_loss_and_lse(x, w, t, c=2048)
    print(f"full size: loss {loss:.6f} want {want:.6f}")
    assert abs(loss - want) <= 5e-3 * abs(want)
    assert_close(to64(lse), lse_ref, "lse (every row)", bf16_out=False)
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([[0, 1, cfg.n - 1], rng.choice(cfg.n, 61, replace=False)]))
    # dx of a row depends on that row alone: the oracle's gradient of the
    # sampled rows' own mean loss, rescaled from 1/len(rows) to 1/n
    dx_ref, _ = L.lm_loss_backward(x[rows], w, t[rows])
    assert_close(to64(dx)[rows], dx_ref * (len(rows) / cfg.n), "dx (sampled rows)", grad=True)
    # dW at sampled vocabulary rows: targets of sampled positions, the first
    # and last entries (the ragged last tile and block) and random ones
    vrows = np.unique(np.concatenate([t[rows[:24]], [0, 1, cfg.vocab - 1], rng.choice(cfg.vocab, 37)]))
    dw_ref = L.lm_dw_rows(x, w, t, lse_ref, vrows)
    assert_close_grad(to64(dw)[vrows], dw_ref, "dW (sampled vocabulary rows)", name="w_vocab")
