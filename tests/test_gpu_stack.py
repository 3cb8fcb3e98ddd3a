"""The layer stack with a checkpoint every k layers on the GPU: for every k,
its output equals chaining the layer calls by hand bit for bit, and its
gradients equal the hand-chained backward up to the summation order of the
weight-gradient reductions.  (The schedule itself is pinned against the
oracle's stack on the CPU; each layer call against the oracle elsewhere.)"""
import pytest
import torch

import blockwise_attention_ffn_gb300 as bpt
from blockwise_attention_ffn_gb300 import stack
from blockwise_attention_ffn_gb300.presets import LayerConfig
from blockwise_attention_ffn_gb300.synth import make_layer_inputs

pytestmark = pytest.mark.gpu

CFG = LayerConfig(b=1, s=300, h=256, n_heads=4, n_kv_heads=4, head_dim=64, ffn_dim=1024, ffn_block=128,
                  name="gpt stack")
L = 3


def _weights():
    return [{k: (None if v is None else v.cuda()) for k, v in
             make_layer_inputs(CFG, seed=30 + i, device="cpu", with_dy=False)["weights"].items()}
            for i in range(L)]


def test_checkpointed_stack_equals_chained_layer_calls():
    Ws = _weights()
    inp = make_layer_inputs(CFG, seed=40, device="cpu")
    x, dy = inp["x"].cuda(), inp["dy"].cuda()
    ws = bpt.alloc_bytes(max(bpt.bpt_workspace_bytes(CFG, bpt.BPT_PASS_FWD),
                             bpt.bpt_workspace_bytes(CFG, bpt.BPT_PASS_BWD)))
    # by hand: every layer input kept
    xs, saved = [x], []
    for W in Ws:
        y = torch.empty_like(x)
        sv = bpt.alloc_bytes(bpt.bpt_saved_bytes(CFG))
        bpt.bpt_layer_fwd(CFG, W, xs[-1], y, sv, ws)
        xs.append(y)
        saved.append(sv)
    g, grads_ref = dy, [None] * L
    for i in range(L - 1, -1, -1):
        dx = torch.empty_like(x)
        grads_ref[i] = bpt.alloc_grads(Ws[i])
        bpt.bpt_layer_bwd(CFG, Ws[i], xs[i], saved[i], g, dx, grads_ref[i], ws)
        g = dx
    torch.cuda.synchronize()
    assert bpt.bpt_last_device_error() == (bpt.BPT_OK, 0)

    for k in (1, 2, 3):
        y, st = stack.stack_fwd(CFG, Ws, x, k, ws=ws)
        assert torch.equal(y, xs[-1]), k
        dx, grads = stack.stack_bwd(CFG, Ws, st, dy, ws=ws)
        torch.cuda.synchronize()
        assert bpt.bpt_last_device_error() == (bpt.BPT_OK, 0)
        assert st.peak_held == stack.held_inputs(L, k)
        # dx: at most one bf16 unit apart (it is not reduced across CTAs, so
        # normally identical)
        d = (dx.float() - g.float()).abs()
        assert torch.all(d <= 2.0 ** -7 * g.float().abs().clamp_min(2.0 ** -10)), (k, float(d.max()))
        for i in range(L):
            for name, ref_g in grads_ref[i].items():
                if ref_g is None:
                    continue
                got = grads[i][name]
                den = float(ref_g.norm()) or 1.0
                rel = float((got - ref_g).norm()) / den
                assert rel <= 1e-5, (k, i, name, rel)
