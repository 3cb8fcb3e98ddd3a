"""The layer stack with a checkpoint every k layers on the GPU, against
chaining the layer calls by hand.

With BPT_FLAG_DETERMINISTIC every sum of a layer call is taken in a fixed
order, and the stack repeats exactly the layer calls of the hand-chained
backward on exactly the same values (the re-run forward of a segment gives
its layer inputs bit for bit), so output, input gradient and every weight
gradient are bitwise equal for every k.

Without the flag the attention backward, the split weight-gradient products
and the bias and norm gradients add in the order their parts arrive, so two
calls on the same values may differ in the last bits of an fp32 sum and,
after rounding, by one bf16 unit in dQ/dK/dV and dx.  That difference is
bounded here by a tenth of the acceptance bound against the exact gradient
that every layer call meets on its own (the parity tests), a margin that a
wrong schedule (a stale or skipped segment) exceeds by orders of magnitude.
(The schedule itself is pinned against the oracle's stack on the CPU.)"""
import pytest
import torch

import blockwise_attention_ffn_gb300 as bpt
from blockwise_attention_ffn_gb300 import stack
from blockwise_attention_ffn_gb300.presets import LayerConfig
from blockwise_attention_ffn_gb300.synth import make_layer_inputs
from tests.gpu_helpers import REL_FRO, rel_bound

pytestmark = pytest.mark.gpu

CFG = LayerConfig(b=1, s=300, h=256, n_heads=4, n_kv_heads=4, head_dim=64, ffn_dim=1024, ffn_block=128,
                  name="gpt stack")
L = 3


def _weights():
    return [{k: (None if v is None else v.cuda()) for k, v in
             make_layer_inputs(CFG, seed=30 + i, device="cpu", with_dy=False)["weights"].items()}
            for i in range(L)]


def _hand_chained(cfg, Ws, x, dy, ws):
    xs, saved = [x], []
    for W in Ws:
        y = torch.empty_like(x)
        sv = bpt.alloc_bytes(bpt.bpt_saved_bytes(cfg))
        bpt.bpt_layer_fwd(cfg, W, xs[-1], y, sv, ws)
        xs.append(y)
        saved.append(sv)
    g, grads = dy, [None] * L
    for i in range(L - 1, -1, -1):
        dx = torch.empty_like(x)
        grads[i] = bpt.alloc_grads(Ws[i])
        bpt.bpt_layer_bwd(cfg, Ws[i], xs[i], saved[i], g, dx, grads[i], ws)
        g = dx
    torch.cuda.synchronize()
    assert bpt.bpt_last_device_error() == (bpt.BPT_OK, 0)
    return xs[-1], g, grads


@pytest.mark.parametrize("flags", [bpt.BPT_FLAG_DETERMINISTIC, 0], ids=["fixed order", "default"])
def test_checkpointed_stack_equals_chained_layer_calls(flags):
    cfg = CFG.with_(flags=flags)
    Ws = _weights()
    inp = make_layer_inputs(cfg, seed=40, device="cpu")
    x, dy = inp["x"].cuda(), inp["dy"].cuda()
    ws = bpt.alloc_bytes(max(bpt.bpt_workspace_bytes(cfg, bpt.BPT_PASS_FWD),
                             bpt.bpt_workspace_bytes(cfg, bpt.BPT_PASS_BWD)))
    y_ref, dx_ref, grads_ref = _hand_chained(cfg, Ws, x, dy, ws)

    for k in (1, 2, 3):
        y, st = stack.stack_fwd(cfg, Ws, x, k, ws=ws)
        assert torch.equal(y, y_ref), k
        dx, grads = stack.stack_bwd(cfg, Ws, st, dy, ws=ws)
        torch.cuda.synchronize()
        assert bpt.bpt_last_device_error() == (bpt.BPT_OK, 0)
        assert st.peak_held == stack.held_inputs(L, k)
        if flags & bpt.BPT_FLAG_DETERMINISTIC:
            assert torch.equal(dx, dx_ref), k
            for i in range(L):
                for name, ref_g in grads_ref[i].items():
                    if ref_g is not None:
                        assert torch.equal(grads[i][name], ref_g), (k, i, name)
            continue
        rel = float((dx.float() - dx_ref.float()).norm() / dx_ref.float().norm())
        print(f"k={k} dx rel {rel:.2e}")
        assert rel <= 0.1 * REL_FRO, (k, rel)
        for i in range(L):
            for name, ref_g in grads_ref[i].items():
                if ref_g is None:
                    continue
                got = grads[i][name]
                den = float(ref_g.norm())
                rel = float((got - ref_g).norm()) / den if den > 0 else float((got - ref_g).norm())
                bound = 0.1 * rel_bound(name)
                print(f"k={k} layer {i} d{name} rel {rel:.2e} (bound {bound:.1e})")
                assert rel <= bound, (k, i, name, rel)
