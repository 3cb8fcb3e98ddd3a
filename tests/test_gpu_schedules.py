"""The pages' schedule variants change memory and time, not the result.

* Interleaved head-chunk stages ("Untied Ulysses ...", section 4.1 "The GQA
  Scheduling Algorithm"): stage k takes m = U / H_kv query heads of every
  group and all key/value heads stay resident.  The forward's output and
  log-sum-exp are bitwise those of the contiguous stages (every head's
  attention runs on the same values with the same kernel), so the backward,
  which always runs the contiguous stages, is bitwise equal too.
* Save policies ("Blockwise Parallel Transformer ...", the checkpoint
  policies searched for attention): the backward takes Q/K/V (and O) from
  what the forward kept instead of rebuilding them; the rebuilt values are
  bitwise the kept ones, so the gradients are bitwise equal in the
  fixed-order mode.

Both are also checked against the oracle once, so a variant that is equal
to a wrong default would not pass either."""
import pytest
import torch

import blockwise_attention_ffn_gb300 as bpt
from blockwise_attention_ffn_gb300.presets import LayerConfig
from oracle import ref
from tests.gpu_helpers import assert_close, assert_close_grad, device_inputs, run_bwd, run_fwd, to64
from tests.oracle_helpers import inputs_to_oracle, oracle_cfg

pytestmark = pytest.mark.gpu

DET = bpt.BPT_FLAG_DETERMINISTIC
# 16 query heads over 4 key/value heads (G = 4), stages of U = 4: one query
# head of every group per interleaved stage (m = 1); GPT-style with biases
# and rotary embedding so the permuted query bias and the rotation of the
# resident keys are exercised
GQA_M1 = LayerConfig(b=1, s=400, h=1024, n_heads=16, n_kv_heads=4, head_dim=64, ffn_dim=512, head_chunk=4,
                     ffn_block=256, rope_base=10000.0, flags=DET, name="gqa m=1 bias rope")
# 8 over 2 (G = 4), U = 4: two query heads of each group per stage (m = 2);
# Llama-style, batch of two
GQA_M2 = LayerConfig(b=2, s=300, h=512, n_heads=8, n_kv_heads=2, head_dim=64, ffn_dim=768, head_chunk=4,
                     norm=1, act=2, has_bias=0, flags=DET, name="gqa m=2 llama b2")
# d = 128, 32 query heads over 8 (the Llama-8B head layout), U = 8
GQA_D128 = LayerConfig(b=1, s=260, h=4096, n_heads=32, n_kv_heads=8, head_dim=128, ffn_dim=1024, head_chunk=8,
                       norm=1, act=2, has_bias=0, flags=DET, name="gqa d128 llama heads")
INTERLEAVED = [GQA_M1, GQA_M2, GQA_D128]


def _equal_backward(dx0, g0, dx1, g1):
    assert torch.equal(dx0, dx1)
    for k, v in g0.items():
        if v is not None:
            assert torch.equal(v, g1[k]), k


@pytest.mark.parametrize("cfg", INTERLEAVED, ids=lambda c: c.name)
def test_interleaved_stages_equal_contiguous(cfg):
    _, dev = device_inputs(cfg, seed=60)
    y0, s0 = run_fwd(cfg, dev)
    dx0, g0 = run_bwd(cfg, dev, s0)
    il = cfg.with_(stage_order=bpt.BPT_STAGE_INTERLEAVED)
    y1, s1 = run_fwd(il, dev)
    assert torch.equal(y0, y1)
    assert torch.equal(s0, s1)  # the log-sum-exp of every head at its own place
    dx1, g1 = run_bwd(il, dev, s1)
    _equal_backward(dx0, g0, dx1, g1)
    # the head-chunk call too
    H, d = cfg.n_heads, cfg.head_dim
    outs = []
    for c in (cfg, il):
        o = torch.full((cfg.b * cfg.s, H * d), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((cfg.b, H, bpt.s_pad(cfg)), float("nan"), device="cuda")
        ws = bpt.alloc_bytes(bpt.bpt_workspace_bytes(c, bpt.BPT_PASS_HEADCHUNK))
        bpt.bpt_attn_headchunk(c, dev["weights"], dev["x"], o, lse, ws)
        outs.append((o, lse))
    torch.cuda.synchronize()
    assert torch.equal(outs[0][0], outs[1][0])
    assert torch.equal(outs[0][1][:, :, :cfg.s], outs[1][1][:, :, :cfg.s])


def test_interleaved_stages_against_the_oracle():
    cfg = GQA_M1.with_(stage_order=bpt.BPT_STAGE_INTERLEAVED)
    inp, dev = device_inputs(cfg, seed=61)
    y, saved = run_fwd(cfg, dev)
    dx, grads = run_bwd(cfg, dev, saved)
    o = inputs_to_oracle(inp)
    oc = oracle_cfg(cfg)
    assert_close(to64(y), ref.layer_forward(o["x"], o["W"], oc), "y")
    dx_ref, g_ref = ref.layer_backward(o["x"], o["W"], o["dy"], oc)
    assert_close(to64(dx), dx_ref, "dx", grad=True)
    for k, v in g_ref.items():
        assert_close_grad(to64(grads[k]), v, f"d{k}", name=k)


GPT_UNCHUNKED = LayerConfig(b=2, s=640, h=256, n_heads=4, n_kv_heads=4, head_dim=64, ffn_dim=1024, ffn_block=256,
                            flags=DET, name="gpt unchunked b2")


@pytest.mark.parametrize("base", [GPT_UNCHUNKED, GQA_M2, GQA_M1.with_(stage_order=bpt.BPT_STAGE_INTERLEAVED)],
                         ids=["gpt unchunked", "llama chunked", "interleaved rope"])
def test_save_policies_give_the_same_result(base):
    _, dev = device_inputs(base, seed=62)
    y0, s0 = run_fwd(base, dev)
    dx0, g0 = run_bwd(base, dev, s0)
    lse_bytes = bpt.bpt_saved_bytes(base)
    rows, H, Hk, d = base.b * base.s, base.n_heads, base.n_kv_heads, base.head_dim

    def up(n):
        return (n + 255) // 256 * 256
    for pol in (bpt.BPT_SAVE_PROJECTIONS, bpt.BPT_SAVE_ATTN_OUT):
        c = base.with_(save_policy=pol)
        want = up(lse_bytes) + up(rows * (H + 2 * Hk) * d * 2) + (up(rows * H * d * 2) if pol == 2 else 0)
        assert bpt.bpt_saved_bytes(c) == want
        # the backward needs less workspace when the forward kept more
        assert bpt.bpt_workspace_bytes(c, bpt.BPT_PASS_BWD) < bpt.bpt_workspace_bytes(base, bpt.BPT_PASS_BWD)
        y1, s1 = run_fwd(c, dev)
        assert torch.equal(y0, y1)
        assert torch.equal(s0, s1[:lse_bytes])
        dx1, g1 = run_bwd(c, dev, s1)
        _equal_backward(dx0, g0, dx1, g1)


def test_save_policy_kept_values_are_the_layer_s():
    """What the forward keeps is what the layer computes: the kept Q, K, V
    and O equal the oracle's (all heads; O before the output projection)."""
    cfg = GQA_M2.with_(save_policy=bpt.BPT_SAVE_ATTN_OUT, b=1)
    inp, dev = device_inputs(cfg, seed=63)
    _, saved = run_fwd(cfg, dev)
    rows, H, Hk, d = cfg.s, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim
    off = (bpt.bpt_saved_bytes(cfg.with_(save_policy=0)) + 255) // 256 * 256
    qkv_bytes = rows * (H + 2 * Hk) * d * 2
    qkv = to64(saved[off:off + qkv_bytes].view(torch.bfloat16).view(rows, (H + 2 * Hk) * d))
    off += (qkv_bytes + 255) // 256 * 256
    o_kept = to64(saved[off:off + rows * H * d * 2].view(torch.bfloat16).view(rows, H * d))
    o = inputs_to_oracle(inp)
    _, caches = ref.layer_forward(o["x"], o["W"], oracle_cfg(cfg), keep=True)
    c = caches[0]
    assert_close(qkv[:, :H * d], c["q"].reshape(rows, H * d), "kept Q")
    assert_close(qkv[:, H * d:(H + Hk) * d], c["k"].reshape(rows, Hk * d), "kept K")
    assert_close(qkv[:, (H + Hk) * d:], c["v"].reshape(rows, Hk * d), "kept V")
    assert_close(o_kept, c["o"], "kept O")


def test_interleaved_needs_whole_groups_per_stage():
    """U must be a multiple of H_kv (one or more query heads of every group
    per stage) for the interleaved order."""
    bad = GQA_M2.with_(n_heads=16, n_kv_heads=8, h=1024, head_chunk=4, stage_order=bpt.BPT_STAGE_INTERLEAVED)
    assert bpt.bpt_workspace_bytes(bad, bpt.BPT_PASS_FWD) == 0
    assert bpt.bpt_workspace_bytes(bad.with_(stage_order=0), bpt.BPT_PASS_FWD) > 0
