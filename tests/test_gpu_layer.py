"""The whole layer (forward and recompute backward) against the fp64 oracle,
element by element, on seeded inputs of both layer variants: GPT (LayerNorm,
GeLU, biases) and Llama (RMSNorm, SwiGLU, no biases, grouped-query attention,
head-chunked)."""
import numpy as np
import pytest
import torch

import blockwise_attention_ffn_gb300 as bpt
from blockwise_attention_ffn_gb300.presets import C1, LayerConfig
from oracle import ref
from tests.gpu_helpers import (LSE_MAX_ABS, LSE_REL_FRO, assert_close, assert_close_grad, device_inputs,
                               half_ulp_bf16, run_bwd, run_fwd, to64)
from tests.oracle_helpers import inputs_to_oracle, oracle_cfg

pytestmark = pytest.mark.gpu

GPT_SMALL = LayerConfig(b=1, s=300, h=256, n_heads=4, n_kv_heads=4, head_dim=64, ffn_dim=1024,
                        ffn_block=128, name="gpt ragged")
GPT_D80 = LayerConfig(b=1, s=520, h=320, n_heads=4, n_kv_heads=4, head_dim=80, ffn_dim=640,
                      ffn_block=256, act=1, name="gpt d80 tanh")
LLAMA_SMALL = LayerConfig(b=1, s=384, h=512, n_heads=8, n_kv_heads=2, head_dim=64, ffn_dim=768,
                          head_chunk=4, norm=1, act=2, has_bias=0, name="llama gqa chunked")
GPT_B2 = LayerConfig(b=2, s=200, h=256, n_heads=2, n_kv_heads=2, head_dim=128, ffn_dim=512,
                     causal=0, name="gpt b2 noncausal")

# enough tiles (fc1: 16 x 32 = 512 per FFN block) that every persistent GEMM
# CTA walks several and reuses both of its TMEM accumulators; ragged in M and N
GPT_MANY_TILES = LayerConfig(b=1, s=2500, h=384, n_heads=6, n_kv_heads=6, head_dim=64, ffn_dim=8192,
                             name="gpt many tiles")

# model width above 4096 (attention narrower than the model): the norms'
# unstaged backward kernel, which takes the rows the shared-memory-staged one
# does not, and N = 4352 products; only the tensors of WIDE_TENSORS have an
# emulated bf16 floor above 5e-3 at these shapes (at most 7.1e-3)
GPT_WIDE = LayerConfig(b=1, s=160, h=4352, n_heads=4, n_kv_heads=4, head_dim=64, ffn_dim=256, ffn_block=128,
                       name="gpt h4352")
LLAMA_WIDE = LayerConfig(b=1, s=160, h=4352, n_heads=4, n_kv_heads=2, head_dim=64, ffn_dim=256, ffn_block=128,
                         norm=1, act=2, has_bias=0, name="llama h4352")

LAYERS = [GPT_SMALL, GPT_D80, LLAMA_SMALL, GPT_B2, GPT_MANY_TILES, GPT_WIDE, LLAMA_WIDE]


@pytest.mark.parametrize("cfg", LAYERS, ids=lambda c: c.name)
def test_layer_forward(cfg):
    inp, dev = device_inputs(cfg, seed=11)
    y, _ = run_fwd(cfg, dev)
    o = inputs_to_oracle(inp)
    y_ref = ref.layer_forward(o["x"], o["W"], oracle_cfg(cfg))
    assert_close(to64(y), y_ref, "y")


@pytest.mark.parametrize("cfg", LAYERS, ids=lambda c: c.name)
def test_layer_backward(cfg):
    inp, dev = device_inputs(cfg, seed=12)
    _, saved = run_fwd(cfg, dev)
    dx, grads = run_bwd(cfg, dev, saved)
    o = inputs_to_oracle(inp)
    dx_ref, g_ref = ref.layer_backward(o["x"], o["W"], o["dy"], oracle_cfg(cfg))
    assert_close(to64(dx), dx_ref, "dx", grad=True)
    for k, v in g_ref.items():
        assert_close_grad(to64(grads[k]), v, f"d{k}", name=k)


def test_c1_forward_full_oracle():
    inp, dev = device_inputs(C1, seed=C1.seed)
    y, _ = run_fwd(C1, dev)
    o = inputs_to_oracle(inp)
    assert_close(to64(y), ref.layer_forward(o["x"], o["W"], oracle_cfg(C1)), "y")


def test_headchunk_attention_matches_oracle():
    cfg = LLAMA_SMALL
    inp, dev = device_inputs(cfg, seed=13, with_dy=False)
    xn = dev["x"]  # any normalised-input stand-in: the call projects whatever it gets
    H, d = cfg.n_heads, cfg.head_dim
    o = torch.zeros(cfg.b * cfg.s, H * d, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(cfg.b, H, bpt.s_pad(cfg), dtype=torch.float32, device="cuda")
    ws = bpt.alloc_bytes(bpt.bpt_workspace_bytes(cfg, bpt.BPT_PASS_HEADCHUNK))
    bpt.bpt_attn_headchunk(cfg, dev["weights"], xn, o, lse, ws)
    torch.cuda.synchronize()
    W = inputs_to_oracle(inp)["W"]
    o_ref, lse_ref, _, _, _ = ref.attention_block(to64(inp["x"])[0], W, oracle_cfg(cfg))
    assert_close(to64(o), o_ref, "O")
    assert_close(to64(lse)[0, :, :cfg.s], lse_ref, "LSE", max_abs=LSE_MAX_ABS, rel_fro=LSE_REL_FRO, bf16_out=False)


@pytest.mark.parametrize("base,variant", [
    (LLAMA_SMALL, dict(head_chunk=8)), (LLAMA_SMALL, dict(ffn_block=384)),
    (LLAMA_SMALL, dict(ffn_block=128)), (GPT_SMALL, dict(head_chunk=1)),
    (GPT_SMALL, dict(head_chunk=2)), (GPT_SMALL, dict(ffn_block=256, q_block=256, kv_block=256)),
    (LLAMA_SMALL, dict(flags=bpt.BPT_FLAG_ONE_STREAM)),
], ids=lambda v: v.name if hasattr(v, "name") else str(v))
def test_schedule_invariance(base, variant):
    """Head chunk U, FFN block, attention block sizes and running on one
    stream change the schedule, not the result."""
    _, dev = device_inputs(base, seed=14)
    y0, s0 = run_fwd(base, dev)
    dx0, g0 = run_bwd(base, dev, s0)
    cfg = base.with_(**variant)
    y1, s1 = run_fwd(cfg, dev)
    dx1, g1 = run_bwd(cfg, dev, s1)
    assert torch.equal(y0, y1)
    # dx is stored in bf16 after fp32 sums whose order depends on the head
    # chunk (the input-gradient product accumulates stage by stage), so an
    # element may round to the neighbouring bf16 value: one ulp, no more
    d0, d1 = to64(dx0), to64(dx1)
    assert np.all(np.abs(d1 - d0) <= 2 * half_ulp_bf16(d0) + 1e-3), float(np.max(np.abs(d1 - d0)))
    assert_close(d1, d0, "dx", max_abs=1e30, rel_fro=1e-4, bf16_out=False)
    for k in g0:
        if g0[k] is not None:
            assert_close(to64(g1[k]), to64(g0[k]), k, max_abs=1e-3 * max(1, float(g0[k].abs().max())),
                         rel_fro=1e-4, bf16_out=False)


def test_accumulate_flag_adds_to_existing_gradients():
    cfg = GPT_SMALL
    _, dev = device_inputs(cfg, seed=15)
    _, saved = run_fwd(cfg, dev)
    _, g0 = run_bwd(cfg, dev, saved)
    acc = cfg.with_(flags=bpt.BPT_FLAG_ACCUM_GRADS)
    dx = torch.empty_like(dev["x"])
    grads = {k: (None if v is None else v.clone()) for k, v in g0.items()}
    ws = bpt.alloc_bytes(bpt.bpt_workspace_bytes(acc, bpt.BPT_PASS_BWD))
    bpt.bpt_layer_bwd(acc, dev["weights"], dev["x"], saved, dev["dy"], dx, grads, ws)
    torch.cuda.synchronize()
    for k, v in g0.items():
        if v is not None:
            assert_close(to64(grads[k]), 2 * to64(v), k, max_abs=1e-3 * max(1, float(v.abs().max())),
                         rel_fro=1e-5, bf16_out=False)


def causal_prefix_mean(v, n_heads, n_kv_heads, d):
    """O of uniform causal attention: row i of query head n is the mean of
    rows 0..i of its key/value head n // G (v: [s, H_kv * d])."""
    g = n_heads // n_kv_heads
    cum = np.cumsum(v, axis=0) / np.arange(1, v.shape[0] + 1)[:, None]
    return np.concatenate([cum[:, (n // g) * d:(n // g + 1) * d] for n in range(n_heads)], axis=1)


def test_zero_query_projection_gives_uniform_causal_attention():
    """Wq = 0 makes every score zero, so each query attends uniformly to its
    causal prefix: O_i = mean of V_0..V_i and LSE_i = ln(i + 1).  A closed
    form that needs no oracle; grouped-query heads and head chunks included."""
    cfg = LLAMA_SMALL
    inp, dev = device_inputs(cfg, seed=16, with_dy=False)
    dev["weights"]["wq"].zero_()
    H, d = cfg.n_heads, cfg.head_dim
    o = torch.zeros(cfg.b * cfg.s, H * d, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(cfg.b, H, bpt.s_pad(cfg), dtype=torch.float32, device="cuda")
    ws = bpt.alloc_bytes(bpt.bpt_workspace_bytes(cfg, bpt.BPT_PASS_HEADCHUNK))
    bpt.bpt_attn_headchunk(cfg, dev["weights"], dev["x"], o, lse, ws)
    torch.cuda.synchronize()
    v = to64(inp["x"])[0] @ to64(inp["weights"]["wv"]).T
    assert_close(to64(o), causal_prefix_mean(v, H, cfg.n_kv_heads, d), "O")
    want_lse = np.tile(np.log(np.arange(1, cfg.s + 1, dtype=np.float64)), (H, 1))
    assert_close(to64(lse)[0, :, :cfg.s], want_lse, "LSE", max_abs=LSE_MAX_ABS, rel_fro=LSE_REL_FRO,
                 bf16_out=False)


def test_zero_output_projection_and_fc1_leave_residual_plus_b2():
    """Wo = bo = 0 removes the attention branch and W1 = b1 = 0 makes the
    FFN GeLU(0) W2^T + b2 = b2, so y = x + b2: the fp32 residual sum rounded
    once to bf16.  Every other element of the layer still runs."""
    cfg = GPT_SMALL
    inp, dev = device_inputs(cfg, seed=17, with_dy=False)
    for k in ("wo", "bo", "w1", "b1"):
        dev["weights"][k].zero_()
    y, _ = run_fwd(cfg, dev)
    want = to64(inp["x"]) + to64(inp["weights"]["b2"])
    assert_close(to64(y), want, "y", max_abs=1e-6)
