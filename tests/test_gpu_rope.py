"""Rotary position embedding in the layer (rope_base > 0) against the fp64
oracle, which rotates Q and K after their projection and bias: forward and
backward of a grouped-query, head-chunked Llama layer and of a GPT layer with
biases (whose key-bias gradient is no longer zero once keys are rotated), and
the head-chunk call's output and log-sum-exp."""
import pytest
import torch

import blockwise_attention_ffn_gb300 as bpt
from oracle import ref
from tests.gpu_helpers import (LSE_MAX_ABS, LSE_REL_FRO, assert_close, assert_close_grad, device_inputs, run_bwd,
                               run_fwd, to64)
from tests.oracle_helpers import inputs_to_oracle, oracle_cfg
from tests.test_gpu_layer import GPT_SMALL, LLAMA_SMALL

pytestmark = pytest.mark.gpu

ROPE = [LLAMA_SMALL.with_(rope_base=10000.0, name="llama gqa chunked rope"),
        GPT_SMALL.with_(rope_base=10000.0, name="gpt ragged rope")]


@pytest.mark.parametrize("cfg", ROPE, ids=lambda c: c.name)
def test_rope_layer_forward_and_backward(cfg):
    inp, dev = device_inputs(cfg, seed=21)
    y, saved = run_fwd(cfg, dev)
    dx, grads = run_bwd(cfg, dev, saved)
    o = inputs_to_oracle(inp)
    oc = oracle_cfg(cfg)
    assert oc.rope_base == 10000.0
    assert_close(to64(y), ref.layer_forward(o["x"], o["W"], oc), "y")
    dx_ref, g_ref = ref.layer_backward(o["x"], o["W"], o["dy"], oc)
    assert_close(to64(dx), dx_ref, "dx", grad=True)
    for k, v in g_ref.items():
        assert_close_grad(to64(grads[k]), v, f"d{k}", name=k)


def test_rope_headchunk_attention_matches_oracle():
    cfg = ROPE[0]
    inp, dev = device_inputs(cfg, seed=22, with_dy=False)
    H, d = cfg.n_heads, cfg.head_dim
    o = torch.zeros(cfg.b * cfg.s, H * d, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(cfg.b, H, bpt.s_pad(cfg), dtype=torch.float32, device="cuda")
    ws = bpt.alloc_bytes(bpt.bpt_workspace_bytes(cfg, bpt.BPT_PASS_HEADCHUNK))
    bpt.bpt_attn_headchunk(cfg, dev["weights"], dev["x"], o, lse, ws)
    torch.cuda.synchronize()
    assert bpt.bpt_last_device_error() == (bpt.BPT_OK, 0)
    W = inputs_to_oracle(inp)["W"]
    o_ref, lse_ref, _, _, _ = ref.attention_block(to64(inp["x"])[0], W, oracle_cfg(cfg))
    assert_close(to64(o), o_ref, "O")
    assert_close(to64(lse)[0, :, :cfg.s], lse_ref, "LSE", max_abs=LSE_MAX_ABS, rel_fro=LSE_REL_FRO, bf16_out=False)
