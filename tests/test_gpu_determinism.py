"""The fixed-order mode (BPT_FLAG_DETERMINISTIC) and the debug checks
(BPT_FLAG_DEBUG_CHECKS) on the GPU.

With the fixed order, two backward calls on the same inputs give bitwise
equal results: the attention backward has one MMA-issuing thread per CTA, the
weight-gradient products are not split along K, and the bias and norm
gradients are added in block order.  The layers below are long enough
(s >= 2048) that the default mode would split the weight-gradient products
and take its bias and norm sums with atomics, so every one of the three
order-dependent sums is exercised.  The fixed-order results must still meet
the oracle's acceptance bounds."""
import ctypes

import numpy as np
import pytest
import torch

import blockwise_attention_ffn_gb300 as bpt
from blockwise_attention_ffn_gb300.presets import LayerConfig
from oracle import ref
from tests.gpu_helpers import assert_close, assert_close_grad, device_inputs, run_bwd, run_fwd, to64
from tests.oracle_helpers import inputs_to_oracle, oracle_cfg

pytestmark = pytest.mark.gpu

DET = bpt.BPT_FLAG_DETERMINISTIC
GPT_LONG = LayerConfig(b=1, s=2304, h=256, n_heads=4, n_kv_heads=4, head_dim=64, ffn_dim=1024,
                       ffn_block=768, name="gpt s2304")
LLAMA_LONG = LayerConfig(b=1, s=2176, h=512, n_heads=8, n_kv_heads=2, head_dim=128, ffn_dim=768,
                         head_chunk=4, norm=1, act=2, has_bias=0, name="llama gqa chunked s2176")
GPT_D80 = LayerConfig(b=2, s=1100, h=320, n_heads=4, n_kv_heads=4, head_dim=80, ffn_dim=640,
                      ffn_block=512, name="gpt d80 b2")
LAYERS = [GPT_LONG, LLAMA_LONG, GPT_D80]


@pytest.mark.parametrize("base", LAYERS, ids=lambda c: c.name)
def test_fixed_order_backward_is_bitwise_repeatable_and_within_tolerance(base):
    cfg = base.with_(flags=DET)
    inp, dev = device_inputs(cfg, seed=21)
    y, saved = run_fwd(cfg, dev)
    dx0, g0 = run_bwd(cfg, dev, saved)
    dx1, g1 = run_bwd(cfg, dev, saved)
    assert torch.equal(dx0, dx1)
    for k, v in g0.items():
        if v is not None:
            assert torch.equal(v, g1[k]), k
    o = inputs_to_oracle(inp)
    oc = oracle_cfg(cfg)
    assert_close(to64(y), ref.layer_forward(o["x"], o["W"], oc), "y")
    dx_ref, g_ref = ref.layer_backward(o["x"], o["W"], o["dy"], oc)
    assert_close(to64(dx0), dx_ref, "dx", grad=True)
    for k, v in g_ref.items():
        assert_close_grad(to64(g0[k]), v, f"d{k}", name=k)


@pytest.mark.parametrize("d,H,Hkv,s,causal", [(64, 4, 2, 1000, 1), (80, 2, 2, 700, 1), (128, 4, 1, 520, 0),
                                              (96, 2, 2, 384, 1), (112, 2, 1, 300, 1)])
def test_fixed_order_attention_backward_is_bitwise_repeatable(d, H, Hkv, s, causal):
    cfg = LayerConfig(b=1, s=s, h=H * d, n_heads=H, n_kv_heads=Hkv, head_dim=d, ffn_dim=64, causal=causal,
                      flags=DET)
    g = torch.Generator().manual_seed(d + s)
    qkv = torch.randn(s, (H + 2 * Hkv) * d, generator=g).to(torch.bfloat16).cuda()
    dout = torch.randn(s, H * d, generator=g).to(torch.bfloat16).cuda()
    o = torch.empty(s, H * d, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(1, H, bpt.s_pad(cfg), dtype=torch.float32, device="cuda")
    bpt.bpt_attention_fwd(cfg, qkv, o, lse)
    ws = bpt.alloc_bytes(bpt.bpt_attention_bwd_workspace_bytes(cfg))
    outs = []
    for _ in range(3):
        dq = torch.full_like(qkv, float("nan"))
        bpt.bpt_attention_bwd(cfg, qkv, o, lse, dout, dq, ws)
        outs.append(dq)
    # the default mode computes the same thing up to the order of its sums
    dflt = torch.empty_like(qkv)
    bpt.bpt_attention_bwd(cfg.with_(flags=0), qkv, o, lse, dout, dflt, ws)
    torch.cuda.synchronize()
    assert bpt.bpt_last_device_error() == (bpt.BPT_OK, 0)
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    assert_close(to64(dflt), to64(outs[0]), "default vs fixed order", max_abs=1e30, rel_fro=1e-3, bf16_out=False)


def _segment_of(t):
    """(base, size) of the caching allocator's segment (one cudaMalloc) that
    holds tensor t."""
    p = t.data_ptr()
    for seg in torch.cuda.memory_snapshot():
        if seg["address"] <= p < seg["address"] + seg["total_size"]:
            return seg["address"], seg["total_size"]
    raise AssertionError("tensor not found in the allocator's segments")


def test_device_range_check():
    t = torch.empty(3 << 20, dtype=torch.uint8, device="cuda")
    base, size = _segment_of(t)
    assert bpt.bpt_check_device_range(t.data_ptr(), t.numel()) == bpt.BPT_OK
    assert bpt.bpt_check_device_range(base, size) == bpt.BPT_OK
    assert bpt.bpt_check_device_range(base + size - 16, 16) == bpt.BPT_OK
    assert bpt.bpt_check_device_range(base + size - 16, 32) == bpt.BPT_EINVAL
    host = torch.empty(1 << 16, dtype=torch.uint8).pin_memory()
    assert bpt.bpt_check_device_range(host.data_ptr(), 16) == bpt.BPT_EINVAL
    a = np.zeros(1 << 16, np.uint8)
    assert bpt.bpt_check_device_range(a.ctypes.data, 16) == bpt.BPT_EINVAL


def test_debug_checks_pass_good_calls_and_refuse_host_buffers():
    base = GPT_LONG.with_(s=640, ffn_block=256)
    det = base.with_(flags=DET)
    dbg = base.with_(flags=DET | bpt.BPT_FLAG_DEBUG_CHECKS)
    _, dev = device_inputs(base, seed=22)
    y0, s0 = run_fwd(det, dev)
    dx0, g0 = run_bwd(det, dev, s0)
    y1, s1 = run_fwd(dbg, dev)
    dx1, g1 = run_bwd(dbg, dev, s1)
    assert torch.equal(y0, y1) and torch.equal(dx0, dx1)
    for k, v in g0.items():
        if v is not None:
            assert torch.equal(v, g1[k]), k
    # pinned host memory as the input: refused before anything is launched
    x_host = dev["x"].cpu().pin_memory()
    y = torch.empty_like(dev["x"])
    ws = bpt.alloc_bytes(bpt.bpt_workspace_bytes(dbg, bpt.BPT_PASS_FWD))
    with pytest.raises(bpt.BptError) as e:
        bpt.bpt_layer_fwd(dbg, dev["weights"], x_host, y, None, ws)
    assert e.value.status == bpt.BPT_EINVAL
    # a workspace that ends before the bytes the call needs (the end of its
    # allocation inside the claimed size): refused too
    need = bpt.bpt_workspace_bytes(dbg, bpt.BPT_PASS_FWD)
    sbase, ssize = _segment_of(ws)
    tail = sbase + ssize - need // 2
    tail -= tail % 256
    # the call below is made only once the checker itself has refused this
    # range, so nothing runs past the allocation
    assert bpt.bpt_check_device_range(tail, need) == bpt.BPT_EINVAL
    c = bpt.make_config(dbg)
    w = bpt.make_weights(dev["weights"])
    rc = bpt.lib().bpt_layer_fwd(ctypes.byref(c), ctypes.byref(w), ctypes.c_void_p(dev["x"].data_ptr()),
                                 ctypes.c_void_p(y.data_ptr()), None, ctypes.c_void_p(tail), need,
                                 ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == bpt.BPT_EINVAL
    torch.cuda.synchronize()
    assert bpt.bpt_last_device_error() == (bpt.BPT_OK, 0)
