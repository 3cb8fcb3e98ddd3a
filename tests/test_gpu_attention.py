"""Attention kernels (forward and backward) against the fp64 oracle, element by
element, on shapes that span several tiles, ragged tails, a single row,
grouped-query heads, both masks and every supported head dimension."""
import numpy as np
import pytest
import torch

import blockwise_attention_ffn_gb300 as bpt
from blockwise_attention_ffn_gb300.presets import LayerConfig
from oracle import ref
from tests.gpu_helpers import LSE_MAX_ABS, LSE_REL_FRO, assert_close, to64

pytestmark = pytest.mark.gpu

SHAPES = [
    # b, s, H, Hkv, d, causal
    (1, 128, 2, 2, 64, 1),
    (1, 300, 2, 1, 80, 1),
    (2, 200, 2, 2, 128, 0),
    (1, 513, 4, 2, 128, 1),
    (1, 1, 1, 1, 64, 1),
    (1, 384, 2, 2, 96, 1),
    (1, 260, 2, 2, 112, 0),
    (1, 640, 4, 1, 80, 0),
]


def _cfg(b, s, H, Hkv, d, causal):
    return LayerConfig(b=b, s=s, h=H * d, n_heads=H, n_kv_heads=Hkv, head_dim=d, ffn_dim=64,
                       causal=causal)


def _qkv(b, s, H, Hkv, d, seed, scale=1.0):
    """q, k, v ~ N(0, scale^2): in the layer workloads the projections of the
    normalised input by N(0, 0.02^2) weights have unit scale at h ~ 2500."""
    g = torch.Generator().manual_seed(seed)
    qkv = torch.randn(b * s, (H + 2 * Hkv) * d, generator=g) * scale
    return qkv.to(torch.bfloat16)


def _split(qkv64, b, s, H, Hkv, d):
    t = qkv64.reshape(b, s, H + 2 * Hkv, d)
    return t[:, :, :H], t[:, :, H:H + Hkv], t[:, :, H + Hkv:]


@pytest.mark.parametrize("shape", SHAPES)
def test_attention_forward(shape):
    b, s, H, Hkv, d, causal = shape
    cfg = _cfg(*shape)
    qkv = _qkv(b, s, H, Hkv, d, seed=s + d, scale=1.5)  # peakier softmax than the workloads
    o = torch.zeros(b * s, H * d, dtype=torch.bfloat16, device="cuda")
    sp = bpt.s_pad(cfg)
    lse = torch.zeros(b, H, sp, dtype=torch.float32, device="cuda")
    bpt.bpt_attention_fwd(cfg, qkv.cuda(), o, lse)
    torch.cuda.synchronize()
    assert bpt.bpt_last_device_error()[0] == bpt.BPT_OK
    q, k, v = _split(to64(qkv), b, s, H, Hkv, d)
    G = H // Hkv
    o_ref = np.empty((b, s, H, d))
    lse_ref = np.empty((b, H, s))
    for bi in range(b):
        for n in range(H):
            o_ref[bi, :, n], lse_ref[bi, n] = ref.attention_head(q[bi, :, n], k[bi, :, n // G],
                                                                 v[bi, :, n // G], bool(causal))
    assert_close(to64(o).reshape(b, s, H, d), o_ref, "O")
    assert_close(to64(lse)[:, :, :s], lse_ref, "LSE", max_abs=LSE_MAX_ABS, rel_fro=LSE_REL_FRO, bf16_out=False)


@pytest.mark.parametrize("shape", SHAPES)
def test_attention_backward(shape):
    b, s, H, Hkv, d, causal = shape
    cfg = _cfg(*shape)
    qkv = _qkv(b, s, H, Hkv, d, seed=2 * s + d)
    g = torch.Generator().manual_seed(7 + s)
    dout = torch.randn(b * s, H * d, generator=g).to(torch.bfloat16)
    qkv_d = qkv.cuda()
    o = torch.zeros(b * s, H * d, dtype=torch.bfloat16, device="cuda")
    sp = bpt.s_pad(cfg)
    lse = torch.zeros(b, H, sp, dtype=torch.float32, device="cuda")
    bpt.bpt_attention_fwd(cfg, qkv_d, o, lse)
    dqkv = torch.full_like(qkv_d, float("nan"))
    ws = bpt.alloc_bytes(bpt.bpt_attention_bwd_workspace_bytes(cfg))
    bpt.bpt_attention_bwd(cfg, qkv_d, o, lse, dout.cuda(), dqkv, ws)
    torch.cuda.synchronize()
    assert bpt.bpt_last_device_error()[0] == bpt.BPT_OK
    q, k, v = _split(to64(qkv), b, s, H, Hkv, d)
    do = to64(dout).reshape(b, s, H, d)
    G = H // Hkv
    dq = np.zeros((b, s, H, d))
    dk = np.zeros((b, s, Hkv, d))
    dv = np.zeros((b, s, Hkv, d))
    for bi in range(b):
        for n in range(H):
            a_, b_, c_ = ref.attention_head_backward(q[bi, :, n], k[bi, :, n // G], v[bi, :, n // G],
                                                     do[bi, :, n], bool(causal))
            dq[bi, :, n] += a_
            dk[bi, :, n // G] += b_
            dv[bi, :, n // G] += c_
    got = to64(dqkv).reshape(b, s, H + 2 * Hkv, d)
    assert_close(got[:, :, :H], dq, "dQ", grad=True)
    assert_close(got[:, :, H:H + Hkv], dk, "dK", grad=True)
    assert_close(got[:, :, H + Hkv:], dv, "dV", grad=True)


def test_identical_keys_give_prefix_mean():
    """Closed form on the GPU: equal keys make causal attention the running
    mean of the values; row 0 is V_0."""
    b, s, H, Hkv, d = 1, 300, 2, 2, 64
    cfg = _cfg(b, s, H, Hkv, d, 1)
    qkv = _qkv(b, s, H, Hkv, d, seed=5).float()
    qkv[:, H * d:(H + Hkv) * d] = qkv[0:1, H * d:(H + Hkv) * d]
    qkv = qkv.to(torch.bfloat16)
    o = torch.zeros(b * s, H * d, dtype=torch.bfloat16, device="cuda")
    bpt.bpt_attention_fwd(cfg, qkv.cuda(), o, None)
    torch.cuda.synchronize()
    v = to64(qkv)[:, (H + Hkv) * d:].reshape(s, Hkv, d)
    want = np.cumsum(v, 0) / np.arange(1, s + 1)[:, None, None]
    got = to64(o).reshape(s, H, d)
    assert_close(got, want, "prefix mean")
    assert np.max(np.abs(got[0] - v[0])) <= 4e-3  # bf16 rounding of V_0 itself only


@pytest.mark.parametrize("shape", [(1, 640, 4, 1, 80, 0), (2, 200, 2, 2, 128, 0)])
def test_noncausal_key_order_does_not_matter(shape):
    """Without the mask the keys form a set: permuting the key/value rows
    (across tiles and within them) changes only the order of the online
    softmax's blocks, not the result (GPU against GPU, each within the
    acceptance bound of the exact value)."""
    b, s, H, Hkv, d, causal = shape
    cfg = _cfg(*shape)
    qkv = _qkv(b, s, H, Hkv, d, seed=s + d + 1, scale=1.5)
    perm = torch.randperm(s, generator=torch.Generator().manual_seed(s))
    t = qkv.reshape(b, s, H + 2 * Hkv, d).clone()
    t[:, :, H:] = t[:, perm, H:]
    qkv_p = t.reshape(b * s, -1)
    outs = []
    for x in (qkv, qkv_p):
        o = torch.zeros(b * s, H * d, dtype=torch.bfloat16, device="cuda")
        lse = torch.zeros(b, H, bpt.s_pad(cfg), dtype=torch.float32, device="cuda")
        bpt.bpt_attention_fwd(cfg, x.cuda(), o, lse)
        torch.cuda.synchronize()
        assert bpt.bpt_last_device_error()[0] == bpt.BPT_OK
        outs.append((to64(o), to64(lse)[:, :, :s]))
    assert_close(outs[1][0], outs[0][0], "O, keys permuted")
    assert_close(outs[1][1], outs[0][1], "LSE, keys permuted", max_abs=2 * LSE_MAX_ABS, rel_fro=2 * LSE_REL_FRO,
                 bf16_out=False)
