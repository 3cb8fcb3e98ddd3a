"""The oracle against an independent library implementation: PyTorch's own
fp64 CPU ops (layer_norm / rms_norm, linear, scaled_dot_product_attention,
gelu, silu) and its autograd.  Same definition, different code: a wrong scale,
mask, transposition or gradient rule in the oracle fails here."""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import ref
from oracle.ref import LayerCfg
from tests.oracle_helpers import rand_layer


def _torch_layer(x, W, cfg: LayerCfg):
    H, Hk, d = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim

    def norm(t, w, b):
        if cfg.norm == 0:
            return F.layer_norm(t, (cfg.h,), w, b, cfg.norm_eps)
        ms = (t * t).mean(-1, keepdim=True)
        return t * torch.rsqrt(ms + cfg.norm_eps) * w

    b_, s_ = x.shape[0], x.shape[1]
    xn = norm(x, W["ln1_w"], W.get("ln1_b"))
    q = F.linear(xn, W["wq"], W.get("bq")).view(b_, s_, H, d).transpose(1, 2)
    k = F.linear(xn, W["wk"], W.get("bk")).view(b_, s_, Hk, d).transpose(1, 2)
    v = F.linear(xn, W["wv"], W.get("bv")).view(b_, s_, Hk, d).transpose(1, 2)
    G = H // Hk
    k = k.repeat_interleave(G, dim=1)
    v = v.repeat_interleave(G, dim=1)
    o = F.scaled_dot_product_attention(q, k, v, is_causal=cfg.causal)
    o = o.transpose(1, 2).reshape(b_, s_, H * d)
    x1 = x + F.linear(o, W["wo"], W.get("bo"))
    x1n = norm(x1, W["ln2_w"], W.get("ln2_b"))
    if cfg.act == 2:
        a = F.silu(F.linear(x1n, W["w1"])) * F.linear(x1n, W["w3"])
    else:
        a = F.gelu(F.linear(x1n, W["w1"], W.get("b1")),
                   approximate="none" if cfg.act == 0 else "tanh")
    return x1 + F.linear(a, W["w2"], W.get("b2"))


CFGS = [
    LayerCfg(s=70, h=32, n_heads=4, n_kv_heads=4, head_dim=8, ffn_dim=64),
    LayerCfg(s=45, h=32, n_heads=4, n_kv_heads=4, head_dim=8, ffn_dim=64, act=1, causal=False),
    LayerCfg(s=66, h=64, n_heads=8, n_kv_heads=2, head_dim=8, ffn_dim=96, norm=1, act=2,
             has_bias=False, b=2),
]


@pytest.mark.parametrize("cfg", CFGS)
def test_forward_and_backward_match_torch_fp64(cfg):
    x, W, dy = rand_layer(cfg, seed=11)
    y = ref.layer_forward(x, W, cfg)
    dx, grads = ref.layer_backward(x, W, dy, cfg)

    tx = torch.tensor(x, dtype=torch.float64, requires_grad=True)
    tW = {k: torch.tensor(v, dtype=torch.float64, requires_grad=True) for k, v in W.items()}
    ty = _torch_layer(tx, tW, cfg)
    assert np.max(np.abs(ty.detach().numpy() - y)) < 1e-11
    ty.backward(torch.tensor(dy))
    assert np.max(np.abs(tx.grad.numpy() - dx)) < 1e-10
    for k, v in tW.items():
        assert np.max(np.abs(v.grad.numpy() - grads[k])) < 1e-9 * max(1, np.abs(grads[k]).max()), k
