"""The row-sampled forward and sparse-dy backward equal the dense oracle."""
import numpy as np
import pytest

from oracle import ref, sampled
from oracle.ref import LayerCfg
from tests.oracle_helpers import rand_layer


@pytest.mark.parametrize("cfg", [
    LayerCfg(s=80, h=32, n_heads=4, n_kv_heads=4, head_dim=8, ffn_dim=64),
    LayerCfg(s=64, h=32, n_heads=4, n_kv_heads=2, head_dim=8, ffn_dim=48, norm=1, act=2,
             has_bias=False),
    LayerCfg(s=50, h=32, n_heads=4, n_kv_heads=4, head_dim=8, ffn_dim=64, causal=False, act=1),
    LayerCfg(s=72, h=32, n_heads=4, n_kv_heads=2, head_dim=8, ffn_dim=48, norm=1, act=2,
             has_bias=False, rope_base=500000.0),
    LayerCfg(s=40, h=32, n_heads=4, n_kv_heads=4, head_dim=8, ffn_dim=64, rope_base=10.0),
])
def test_sampled_forward_and_sparse_backward(cfg):
    x, W, dy = rand_layer(cfg, seed=12)
    rows = np.array([0, 3, 17, cfg.s - 1])
    y = ref.layer_forward(x, W, cfg)
    yr = sampled.forward_rows(x, W, cfg, rows)
    assert np.max(np.abs(yr - y[0, rows])) < 1e-12

    dys = np.zeros_like(dy)
    dys[0, rows] = dy[0, rows]
    dx, g = ref.layer_backward(x, W, dys, cfg)
    dx2, g2 = sampled.backward_sparse_dy(x, W, dy[0, rows], rows, cfg)
    assert np.max(np.abs(dx2 - dx[0])) < 1e-11
    for k in g:
        assert np.max(np.abs(g2[k] - g[k])) < 1e-11 * max(1, np.abs(g[k]).max()), k
