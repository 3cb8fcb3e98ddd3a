"""Helpers for the oracle tests: fp64 random layers (NumPy) and conversion of the
seeded bf16 inputs to the oracle's fp64 arrays."""
from __future__ import annotations

import numpy as np

from oracle.ref import LayerCfg, weight_shapes


def rand_layer(cfg: LayerCfg, seed=0, wscale=0.3):
    rng = np.random.default_rng(seed)
    W = {}
    for name, shp in weight_shapes(cfg).items():
        t = rng.standard_normal(shp) * wscale
        if name in ("ln1_w", "ln2_w"):
            t = 1.0 + 0.2 * rng.standard_normal(shp)
        W[name] = t
    x = rng.standard_normal((cfg.b, cfg.s, cfg.h))
    dy = rng.standard_normal((cfg.b, cfg.s, cfg.h))
    return x, W, dy


def to_np64(t):
    return None if t is None else t.detach().to("cpu").double().numpy()


def inputs_to_oracle(inp):
    W = {k: to_np64(v) for k, v in inp["weights"].items() if v is not None}
    out = {"x": to_np64(inp["x"]), "W": W}
    if "dy" in inp:
        out["dy"] = to_np64(inp["dy"])
    return out


def oracle_cfg(c) -> LayerCfg:
    """LayerCfg from any object with the library config's field names."""
    return LayerCfg(s=c.s, h=c.h, n_heads=c.n_heads, n_kv_heads=c.n_kv_heads,
                    head_dim=c.head_dim, ffn_dim=c.ffn_dim, b=c.b, causal=bool(c.causal),
                    norm=c.norm, act=c.act, has_bias=bool(c.has_bias), norm_eps=c.norm_eps,
                    rope_base=float(getattr(c, "rope_base", 0.0)))
