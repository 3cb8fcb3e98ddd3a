"""Seeded synthetic inputs shared by the tests, the bench and the smoke check.

This module holds no arithmetic of the layer: it only draws random numbers of
the right shapes.  The recipe follows the workloads the pages describe
(synthetic sequences of GPT- and Llama-shaped layers):

* x  ~ N(0, 1), shape [b, s, h]
* every matrix and bias ~ N(0, 0.02)  (nn.Linear convention [out, in])
* norm scales = 1 + N(0, 0.02), LayerNorm shifts ~ N(0, 0.02)
* upstream gradient dy ~ N(0, 1), shape [b, s, h]

Everything is drawn in float32 from one ``torch.Generator`` seeded with
``seed`` and then cast to bf16; the draw order is fixed (x, the weights in
``WEIGHT_ORDER``, dy) so a (config, seed, device) triple always yields the same
tensors.
"""
from __future__ import annotations

import torch

WEIGHT_ORDER = ("ln1_w", "ln1_b", "wq", "bq", "wk", "bk", "wv", "bv", "wo", "bo",
                "ln2_w", "ln2_b", "w1", "b1", "w2", "b2", "w3")


def weight_shapes(h, n_heads, n_kv_heads, head_dim, ffn_dim, norm, act, has_bias):
    """Shapes of the parameters a layer variant takes (None = absent)."""
    Hd, Kd = n_heads * head_dim, n_kv_heads * head_dim
    shp = {"ln1_w": (h,), "ln1_b": (h,) if norm == 0 else None,
           "wq": (Hd, h), "bq": (Hd,) if has_bias else None,
           "wk": (Kd, h), "bk": (Kd,) if has_bias else None,
           "wv": (Kd, h), "bv": (Kd,) if has_bias else None,
           "wo": (h, Hd), "bo": (h,) if has_bias else None,
           "ln2_w": (h,), "ln2_b": (h,) if norm == 0 else None,
           "w1": (ffn_dim, h), "b1": (ffn_dim,) if (has_bias and act != 2) else None,
           "w2": (h, ffn_dim), "b2": (h,) if has_bias else None,
           "w3": (ffn_dim, h) if act == 2 else None}
    return shp


def make_layer_inputs(cfg, seed: int, device="cpu", with_dy=True, dtype=torch.bfloat16):
    """Return dict(x=..., dy=..., weights={name: tensor or None}).

    ``cfg`` is any object with fields b, s, h, n_heads, n_kv_heads, head_dim,
    ffn_dim, norm, act, has_bias."""
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))

    def randn(*shape):
        return torch.randn(*shape, generator=gen, device=device, dtype=torch.float32)

    x = randn(cfg.b, cfg.s, cfg.h).to(dtype)
    shapes = weight_shapes(cfg.h, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.ffn_dim,
                           cfg.norm, cfg.act, cfg.has_bias)
    weights = {}
    for name in WEIGHT_ORDER:
        shp = shapes[name]
        if shp is None:
            weights[name] = None
            continue
        t = randn(*shp) * 0.02
        if name in ("ln1_w", "ln2_w"):
            t = t + 1.0
        weights[name] = t.to(dtype)
    out = {"x": x, "weights": weights}
    if with_dy:
        out["dy"] = randn(cfg.b, cfg.s, cfg.h).to(dtype)
    return out


def make_lm_inputs(cfg, seed: int, device="cpu", dtype=torch.bfloat16):
    """Inputs of the language-model loss: dict(x=[n, h], w=[V, h],
    targets=[n] int32).  x ~ N(0, 1) (the last layer's normalised output),
    w ~ N(0, 0.02) like every other matrix (logits then have a standard
    deviation of about 0.02 sqrt(h)), targets uniform over the vocabulary.
    Drawn in that order from one generator seeded with ``seed``.

    ``cfg`` is any object with fields n, h, vocab."""
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    x = torch.randn(cfg.n, cfg.h, generator=gen, device=device, dtype=torch.float32).to(dtype)
    w = (torch.randn(cfg.vocab, cfg.h, generator=gen, device=device, dtype=torch.float32) * 0.02).to(dtype)
    t = torch.randint(0, cfg.vocab, (cfg.n,), generator=gen, device=device, dtype=torch.int64).to(torch.int32)
    return {"x": x, "w": w, "targets": t}
