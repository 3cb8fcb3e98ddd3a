"""Writes tests/golden/bf16_floor.json: the error floor of the layer's
bf16-operand pipeline (tests/bf16_emulation.py) against the fp64 oracle, per
tensor, at the workload shapes (sequence shortened to what fp64 NumPy runs in
minutes) and at the GPU test layers.  Calls nothing but the oracle and the
emulation (no CUDA).

    python tests/golden/make_bf16_floor.py        # about 5 minutes on 8 cores
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

from blockwise_attention_ffn_gb300.presets import PRESETS, LayerConfig  # noqa: E402
from tests.bf16_emulation import floor_errors  # noqa: E402

# (name, config, seed): the three backward workloads, and two of the layers
# the GPU parity tests run
CASES = [
    ("gpt-3b s=2048", PRESETS["c3"].with_(s=2048), 3),
    ("gpt-1b long s=1024", PRESETS["c4"].with_(s=1024), 3),
    ("llama-8b s=1024", PRESETS["c5"].with_(s=1024), 3),
    ("gpt ragged s=300", LayerConfig(b=1, s=300, h=256, n_heads=4, n_kv_heads=4, head_dim=64, ffn_dim=1024,
                                     ffn_block=128), 3),
    ("llama gqa s=384", LayerConfig(b=1, s=384, h=512, n_heads=8, n_kv_heads=2, head_dim=64, ffn_dim=768,
                                    head_chunk=4, norm=1, act=2, has_bias=0), 3),
    # with rotary embedding the key bias gradient is no longer zero
    ("gpt ragged rope s=300", LayerConfig(b=1, s=300, h=256, n_heads=4, n_kv_heads=4, head_dim=64, ffn_dim=1024,
                                          ffn_block=128, rope_base=10000.0), 3),
    ("gqa bias rope s=400", LayerConfig(b=1, s=400, h=1024, n_heads=16, n_kv_heads=4, head_dim=64, ffn_dim=512,
                                        head_chunk=4, rope_base=10000.0), 3),
]


def main():
    out = {"_about": "relative Frobenius error and max-abs error (in units of the tensor's largest entry, "
                     "or 1) of the bf16-operand pipeline against the fp64 oracle, per tensor; written by "
                     "tests/golden/make_bf16_floor.py", "cases": {}}
    for name, cfg, seed in CASES:
        e = floor_errors(cfg, seed=seed)
        if not cfg.rope_base:
            e.pop("bk", None)  # exactly zero in exact arithmetic: no relative error to speak of
        out["cases"][name] = {"config": {k: getattr(cfg, k) for k in (
            "s", "h", "n_heads", "n_kv_heads", "head_dim", "ffn_dim", "norm", "act", "has_bias", "rope_base")},
            "seed": seed, "rel_fro": {k: v[0] for k, v in e.items()}, "max_abs": {k: v[1] for k, v in e.items()}}
        print(name, "done", flush=True)
    with open(os.path.join(HERE, "bf16_floor.json"), "w") as f:
        json.dump(out, f, indent=1, sort_keys=True)


if __name__ == "__main__":
    main()
