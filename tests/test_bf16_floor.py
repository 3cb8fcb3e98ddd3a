"""The error floor of a bf16-storage / fp32-accumulation layer, emulated on
the CPU, and the per-tensor bounds of the GPU parity tests derived from it.

tests/bf16_emulation.py runs the exact fp64 layer with exactly the bf16
roundings the kernels make (the operands of every product and every stored
activation); tests/golden/bf16_floor.json holds its relative Frobenius error
per tensor at the three backward workloads (GPT-3B at s = 2048, the long
GPT-1B and the Llama-8B layers at s = 1024) and at four GPU test layers (two
with rotary embedding), written by tests/golden/make_bf16_floor.py.  These tests pin that file to
the emulation, the emulation to the oracle, and the bounds to the file:

* a tensor gets the wider bound ATTN_GRAD_REL_FRO exactly when its floor
  exceeds the acceptance bound REL_FRO (5e-3) in some case: no
  bf16-operand implementation of this schedule can meet 5e-3 there;
* ATTN_GRAD_REL_FRO is at least 1.5 times the largest of those floors;
* every other tensor's floor is below REL_FRO, so it keeps REL_FRO.
"""
import json
import os

import numpy as np
import pytest

from blockwise_attention_ffn_gb300.presets import PRESETS, LayerConfig
from tests import bf16_emulation
from tests.gpu_helpers import ATTN_GRAD_REL_FRO, REL_FRO, WIDE_TENSORS, rel_bound

HERE = os.path.dirname(os.path.abspath(__file__))
GOLD = json.load(open(os.path.join(HERE, "golden", "bf16_floor.json")))
WORKLOADS = ("gpt-3b s=2048", "gpt-1b long s=1024", "llama-8b s=1024")


def _floors(cases=None):
    out = {}
    for case in cases or GOLD["cases"]:
        for k, v in GOLD["cases"][case]["rel_fro"].items():
            out[k] = max(out.get(k, 0.0), v)
    return out


def test_workloads_are_in_the_file():
    assert set(WORKLOADS) <= set(GOLD["cases"])


def test_wide_bound_goes_to_exactly_the_tensors_whose_floor_exceeds_the_acceptance_bound():
    """Over every case of the file: the three workloads and the GPU test
    layers (with and without rotary embedding, which makes the key bias
    gradient nonzero)."""
    fl = _floors()
    above = {k for k, v in fl.items() if v > REL_FRO}
    assert above == set(WIDE_TENSORS), (above, fl)
    assert ATTN_GRAD_REL_FRO >= 1.5 * max(fl[k] for k in above)
    for k, v in fl.items():
        assert v < rel_bound(k), (k, v)


@pytest.mark.slow
def test_golden_floor_is_the_emulation():
    """Re-run one workload case (about 10 s) and compare with the stored
    floors, so the file cannot drift from the emulation."""
    case = "gpt-1b long s=1024"
    e = bf16_emulation.floor_errors(PRESETS["c4"].with_(s=1024), seed=GOLD["cases"][case]["seed"])
    for k, want in GOLD["cases"][case]["rel_fro"].items():
        assert e[k][0] == pytest.approx(want, rel=1e-6, abs=1e-15), k


def test_emulation_without_rounding_is_the_oracle(monkeypatch):
    """With the rounding switched off the emulation is the exact layer: its
    output and every gradient equal the oracle's to fp64 rounding, so the
    floor measures the roundings and nothing else (a dropped term or a wrong
    operand in the emulation would show here)."""
    monkeypatch.setattr(bf16_emulation, "bf", lambda a: np.asarray(a, np.float64))
    for cfg in (LayerConfig(b=1, s=130, h=128, n_heads=2, n_kv_heads=2, head_dim=64, ffn_dim=256),
                LayerConfig(b=1, s=96, h=256, n_heads=4, n_kv_heads=2, head_dim=64, ffn_dim=192, norm=1, act=2,
                            has_bias=0, rope_base=10000.0)):
        e = bf16_emulation.floor_errors(cfg, seed=5)
        for k, (rel, _) in e.items():
            if k != "bk":
                assert rel < 1e-11, (cfg, k, rel)


def test_rounding_raises_the_floor_in_every_tensor():
    """With rounding on, every gradient (but the exactly known ones) has a
    floor well above fp64 noise: the emulation rounds on every path."""
    cfg = LayerConfig(b=1, s=130, h=128, n_heads=2, n_kv_heads=2, head_dim=64, ffn_dim=256)
    e = bf16_emulation.floor_errors(cfg, seed=5)
    for k, (rel, _) in e.items():
        if k not in ("bk", "b2"):
            assert rel > 1e-4, (k, rel)
