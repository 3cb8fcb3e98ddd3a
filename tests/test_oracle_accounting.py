"""The oracle's accounting formulas against the numbers the pages print."""
import json
import os

import pytest

from oracle import accounting as A
from oracle.ref import LayerCfg

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_numbers.json")))


def test_activation_theorem_in_sbh_units():
    g = GOLD["activation_sbh"]
    s, b, h, a = g["s"], g["b"], g["h"], g["a"]
    sbh = s * b * h
    assert A.vanilla_layer_activation_bytes(s, b, h, a) == g["vanilla"] * sbh
    assert A.flash_layer_activation_bytes(s, b, h) == g["flash"] * sbh
    assert A.full_checkpoint_bytes(s, b, h) == g["checkpoint"] * sbh
    assert sum(A.theorem_items(s, b, h, a).values()) == A.vanilla_layer_activation_bytes(s, b, h, a)


def test_worked_example_1p3b():
    g = GOLD["worked_example_1p3b"]
    L, h, a, V, s, b = g["L"], g["h"], g["a"], g["V"], g["s"], g["b"]
    psi = A.gpt_model_params(L, h, V)
    assert psi == g["psi"]
    assert L * A.gpt_layer_params(h) == g["layers_params"]
    assert V * h == g["embedding"]
    assert round(12 * L * h * h / psi, 3) == g["ratio_12Lh2"]
    gb = 1e9
    states = A.model_state_bytes(psi) / gb
    act = L * A.vanilla_layer_activation_bytes(s, b, h, a) / gb
    logits = A.logits_bytes(s, b, V) / gb
    assert round(states, 1) == g["states_gb"]
    assert round(act, 1) == g["act_gb"]
    assert round(logits, 1) == g["logits_gb"]
    assert round(states + act + logits, 1) == g["total_gb"]
    flash = L * A.flash_layer_activation_bytes(s, b, h) / gb
    assert round(flash, 1) == g["flash_act_gb"]
    assert round(states + flash + logits, 1) == g["flash_total_gb"]
    ck_in = L * A.full_checkpoint_bytes(s, b, h) / gb
    rebuilt = A.flash_layer_activation_bytes(s, b, h) / gb
    assert round(ck_in, 1) == g["ckpt_inputs_gb"]
    assert round(rebuilt, 1) == g["ckpt_rebuilt_gb"]
    assert round(states + ck_in + rebuilt + logits, 1) == g["ckpt_total_gb"]


def test_bpt_memory_terms():
    g = GOLD["bpt_memory_terms"]
    t = A.bpt_activation_terms(g["s"], g["b"], g["h"], g["c"])
    assert round(t["bpt_output"] / 1e6) == g["two_bsh_millions"]
    assert round(t["bpt_ffn_block"] / 1e6) == g["nineteen_bch_millions"]
    assert t["flash_total"] / t["bpt_total"] == g["flash_over_bpt"]
    # attention 2bsh vs FFN 8bsh in the FlashAttention regime: 4x
    assert t["flash_ffn"] == 4 * t["flash_attention"]


def test_upipe_stage_memory_against_the_pages_numbers():
    g = GOLD["upipe_memory"]
    S, d = 1 << 20, 128
    q = g["qwen3_32b"]
    uly = A.ulysses_attention_peak_bytes(S, q["C"], q["H"], d)
    up = A.upipe_stage_peak_bytes(S, q["C"], q["U"], d)
    assert uly == q["ulysses_S_dhead"] * S * d
    assert up == q["upipe_S_dhead"] * S * d
    assert 1 - up / uly == q["reduction"]
    f = g["figure3_example"]
    assert A.upipe_stage_peak_bytes(S, f["C"], f["U"], d) == \
        f["upipe_over_ulysses"] * A.ulysses_attention_peak_bytes(S, f["C"], f["H"], d)
    # one GPU: no all-to-all buffers, so a stage of U heads (no grouping)
    # holds the Q/K/V half of the page's 12 S U d
    for U in (1, 2, 8):
        assert 2 * A.upipe_one_gpu_qkv_bytes(S, U, 1, d) == A.upipe_stage_peak_bytes(S, 1, U, d)
    # grouped queries: U query heads share U/G key/value heads
    assert A.upipe_one_gpu_qkv_bytes(S, 8, 4, d) == 2 * S * (8 + 2 + 2) * d


def test_checkpoint_every_k():
    g = GOLD["checkpoint_every_k"]
    assert A.checkpoint_every_k(g["L"], 1, g["c_sbh"], g["A_sbh"]) == g["M1_sbh"]
    assert A.checkpoint_every_k(g["L"], 2, g["c_sbh"], g["A_sbh"]) == g["M2_sbh"]


def test_step_flops_reduce_to_page_estimate():
    # non-causal, f = 4h, H*d = h, G = 1: 3 * (24 b s h^2 + 4 b s^2 h)
    s, h = 512, 256
    cfg = LayerCfg(s=s, h=h, n_heads=4, n_kv_heads=4, head_dim=64, ffn_dim=4 * h, causal=False)
    f = A.step_flops(cfg)
    assert f["model"] == 3 * (24 * s * h * h + 4 * s * s * h)
    # causal halves the attention part only
    cc = LayerCfg(s=s, h=h, n_heads=4, n_kv_heads=4, head_dim=64, ffn_dim=4 * h)
    fc = A.layer_flops(cc)
    assert fc["attn"] * 2 == A.layer_flops(cfg)["attn"]


@pytest.mark.parametrize("h", [256, 2048, 2560])
def test_gpt_params_identity(h):
    cfg = LayerCfg(s=8, h=h, n_heads=h // 64, n_kv_heads=h // 64, head_dim=64, ffn_dim=4 * h)
    assert A.param_count(cfg) == 12 * h * h + 13 * h


@pytest.mark.parametrize("name", ["c1", "c2", "c3", "c4", "c5"])
def test_bench_flop_count_matches_oracle_accounting(name):
    """The bench's FLOP count (the headline metric's numerator) against the
    oracle's page-pinned formulas.  The bench counts causal pairs exactly,
    s (s + 1) / 2 per head instead of s^2 / 2, so the attention terms differ by
    a factor (1 + 1/s); the head-chunked workload also re-projects Q/K/V for
    the backward, an executed extra the oracle's step estimate does not have."""
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    from blockwise_attention_ffn_gb300.presets import PRESETS
    from tests.oracle_helpers import oracle_cfg
    c = PRESETS[name]
    got = bench.flop_counts(c)
    want = A.step_flops(oracle_cfg(c))
    exact = 1 + 1 / c.s
    assert got["linear"] == want["linear"]
    assert got["attn"] == pytest.approx(want["attn"] * exact, rel=1e-12)
    assert got["forward"] == pytest.approx(want["linear"] + want["attn"] * exact, rel=1e-12)
    if not c.backward:
        assert got["executed"] == got["forward"]
        return
    assert got["model"] == pytest.approx(3 * got["forward"], rel=1e-12)
    extra = 0
    if c.head_chunk and c.head_chunk < c.n_heads:
        extra = want["qkv"]
    want_exec = (2 * want["forward"] - want["fc2"] + 2 * want["linear"] + 2.5 * want["attn"]
                 + (2 + 2.5) * want["attn"] * (exact - 1) + extra)
    assert got["executed"] == pytest.approx(want_exec, rel=1e-12)


@pytest.mark.parametrize("name,policy", [("c3", 1), ("c3", 2), ("c5", 1), ("c5", 2)])
def test_bench_flop_count_drops_what_the_kept_activations_save(name, policy):
    """With a save policy the backward does not rebuild the Q/K/V projection
    (policy 1), nor the attention forward (policy 2): the executed count
    drops by exactly those terms of the oracle's accounting; the model count
    (3 forwards) does not change."""
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    from blockwise_attention_ffn_gb300.presets import PRESETS
    from tests.oracle_helpers import oracle_cfg
    c = PRESETS[name]
    base = bench.flop_counts(c)
    got = bench.flop_counts(c.with_(save_policy=policy))
    want = A.step_flops(oracle_cfg(c))
    exact = 1 + 1 / c.s
    chunk_extra = want["qkv"] if c.head_chunk and c.head_chunk < c.n_heads else 0
    drop = chunk_extra + want["qkv"] + (want["attn"] * exact if policy == 2 else 0)
    assert got["executed"] == pytest.approx(base["executed"] - drop, rel=1e-12)
    assert got["model"] == base["model"]
