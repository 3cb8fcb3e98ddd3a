"""The pages' parameter, activation-memory and FLOP accounting.

TEST INFRASTRUCTURE ONLY.  Each function states the formula of the page it
restates; the tests pin them against the numbers those pages print.

Notation: s sequence, b micro-batch, h hidden size, a attention heads, c block
size, f FFN width.  Bytes assume 2-byte activations and 1-byte dropout masks,
as the pages do.
"""
from __future__ import annotations

from .ref import ACT_SWIGLU, NORM_LAYER, LayerCfg, weight_shapes


def param_count(cfg: LayerCfg) -> int:
    """Number of parameters of one layer as the oracle builds it (sum of the
    sizes of every weight array it consumes)."""
    total = 0
    for shp in weight_shapes(cfg).values():
        n = 1
        for t in shp:
            n *= t
        total += n
    return total


def gpt_layer_params(h: int) -> int:
    """12h^2 + 13h ("Training memory ...", section 3, "Parameters")."""
    return 12 * h * h + 13 * h


def gpt_model_params(L: int, h: int, V: int) -> int:
    """L layers + shared embedding Vh + final LayerNorm 2h (same page, section 4
    worked example and section 5 code)."""
    return L * gpt_layer_params(h) + V * h + 2 * h


def llama_layer_params(h: int, f: int, g: int) -> int:
    """Llama-style layer: Wq, Wo (h x h), Wk, Wv (h x h/g), three h x f SwiGLU
    matrices, two RMSNorm scales (same page, "Parameters", Llama paragraph)."""
    return 2 * h * h + 2 * h * (h // g) + 3 * h * f + 2 * h


# ---------------------------------------------------------------- activations

def vanilla_layer_activation_bytes(s, b, h, a) -> int:
    """34 sbh + 5 a s^2 b ("Training memory ...", section 3, the theorem)."""
    return 34 * s * b * h + 5 * a * s * s * b


def theorem_items(s, b, h, a) -> dict:
    """The theorem's proof, tensor by tensor (bytes), in the order it lists
    them; summing them must give vanilla_layer_activation_bytes."""
    sbh = s * b * h
    core = a * s * s * b
    return {
        "ln1_input": 2 * sbh,
        "qkv_input": 2 * sbh,
        "q_and_k": 4 * sbh,
        "softmax_output": 2 * core,
        "attn_dropout_mask": core,
        "dropout_output": 2 * core,
        "v": 2 * sbh,
        "proj_input": 2 * sbh,
        "proj_dropout_mask": sbh,
        "fc1_input": 2 * sbh,
        "gelu_input": 8 * sbh,
        "fc2_input": 8 * sbh,
        "mlp_dropout_mask": sbh,
        "ln2_input": 2 * sbh,
    }


def flash_layer_activation_bytes(s, b, h) -> int:
    """With fused attention the s^2 core disappears: about 34 sbh."""
    return 34 * s * b * h


def full_checkpoint_bytes(s, b, h) -> int:
    """Full checkpointing keeps the layer input only: 2 sbh."""
    return 2 * s * b * h


def checkpoint_every_k(L, k, c, A) -> float:
    """M(k) ~ (L/k) c + k A (same page, "Checkpoint every k layers")."""
    return (L / k) * c + k * A


def bpt_activation_terms(s, b, h, c) -> dict:
    """Peak activation terms of the BPT page, section 3.4 "Memory Cost
    Analysis": FlashAttention-style attention 2bsh and FFN 8bsh; BPT
    attention inner loop 4bch, FFN block 19bch (2 + 8 + 8 + 1), accumulated
    output 2bsh."""
    return {
        "flash_attention": 2 * b * s * h,
        "flash_ffn": 8 * b * s * h,
        "flash_total": max(2 * b * s * h, 8 * b * s * h),
        "bpt_attention_block": 4 * b * c * h,
        "bpt_ffn_block": (2 + 8 + 8 + 1) * b * c * h,
        "bpt_output": 2 * b * s * h,
        # the page's "peak memory for a BPT layer": max(4bch, 19bch, 2bsh)
        "bpt_total": max(4 * b * c * h, 19 * b * c * h, 2 * b * s * h),
    }


def ulysses_attention_peak_bytes(S, C, H, d) -> int:
    """12 (S/C) H d_head bytes: the full-head Q, K, V of a device's S/C rows
    (6 bytes per row, head and dimension) and all-to-all buffers of the same
    size ("Untied Ulysses ...", "Where Prior Approaches Fall Short", the
    DS-Ulysses paragraph)."""
    return 12 * (S // C) * H * d


def upipe_stage_peak_bytes(S, C, U, d) -> int:
    """12 (S/C) U d_head bytes: the same buffers for the U heads of one stage,
    reused stage after stage (same page, "The Core Mechanism: Headwise
    Chunking via UPipe")."""
    return 12 * (S // C) * U * d


def upipe_one_gpu_qkv_bytes(S, U, G, d, b=1) -> int:
    """One GPU (C = 1) has no all-to-all, so a stage holds only its
    projections: 2 bytes x S x (U query heads + U/G key and U/G value heads)
    x d_head.  With G = 1 this is the Q/K/V half (6 S U d) of the page's
    12 S U d; with grouped queries the key/value heads of the stage's U/G
    groups are made once."""
    return 2 * b * S * (U + 2 * (U // G)) * d


def logits_bytes(s, b, V) -> int:
    """fp32 logits: 4 sbV (same page, "The logits")."""
    return 4 * s * b * V


def model_state_bytes(psi) -> int:
    """Mixed-precision Adam: 16 bytes per parameter (same page)."""
    return 16 * psi


# ----------------------------------------------------------------------- FLOPs

def layer_flops(cfg: LayerCfg) -> dict:
    """Forward FLOPs of one layer (multiply-add = 2 FLOPs), the causal half of
    the attention only when causal.

    F_linear = 2 s h (H + 2 H_kv) d + 2 s H d h + 2 s h f n_mat   (n_mat = 2 GeLU, 3 SwiGLU)
    F_attn   = 2 s^2 H d (causal; 4 s^2 H d when not causal)
    The step estimate 3 (24 b s h^2 + 4 b s^2 h) of "Training memory ...",
    section 3 ("What changes the count") is the non-causal, f = 4h special
    case of 3 (F_linear + F_attn)."""
    s, h, H, Hk, d, f = cfg.s, cfg.h, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.ffn_dim
    n_mat = 3 if cfg.act == ACT_SWIGLU else 2
    qkv = 2 * s * h * (H + 2 * Hk) * d
    wo = 2 * s * H * d * h
    ffn = 2 * s * h * f * n_mat
    attn = (2 if cfg.causal else 4) * s * s * H * d
    b = cfg.b
    return {"qkv": b * qkv, "wo": b * wo, "ffn": b * ffn, "fc2": b * 2 * s * f * h,
            "linear": b * (qkv + wo + ffn), "attn": b * attn,
            "forward": b * (qkv + wo + ffn + attn)}


def step_flops(cfg: LayerCfg) -> dict:
    """Model FLOPs of a training step (3x forward) and the FLOPs a recompute
    backward executes: forward + recompute of everything but fc2 + backward of
    the linears (2 F_linear) + attention backward with the score rebuild
    (2.5 F_attn: S, dP, dV, dK, dQ)."""
    f = layer_flops(cfg)
    model = 3 * f["forward"]
    executed = (f["forward"] + (f["forward"] - f["fc2"]) + 2 * f["linear"] + 2.5 * f["attn"])
    return {"model": model, "executed": executed, **f}


def norm_kind_is_layer(cfg: LayerCfg) -> bool:
    return cfg.norm == NORM_LAYER
