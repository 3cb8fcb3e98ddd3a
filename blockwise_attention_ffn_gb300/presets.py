"""The five layer workloads the library is measured and checked on.

Shapes follow the workloads of "Blockwise Parallel Transformer for Long
Context Large Models" (GPT layers of the 1B and 3B models, section 5
"Evaluation Methodology") and of "Untied Ulysses" (a Llama3-8B layer with
grouped-query attention, section 5), at one layer and batch 1.
"""
from __future__ import annotations

from dataclasses import dataclass, replace


@dataclass(frozen=True)
class LayerConfig:
    b: int
    s: int
    h: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn_dim: int
    q_block: int = 128
    kv_block: int = 128
    ffn_block: int = 0
    head_chunk: int = 0
    causal: int = 1
    norm: int = 0        # 0 LayerNorm, 1 RMSNorm
    act: int = 0         # 0 GeLU (erf), 1 GeLU (tanh), 2 SwiGLU
    has_bias: int = 1
    norm_eps: float = 1e-5
    flags: int = 0
    rope_base: float = 0.0  # rotary position embedding base; 0 = none
    stage_order: int = 0    # head-chunk stages: 0 contiguous, 1 interleaved over the groups
    save_policy: int = 0    # kept for the backward: 0 log-sum-exp, 1 + Q/K/V, 2 + attention output
    name: str = ""
    backward: bool = False  # the workload includes the backward pass
    seed: int = 0

    def with_(self, **kw) -> "LayerConfig":
        return replace(self, **kw)


C1 = LayerConfig(name="gpt-small s=1024 h=256 4x64", b=1, s=1024, h=256, n_heads=4, n_kv_heads=4,
                 head_dim=64, ffn_dim=1024, seed=0)
C2 = LayerConfig(name="gpt-1b s=8192 h=2048 16x128", b=1, s=8192, h=2048, n_heads=16, n_kv_heads=16,
                 head_dim=128, ffn_dim=8192, ffn_block=2048, seed=1)
C3 = LayerConfig(name="gpt-3b s=32768 h=2560 32x80", b=1, s=32768, h=2560, n_heads=32, n_kv_heads=32,
                 head_dim=80, ffn_dim=10240, ffn_block=8192, backward=True, seed=2)
C4 = LayerConfig(name="gpt-1b long s=131072 h=2048 16x128", b=1, s=131072, h=2048, n_heads=16,
                 n_kv_heads=16, head_dim=128, ffn_dim=8192, q_block=256, kv_block=256,
                 ffn_block=8192, backward=True, seed=3)
C5 = LayerConfig(name="llama-8b s=65536 h=4096 32q/8kv x128 U=8", b=1, s=65536, h=4096, n_heads=32,
                 n_kv_heads=8, head_dim=128, ffn_dim=14336, head_chunk=8, norm=1, act=2, has_bias=0,
                 ffn_block=4096, backward=True, seed=4)

PRESETS = {"c1": C1, "c2": C2, "c3": C3, "c4": C4, "c5": C5}


@dataclass(frozen=True)
class LmConfig:
    """The language-model loss after the last layer: n positions of width h
    against a vocabulary of V tokens, the backward in blocks of vocab_block
    vocabulary columns (0: the library's default)."""
    n: int
    h: int
    vocab: int
    vocab_block: int = 0
    flags: int = 0
    name: str = ""
    seed: int = 0

    def with_(self, **kw) -> "LmConfig":
        return replace(self, **kw)


# The loss after the GPT-3B-shaped layer at s = 32768, over the GPT-2 BPE
# vocabulary of the OpenWebText models (50257 tokens).
LM3 = LmConfig(name="gpt-3b lm head s=32768 h=2560 V=50257", n=32768, h=2560, vocab=50257, seed=5)
