"""bpt_attention_bwd_noalloc: the attention backward for callers that cannot
allocate device memory at call time (an engine plugin running on a memory plan
fixed in advance, a hot path that cannot afford cudaMalloc and the device
synchronisation it may cause).  Its scratch is a fixed array inside the
library, so the caller passes only inputs and outputs.

Checked against the regular entry point, which takes a caller-allocated
workspace, on calls in a row that share the array: a large call first, then
smaller ones with another padded length, head count and batch, so each later
call finds the array holding the earlier call's values in the rows it uses
and past them.

This file is collected last so that a run stopping at the first failure has
run every other test before it."""
import pytest
import torch

import blockwise_attention_ffn_gb300 as bpt
from blockwise_attention_ffn_gb300.presets import LayerConfig
from tests.gpu_helpers import assert_close, to64

pytestmark = pytest.mark.gpu

# a large call first (s_pad 1024, 8 heads), then smaller ones (s_pad 384 and
# 256, fewer heads, a batch of two)
CALLS = [
    LayerConfig(b=1, s=1000, h=512, n_heads=8, n_kv_heads=2, head_dim=64, ffn_dim=64),
    LayerConfig(b=1, s=300, h=256, n_heads=4, n_kv_heads=2, head_dim=64, ffn_dim=64),
    LayerConfig(b=2, s=200, h=240, n_heads=3, n_kv_heads=3, head_dim=80, ffn_dim=64, causal=0),
]


def _inputs(cfg, seed):
    g = torch.Generator().manual_seed(seed)
    H, Hk, d, rows = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.b * cfg.s
    qkv = torch.randn(rows, (H + 2 * Hk) * d, generator=g).to(torch.bfloat16).cuda()
    dout = torch.randn(rows, H * d, generator=g).to(torch.bfloat16).cuda()
    o = torch.empty(rows, H * d, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(cfg.b, H, bpt.s_pad(cfg), dtype=torch.float32, device="cuda")
    bpt.bpt_attention_fwd(cfg, qkv, o, lse)
    return qkv, o, lse, dout


def test_noalloc_matches_workspace_entry_point_on_calls_in_a_row():
    for seed, cfg in enumerate(CALLS, start=1):
        qkv, o, lse, dout = _inputs(cfg, seed)
        want = torch.empty_like(qkv)
        ws = bpt.alloc_bytes(bpt.bpt_attention_bwd_workspace_bytes(cfg))
        bpt.bpt_attention_bwd(cfg, qkv, o, lse, dout, want, ws)
        got = torch.full_like(qkv, float("nan"))
        bpt.bpt_attention_bwd_noalloc(cfg, qkv, o, lse, dout, got)
        torch.cuda.synchronize()
        assert bpt.bpt_last_device_error()[0] == bpt.BPT_OK
        # the two entry points run the same kernels; the default mode's sums
        # follow the order the products arrive in, so allow that difference
        assert_close(to64(got), to64(want), f"dQKV (call {seed})", grad=True, rel_fro=1e-3)
        # in the fixed-order mode both must agree bit for bit
        det = cfg.with_(flags=bpt.BPT_FLAG_DETERMINISTIC)
        bpt.bpt_attention_bwd(det, qkv, o, lse, dout, want, ws)
        bpt.bpt_attention_bwd_noalloc(det, qkv, o, lse, dout, got)
        torch.cuda.synchronize()
        assert bpt.bpt_last_device_error()[0] == bpt.BPT_OK
        assert torch.equal(got, want), seed


def test_noalloc_rejects_problems_beyond_the_scratch():
    big = CALLS[0].with_(s=1 << 20, h=4096, n_heads=32, n_kv_heads=8, head_dim=128)
    assert bpt.bpt_attention_bwd_workspace_bytes(big) > bpt.NOALLOC_SCRATCH_BYTES
    t = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(bpt.BptError) as e:
        bpt.bpt_attention_bwd_noalloc(big, t, t, t, t, t)
    assert e.value.status == bpt.BPT_ENOSPC
