"""bpt_attention_bwd_noalloc: the attention backward for callers that cannot
allocate device memory at call time (an engine plugin running on a memory plan
fixed in advance, a hot path that cannot afford cudaMalloc and the device
synchronisation it may cause).  Its scratch is a fixed array inside the
library, so the caller passes only inputs and outputs.  Checked against the
regular entry point, which takes a caller-allocated workspace, on two calls in
a row (the second sees the array as the first left it).

This file is collected last so that a run stopping at the first failure has
run every other test before it."""
import pytest
import torch

import blockwise_attention_ffn_gb300 as bpt
from blockwise_attention_ffn_gb300.presets import LayerConfig
from tests.gpu_helpers import assert_close, to64

pytestmark = pytest.mark.gpu

CFG = LayerConfig(b=1, s=300, h=256, n_heads=4, n_kv_heads=2, head_dim=64, ffn_dim=64)


def _inputs(seed):
    g = torch.Generator().manual_seed(seed)
    H, Hk, d, s = CFG.n_heads, CFG.n_kv_heads, CFG.head_dim, CFG.s
    qkv = torch.randn(s, (H + 2 * Hk) * d, generator=g).to(torch.bfloat16).cuda()
    dout = torch.randn(s, H * d, generator=g).to(torch.bfloat16).cuda()
    o = torch.empty(s, H * d, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(1, H, bpt.s_pad(CFG), dtype=torch.float32, device="cuda")
    bpt.bpt_attention_fwd(CFG, qkv, o, lse)
    return qkv, o, lse, dout


def test_noalloc_matches_workspace_entry_point_twice():
    for seed in (1, 2):
        qkv, o, lse, dout = _inputs(seed)
        want = torch.empty_like(qkv)
        ws = bpt.alloc_bytes(bpt.bpt_attention_bwd_workspace_bytes(CFG))
        bpt.bpt_attention_bwd(CFG, qkv, o, lse, dout, want, ws)
        got = torch.full_like(qkv, float("nan"))
        bpt.bpt_attention_bwd_noalloc(CFG, qkv, o, lse, dout, got)
        torch.cuda.synchronize()
        assert bpt.bpt_last_device_error()[0] == bpt.BPT_OK
        assert_close(to64(got), to64(want), f"dQKV (call {seed})", grad=True)


def test_noalloc_rejects_problems_beyond_the_scratch():
    big = CFG.with_(s=1 << 20, h=4096, n_heads=32, n_kv_heads=8, head_dim=128)
    assert bpt.bpt_attention_bwd_workspace_bytes(big) > bpt.NOALLOC_SCRATCH_BYTES
    t = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(bpt.BptError) as e:
        bpt.bpt_attention_bwd_noalloc(big, t, t, t, t, t)
    assert e.value.status == bpt.BPT_ENOSPC
