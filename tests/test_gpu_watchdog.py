"""The device-side wait limit, exercised without faulting anything: a wait on
a barrier that nothing signals must run out, be reported through the error
word with its wait site, and leave the context usable for the next call."""
import time

import numpy as np
import pytest
import torch

import blockwise_attention_ffn_gb300 as bpt
from blockwise_attention_ffn_gb300.presets import LayerConfig
from tests.gpu_helpers import assert_close, to64

pytestmark = pytest.mark.gpu


def test_a_wait_that_runs_out_is_reported_and_the_context_survives():
    bpt.lib()
    torch.cuda.synchronize()
    assert bpt.bpt_last_device_error() == (bpt.BPT_OK, 0)

    t0 = time.perf_counter()
    bpt.bpt_watchdog_selftest()
    st, site = bpt.bpt_last_device_error()  # synchronises
    waited = time.perf_counter() - t0
    assert (st, site) == (bpt.BPT_ETIMEOUT, bpt.BPT_WATCHDOG_SELFTEST_SITE)
    # the limit is 4e9 SM cycles (4e8 in a BPT_DEBUG=1 build): at the
    # 2.07 GHz maximum clock at least 1.9 s (0.19 s), so the wait really ran
    assert waited >= 0.1, waited
    # reading cleared the word
    assert bpt.bpt_last_device_error() == (bpt.BPT_OK, 0)

    # the next call runs normally: equal keys give the running mean of V
    b, s, H, Hkv, d = 1, 200, 2, 2, 64
    cfg = LayerConfig(b=b, s=s, h=H * d, n_heads=H, n_kv_heads=Hkv, head_dim=d, ffn_dim=64, causal=1)
    g = torch.Generator().manual_seed(7)
    qkv = torch.randn(b * s, (H + 2 * Hkv) * d, generator=g)
    qkv[:, H * d:(H + Hkv) * d] = qkv[0:1, H * d:(H + Hkv) * d]
    qkv = qkv.to(torch.bfloat16)
    o = torch.zeros(b * s, H * d, dtype=torch.bfloat16, device="cuda")
    bpt.bpt_attention_fwd(cfg, qkv.cuda(), o, None)
    assert bpt.bpt_last_device_error() == (bpt.BPT_OK, 0)
    v = to64(qkv)[:, (H + Hkv) * d:].reshape(s, Hkv, d)
    want = np.cumsum(v, 0) / np.arange(1, s + 1)[:, None, None]
    assert_close(to64(o).reshape(s, H, d), want, "prefix mean after the self-test")
