"""The C-ABI library loads on a machine without a GPU, exports every function
include/bpt.h declares, and rejects invalid arguments on the host before it
launches anything."""
import ctypes
import os
import re

import pytest

import blockwise_attention_ffn_gb300 as bpt
from blockwise_attention_ffn_gb300 import presets

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def built():
    from blockwise_attention_ffn_gb300 import build
    build.build()
    return bpt.lib()


def _declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", fn)).read()
            txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
            names |= set(re.findall(r"\b(bpt_[a-z0-9_]+)\s*\(", txt))
    return names


def test_every_declared_symbol_is_exported(built):
    names = _declared_functions()
    assert {"bpt_layer_fwd", "bpt_layer_bwd", "bpt_attn_headchunk"} <= names
    for n in names:
        assert hasattr(built, n), n


def test_config_struct_matches_header():
    hdr = open(os.path.join(ROOT, "include", "bpt.h")).read()
    body = hdr[hdr.index("typedef struct {"):hdr.index("} bpt_config;")]
    fields = re.findall(r"\b([a-z_0-9]+)\b(?=[,;])", body.replace("int32_t", "").replace("float", ""))
    assert fields == [f for f, _ in bpt.BptConfig._fields_]
    assert ctypes.sizeof(bpt.BptConfig) == 4 * len(fields)
    wbody = hdr[hdr.index("const void *ln1_w"):hdr.index("} bpt_weights;")]
    wf = re.findall(r"\*([a-z0-9_]+)", wbody)
    assert tuple(wf) == bpt.WEIGHT_FIELDS


def test_watchdog_selftest_site_matches_header(built):
    hdr = open(os.path.join(ROOT, "include", "bpt.h")).read()
    m = re.search(r"#define BPT_WATCHDOG_SELFTEST_SITE (\d+)", hdr)
    assert m and int(m.group(1)) == bpt.BPT_WATCHDOG_SELFTEST_SITE


def test_watchdog_selftest_without_a_device_launches_nothing(built):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present: the GPU test covers the self-test")
    assert built.bpt_watchdog_selftest(None) == bpt.BPT_ECUDA


@pytest.mark.parametrize("U", [8, 16, 32])
def test_headchunk_workspace_is_one_stage_of_projections(built, U):
    """The head-chunk call's workspace is one stage's Q/K/V buffer, the
    one-GPU form of the headwise-chunking page's per-stage peak: it scales
    with U, not with the number of heads."""
    from oracle import accounting
    c = presets.C5.with_(head_chunk=U)
    G = c.n_heads // c.n_kv_heads
    want = accounting.upipe_one_gpu_qkv_bytes(c.s, U, G, c.head_dim, b=c.b)
    assert bpt.bpt_workspace_bytes(c, bpt.BPT_PASS_HEADCHUNK) == (want + 255) // 256 * 256


def test_status_strings(built):
    for s in range(6):
        assert bpt.bpt_status_string(s)
    assert "unknown" in bpt.bpt_status_string(99)


def test_workspace_sizes_are_host_only(built):
    c3 = presets.C3
    assert bpt.bpt_workspace_bytes(c3, bpt.BPT_PASS_FWD) > 0
    assert bpt.bpt_workspace_bytes(c3, bpt.BPT_PASS_BWD) > bpt.bpt_workspace_bytes(c3, bpt.BPT_PASS_FWD)
    assert bpt.bpt_saved_bytes(c3) == 1 * 32 * 32768 * 4
    # invalid configs report 0 bytes
    assert bpt.bpt_workspace_bytes(c3.with_(h=2561), 0) == 0
    assert bpt.bpt_workspace_bytes(c3.with_(head_chunk=5), 0) == 0
    assert bpt.bpt_workspace_bytes(c3.with_(head_dim=72), 0) == 0
    # head chunking bounds the stage buffer: workspace shrinks with U
    c5 = presets.C5
    full = bpt.bpt_workspace_bytes(c5.with_(head_chunk=32), bpt.BPT_PASS_HEADCHUNK)
    part = bpt.bpt_workspace_bytes(c5.with_(head_chunk=8), bpt.BPT_PASS_HEADCHUNK)
    assert full == pytest.approx(4 * part, rel=1e-3)


def _call_fwd(cfg, x=1 << 20, y=1 << 20, ws=1 << 20, wsz=1 << 40):
    L = bpt.lib()
    c = bpt.make_config(cfg)
    w = bpt.BptWeights(*([1 << 20] * len(bpt.WEIGHT_FIELDS)))
    return L.bpt_layer_fwd(ctypes.byref(c), ctypes.byref(w), x, y, None, ws, wsz, None)


@pytest.mark.parametrize("bad", [
    dict(s=0), dict(h=100), dict(n_heads=5), dict(head_chunk=3), dict(q_block=64),
    dict(ffn_block=100), dict(norm=2), dict(act=3), dict(norm_eps=0.0), dict(flags=16),
    dict(b=0), dict(causal=2), dict(has_bias=2), dict(n_kv_heads=0),
    dict(rope_base=0.5), dict(rope_base=-10000.0), dict(rope_base=float("nan")), dict(rope_base=float("inf")),
    dict(stage_order=2), dict(stage_order=-1), dict(save_policy=3), dict(save_policy=-1),
    # interleaved stages need whole groups: U = 2 over H_kv = 4 key/value heads
    dict(n_heads=4, n_kv_heads=4, head_chunk=2, stage_order=1),
])
def test_invalid_config_rejected_before_launch(built, bad):
    cfg = presets.C1.with_(**bad)
    assert _call_fwd(cfg) == bpt.BPT_EINVAL


def test_known_flags_accepted(built):
    """Every defined flag passes validation.  Accumulation, one stream and the
    debug checks leave the workspace plan alone; the fixed-order mode adds
    room for its per-block partial sums to the backward's workspace only."""
    base = bpt.bpt_workspace_bytes(presets.C1, bpt.BPT_PASS_BWD)
    plain = presets.C1.with_(flags=bpt.BPT_FLAG_ACCUM_GRADS | bpt.BPT_FLAG_ONE_STREAM | bpt.BPT_FLAG_DEBUG_CHECKS)
    assert base > 0
    assert bpt.bpt_workspace_bytes(plain, bpt.BPT_PASS_BWD) == base
    det = presets.C1.with_(flags=bpt.BPT_FLAG_DETERMINISTIC)
    for p in (bpt.BPT_PASS_FWD, bpt.BPT_PASS_HEADCHUNK):
        assert bpt.bpt_workspace_bytes(det, p) == bpt.bpt_workspace_bytes(presets.C1, p)
    # 256 blocks x (dw, db) x h floats for the norm backward, 64 bands x the
    # widest column sum (f here) for the bias gradients
    c = presets.C1
    extra = 256 * 2 * c.h * 4 + 64 * max(c.h, c.ffn_dim, 3 * c.n_heads * c.head_dim) * 4
    assert bpt.bpt_workspace_bytes(det, bpt.BPT_PASS_BWD) == base + extra
    assert bpt.bpt_workspace_bytes(presets.C1.with_(flags=16), bpt.BPT_PASS_BWD) == 0


def test_debug_checks_reject_pointers_outside_device_memory(built):
    """BPT_FLAG_DEBUG_CHECKS refuses, before any launch, pointers that do not
    lie in device memory of the current device (here: no device at all, or
    host addresses)."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present: the GPU test covers the debug checks")
    L = bpt.lib()
    dbg = presets.C1.with_(flags=bpt.BPT_FLAG_DEBUG_CHECKS)
    assert _call_fwd(dbg) == bpt.BPT_EINVAL
    c = bpt.make_config(dbg)
    p = 1 << 20
    assert L.bpt_attention_fwd(ctypes.byref(c), p, p, None, None) == bpt.BPT_EINVAL
    assert bpt.bpt_check_device_range(p, 16) == bpt.BPT_EINVAL
    assert L.bpt_check_device_range(None, 16) == bpt.BPT_EINVAL


def test_rope_base_accepted_and_plan_unchanged(built):
    """Rotary embedding works in place on the projection buffer: it needs no
    workspace of its own."""
    for p in (bpt.BPT_PASS_FWD, bpt.BPT_PASS_BWD, bpt.BPT_PASS_HEADCHUNK):
        for c in (presets.C1, presets.C5):
            assert bpt.bpt_workspace_bytes(c.with_(rope_base=10000.0), p) == bpt.bpt_workspace_bytes(c, p) > 0


def test_unsupported_head_dim(built):
    assert _call_fwd(presets.C1.with_(head_dim=72, h=288)) == bpt.BPT_EUNSUPPORTED


def test_null_and_misaligned_pointers_rejected(built):
    assert _call_fwd(presets.C1, x=None) == bpt.BPT_EINVAL
    assert _call_fwd(presets.C1, y=(1 << 20) + 2) == bpt.BPT_EINVAL


def test_small_workspace_rejected(built):
    assert _call_fwd(presets.C1, wsz=1024) == bpt.BPT_ENOSPC


def test_missing_weight_rejected(built):
    L = bpt.lib()
    c = bpt.make_config(presets.C1)
    ptrs = [1 << 20] * len(bpt.WEIGHT_FIELDS)
    ptrs[bpt.WEIGHT_FIELDS.index("bo")] = None
    w = bpt.BptWeights(*ptrs)
    assert L.bpt_layer_fwd(ctypes.byref(c), ctypes.byref(w), 1 << 20, 1 << 20, None, 1 << 20,
                           1 << 40, None) == bpt.BPT_EINVAL


def test_attention_rows_beyond_int32_unsupported(built):
    """b * H * s_pad past 2^31 - 1 would overflow the extra rows' TMA row
    coordinate: the attention backward refuses it before any launch."""
    L = bpt.lib()
    s = (1 << 24) + 128                      # 128 heads x s_pad = 2^31 + 2^14
    cfg = presets.C1.with_(s=s, h=8192, n_heads=128, n_kv_heads=128, head_dim=64, ffn_dim=8192)
    c = bpt.make_config(cfg)
    p = 1 << 20
    rc = L.bpt_attention_bwd(ctypes.byref(c), p, p, p, p, p, p, 1 << 62, None)
    assert rc == bpt.BPT_EUNSUPPORTED


def test_noalloc_entry_rejects_on_the_host(built):
    """bpt_attention_bwd_noalloc classifies its arguments before touching the
    device: bad pointers, bad configs and problems beyond its fixed scratch."""
    L = bpt.lib()
    p, odd = 1 << 20, (1 << 20) + 2
    ok = bpt.make_config(presets.C1)
    assert L.bpt_attention_bwd_noalloc(ctypes.byref(ok), None, p, p, p, p, None) == bpt.BPT_EINVAL
    assert L.bpt_attention_bwd_noalloc(ctypes.byref(ok), p, p, p, odd, p, None) == bpt.BPT_EINVAL
    bad = bpt.make_config(presets.C1.with_(q_block=64))
    assert L.bpt_attention_bwd_noalloc(ctypes.byref(bad), p, p, p, p, p, None) == bpt.BPT_EINVAL
    odd_d = bpt.make_config(presets.C1.with_(head_dim=72, h=288))
    assert L.bpt_attention_bwd_noalloc(ctypes.byref(odd_d), p, p, p, p, p, None) == bpt.BPT_EUNSUPPORTED
    big = presets.C1.with_(s=1 << 20, h=4096, n_heads=32, n_kv_heads=8, head_dim=128)
    assert bpt.bpt_attention_bwd_workspace_bytes(big) > bpt.NOALLOC_SCRATCH_BYTES
    cb = bpt.make_config(big)
    assert L.bpt_attention_bwd_noalloc(ctypes.byref(cb), p, p, p, p, p, None) == bpt.BPT_ENOSPC


def test_attention_entries_reject_bad_pointers_on_the_host(built):
    L = bpt.lib()
    c = bpt.make_config(presets.C1)
    p, odd = 1 << 20, (1 << 20) + 2
    assert L.bpt_attention_fwd(ctypes.byref(c), None, p, p, None) == bpt.BPT_EINVAL
    assert L.bpt_attention_fwd(ctypes.byref(c), p, odd, p, None) == bpt.BPT_EINVAL
    assert L.bpt_attention_bwd(ctypes.byref(c), p, p, p, p, p, p, 1024, None) == bpt.BPT_ENOSPC
    assert L.bpt_attention_bwd(ctypes.byref(c), p, p, p, p, None, p, 1 << 40, None) == bpt.BPT_EINVAL


def test_backward_and_headchunk_reject_missing_buffers(built):
    L = bpt.lib()
    c = bpt.make_config(presets.C1)
    p = 1 << 20
    w = bpt.BptWeights(*([p] * len(bpt.WEIGHT_FIELDS)))
    g = bpt.BptGrads(*([p] * len(bpt.WEIGHT_FIELDS)))
    args = (ctypes.byref(c), ctypes.byref(w), p, p, p, p, ctypes.byref(g), p, 1 << 40, None)
    # every argument present but the workspace too small: ENOSPC, so the
    # pointer checks below are what reject
    small = list(args)
    small[8] = 1024
    assert L.bpt_layer_bwd(*small) == bpt.BPT_ENOSPC
    for i in (2, 3, 4, 5, 7):                     # x, saved, dy, dx, ws
        a = list(args)
        a[i] = None
        assert L.bpt_layer_bwd(*a) == bpt.BPT_EINVAL, i
    gp = [p] * len(bpt.WEIGHT_FIELDS)
    gp[bpt.WEIGHT_FIELDS.index("w1")] = None      # a weight gradient the layer has
    a = list(args)
    a[6] = ctypes.byref(bpt.BptGrads(*gp))
    assert L.bpt_layer_bwd(*a) == bpt.BPT_EINVAL
    wp = [p] * len(bpt.WEIGHT_FIELDS)
    wp[bpt.WEIGHT_FIELDS.index("wk")] = None
    assert L.bpt_attn_headchunk(ctypes.byref(c), ctypes.byref(bpt.BptWeights(*wp)), p, p, None, p, 1 << 40,
                                None) == bpt.BPT_EINVAL
    assert L.bpt_attn_headchunk(ctypes.byref(c), ctypes.byref(w), p, p, None, p, 1024, None) == bpt.BPT_ENOSPC


def test_profiler_calls_on_the_host(built):
    """With nothing recorded the profiler needs no device: enable, list and
    collect return empty results; bad arguments are rejected."""
    L = bpt.lib()
    bpt.bpt_profile_enable(True)
    assert bpt.bpt_profile_list() == []
    assert all(v["launches"] == 0 and v["ms"] == 0 for v in bpt.bpt_profile_collect().values())
    bpt.bpt_profile_enable(False)
    n = ctypes.c_double * 1
    assert L.bpt_profile_collect(0, n(), n(), n(), (ctypes.c_int * 1)()) == bpt.BPT_EINVAL
    assert L.bpt_profile_collect(1, None, n(), n(), (ctypes.c_int * 1)()) == bpt.BPT_EINVAL
    assert L.bpt_profile_list(-1, None, None, None, None) == -bpt.BPT_EINVAL
    assert L.bpt_profile_list(4, None, None, None, None) == -bpt.BPT_EINVAL
    assert L.bpt_profile_list(0, None, None, None, None) == 0


def test_product_never_reaches_the_oracle():
    """The package and its CUDA sources import, load or name nothing under
    oracle/: the oracle is test infrastructure, never a fallback."""
    pkg = os.path.join(ROOT, "blockwise_attention_ffn_gb300")
    for dirpath, _, files in os.walk(pkg):
        if "_build" in dirpath or "__pycache__" in dirpath:
            continue
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h")):
                txt = open(os.path.join(dirpath, fn)).read()
                assert not re.search(r"^\s*(from|import)\s+oracle\b", txt, flags=re.M), fn
                assert "oracle/" not in txt and "oracle." not in txt, fn


def test_missing_library_raises(monkeypatch):
    """No silent fallback: without libbpt.so the binding refuses to run."""
    monkeypatch.setattr(bpt, "_lib", None)
    monkeypatch.setattr(bpt, "LIB_PATH", os.path.join(ROOT, "no-such-dir", "libbpt.so"))
    with pytest.raises(RuntimeError):
        bpt.lib()
    with pytest.raises(RuntimeError):
        bpt.bpt_workspace_bytes(presets.C1, bpt.BPT_PASS_FWD)


def test_schedule_options_sizes(built):
    """The interleaved order keeps every key/value head resident (forward and
    head-chunk workspaces grow by the difference, plus a copy of Wq in stage
    order); the save policies grow the saved bytes by Q/K/V and O of every
    row and leave the forward's workspace size (with or without a saved
    buffer) alone, while the backward's shrinks."""
    c5 = presets.C5                      # 32 over 8 heads of 128, U = 8
    il = c5.with_(stage_order=bpt.BPT_STAGE_INTERLEAVED)
    rows, d, h, H, Hk, U = c5.b * c5.s, c5.head_dim, c5.h, c5.n_heads, c5.n_kv_heads, c5.head_chunk

    def up(n):
        return (n + 255) // 256 * 256
    contiguous_stage = up(rows * (U + 2 * U // (H // Hk)) * d * 2)
    interleaved_stage = up(rows * (U + 2 * Hk) * d * 2)
    wq_copy = up(H * d * h * 2) + up(H * d * 2)
    assert (bpt.bpt_workspace_bytes(il, bpt.BPT_PASS_HEADCHUNK) ==
            bpt.bpt_workspace_bytes(c5, bpt.BPT_PASS_HEADCHUNK) - contiguous_stage + interleaved_stage + wq_copy)
    assert (bpt.bpt_workspace_bytes(il, bpt.BPT_PASS_FWD) ==
            bpt.bpt_workspace_bytes(c5, bpt.BPT_PASS_FWD) - contiguous_stage + interleaved_stage + wq_copy)
    assert bpt.bpt_workspace_bytes(il, bpt.BPT_PASS_BWD) == bpt.bpt_workspace_bytes(c5, bpt.BPT_PASS_BWD)
    c3 = presets.C3
    lse = bpt.bpt_saved_bytes(c3)
    qkv = up(c3.s * (c3.n_heads + 2 * c3.n_kv_heads) * c3.head_dim * 2)
    o = up(c3.s * c3.n_heads * c3.head_dim * 2)
    assert bpt.bpt_saved_bytes(c3.with_(save_policy=1)) == up(lse) + qkv
    assert bpt.bpt_saved_bytes(c3.with_(save_policy=2)) == up(lse) + qkv + o
    for p in (1, 2):
        assert bpt.bpt_workspace_bytes(c3.with_(save_policy=p), 0) == bpt.bpt_workspace_bytes(c3, 0)
    assert bpt.bpt_workspace_bytes(c3.with_(save_policy=1), 1) == bpt.bpt_workspace_bytes(c3, 1) - qkv
    assert bpt.bpt_workspace_bytes(c3.with_(save_policy=2), 1) == bpt.bpt_workspace_bytes(c3, 1) - qkv - o
