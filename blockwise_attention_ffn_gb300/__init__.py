"""Python binding of libbpt (include/bpt.h): argument marshalling only.

Every step of the layer runs in the CUDA library; this module turns torch
tensors into the pointers and structs the C ABI takes.  PyTorch supplies
device memory and streams.  There is no fallback: if the library is missing
or fails to load, importing the binding's entry points raises.

Entry points keep the C names: bpt_layer_fwd, bpt_layer_bwd,
bpt_attn_headchunk, bpt_attention_fwd, bpt_attention_bwd, bpt_attention_bwd_noalloc,
bpt_lm_loss_fwd, bpt_lm_loss_bwd, bpt_lm_workspace_bytes,
bpt_workspace_bytes, bpt_saved_bytes, bpt_attention_bwd_workspace_bytes,
bpt_status_string, bpt_last_device_error, bpt_check_device_range, bpt_watchdog_selftest,
bpt_profile_enable, bpt_profile_collect, bpt_profile_list.  The layer stack
with a checkpoint every k layers is in :mod:`.stack` (a scheduler over
bpt_layer_fwd / bpt_layer_bwd).
"""
from __future__ import annotations

import ctypes
import os

from .presets import PRESETS, LayerConfig  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libbpt.so")

BPT_OK, BPT_EINVAL, BPT_ENOSPC, BPT_ECUDA, BPT_ETIMEOUT, BPT_EUNSUPPORTED = range(6)
BPT_PASS_FWD, BPT_PASS_BWD, BPT_PASS_HEADCHUNK = 0, 1, 2
BPT_STAGE_CONTIGUOUS, BPT_STAGE_INTERLEAVED = 0, 1
BPT_SAVE_NOTHING, BPT_SAVE_PROJECTIONS, BPT_SAVE_ATTN_OUT = 0, 1, 2
BPT_FLAG_ACCUM_GRADS = 1
BPT_FLAG_ONE_STREAM = 2
BPT_FLAG_DETERMINISTIC = 4
BPT_FLAG_DEBUG_CHECKS = 8

WEIGHT_FIELDS = ("ln1_w", "ln1_b", "wq", "bq", "wk", "bk", "wv", "bv", "wo", "bo",
                 "ln2_w", "ln2_b", "w1", "b1", "w2", "b2", "w3")


class BptConfig(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "b", "s", "h", "n_heads", "n_kv_heads", "head_dim", "ffn_dim",
        "q_block", "kv_block", "ffn_block", "head_chunk", "causal", "norm", "act", "has_bias")] + \
        [("norm_eps", ctypes.c_float), ("flags", ctypes.c_int32), ("rope_base", ctypes.c_float),
         ("stage_order", ctypes.c_int32), ("save_policy", ctypes.c_int32)]


class BptWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in WEIGHT_FIELDS]


class BptGrads(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in WEIGHT_FIELDS]


class BptLmConfig(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("n", "h", "vocab", "vocab_block", "flags")]


class BptError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {bpt_status_string(status)} (status {status})")


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libbpt.so (raises if it is missing: build it first with
    ``python -m blockwise_attention_ffn_gb300.build`` or __graft_entry__.build())."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libbpt.so not built ({LIB_PATH} missing)")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        cfgp = ctypes.POINTER(BptConfig)
        L.bpt_workspace_bytes.argtypes = [cfgp, i32]
        L.bpt_workspace_bytes.restype = sz
        L.bpt_saved_bytes.argtypes = [cfgp]
        L.bpt_saved_bytes.restype = sz
        L.bpt_layer_fwd.argtypes = [cfgp, ctypes.POINTER(BptWeights), vp, vp, vp, vp, sz, vp]
        L.bpt_layer_fwd.restype = i32
        L.bpt_layer_bwd.argtypes = [cfgp, ctypes.POINTER(BptWeights), vp, vp, vp, vp,
                                    ctypes.POINTER(BptGrads), vp, sz, vp]
        L.bpt_layer_bwd.restype = i32
        L.bpt_attn_headchunk.argtypes = [cfgp, ctypes.POINTER(BptWeights), vp, vp, vp, vp, sz, vp]
        L.bpt_attn_headchunk.restype = i32
        L.bpt_attention_fwd.argtypes = [cfgp, vp, vp, vp, vp]
        L.bpt_attention_fwd.restype = i32
        L.bpt_attention_bwd_workspace_bytes.argtypes = [cfgp]
        L.bpt_attention_bwd_workspace_bytes.restype = sz
        L.bpt_attention_bwd.argtypes = [cfgp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.bpt_attention_bwd.restype = i32
        L.bpt_attention_bwd_noalloc.argtypes = [cfgp, vp, vp, vp, vp, vp, vp]
        L.bpt_attention_bwd_noalloc.restype = i32
        L.bpt_status_string.argtypes = [i32]
        L.bpt_status_string.restype = ctypes.c_char_p
        L.bpt_last_device_error.argtypes = [vp, ctypes.POINTER(ctypes.c_int)]
        L.bpt_last_device_error.restype = i32
        lmp = ctypes.POINTER(BptLmConfig)
        L.bpt_lm_workspace_bytes.argtypes = [lmp, i32]
        L.bpt_lm_workspace_bytes.restype = sz
        L.bpt_lm_loss_fwd.argtypes = [lmp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.bpt_lm_loss_fwd.restype = i32
        L.bpt_lm_loss_bwd.argtypes = [lmp, vp, vp, vp, vp, ctypes.c_float, vp, vp, vp, sz, vp]
        L.bpt_lm_loss_bwd.restype = i32
        L.bpt_check_device_range.argtypes = [vp, sz]
        L.bpt_check_device_range.restype = i32
        L.bpt_watchdog_selftest.argtypes = [vp]
        L.bpt_watchdog_selftest.restype = i32
        L.bpt_profile_enable.argtypes = [i32]
        L.bpt_profile_enable.restype = i32
        dp = ctypes.POINTER(ctypes.c_double)
        L.bpt_profile_collect.argtypes = [i32, dp, dp, dp, ctypes.POINTER(ctypes.c_int)]
        L.bpt_profile_collect.restype = i32
        L.bpt_profile_list.argtypes = [i32, ctypes.POINTER(ctypes.c_int), dp, dp, dp]
        L.bpt_profile_list.restype = i32
        _lib = L
    return _lib


# ------------------------------------------------------------------ marshalling

def make_config(c) -> BptConfig:
    """BptConfig from a LayerConfig (or any object with the same fields)."""
    return BptConfig(c.b, c.s, c.h, c.n_heads, c.n_kv_heads, c.head_dim, c.ffn_dim, c.q_block,
                     c.kv_block, c.ffn_block, c.head_chunk, c.causal, c.norm, c.act, c.has_bias,
                     c.norm_eps, c.flags, float(getattr(c, "rope_base", 0.0)),
                     int(getattr(c, "stage_order", 0)), int(getattr(c, "save_policy", 0)))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def make_weights(w: dict) -> BptWeights:
    return BptWeights(*[(None if w.get(n) is None else w[n].data_ptr()) for n in WEIGHT_FIELDS])


def make_grads(g: dict) -> BptGrads:
    return BptGrads(*[(None if g.get(n) is None else g[n].data_ptr()) for n in WEIGHT_FIELDS])


def _stream(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _check(rc, where):
    if rc != BPT_OK:
        raise BptError(rc, where)


def bpt_status_string(status: int) -> str:
    return lib().bpt_status_string(int(status)).decode()


def bpt_workspace_bytes(cfg, pass_: int) -> int:
    return int(lib().bpt_workspace_bytes(ctypes.byref(make_config(cfg)), int(pass_)))


def bpt_saved_bytes(cfg) -> int:
    return int(lib().bpt_saved_bytes(ctypes.byref(make_config(cfg))))


def bpt_attention_bwd_workspace_bytes(cfg) -> int:
    return int(lib().bpt_attention_bwd_workspace_bytes(ctypes.byref(make_config(cfg))))


def bpt_layer_fwd(cfg, weights: dict, x, y, saved, ws, stream=None) -> None:
    c = make_config(cfg)
    w = make_weights(weights)
    rc = lib().bpt_layer_fwd(ctypes.byref(c), ctypes.byref(w), _ptr(x), _ptr(y), _ptr(saved),
                             _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))
    _check(rc, "bpt_layer_fwd")


def bpt_layer_bwd(cfg, weights: dict, x, saved, dy, dx, grads: dict, ws, stream=None) -> None:
    c = make_config(cfg)
    w = make_weights(weights)
    g = make_grads(grads)
    rc = lib().bpt_layer_bwd(ctypes.byref(c), ctypes.byref(w), _ptr(x), _ptr(saved), _ptr(dy),
                             _ptr(dx), ctypes.byref(g), _ptr(ws), ws.numel() * ws.element_size(),
                             _stream(stream))
    _check(rc, "bpt_layer_bwd")


def bpt_attn_headchunk(cfg, weights: dict, xn, o, lse, ws, stream=None) -> None:
    c = make_config(cfg)
    w = make_weights(weights)
    rc = lib().bpt_attn_headchunk(ctypes.byref(c), ctypes.byref(w), _ptr(xn), _ptr(o), _ptr(lse),
                                  _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))
    _check(rc, "bpt_attn_headchunk")


def bpt_attention_fwd(cfg, qkv, o, lse, stream=None) -> None:
    c = make_config(cfg)
    rc = lib().bpt_attention_fwd(ctypes.byref(c), _ptr(qkv), _ptr(o), _ptr(lse), _stream(stream))
    _check(rc, "bpt_attention_fwd")


def bpt_attention_bwd(cfg, qkv, o, lse, dout, dqkv, ws, stream=None) -> None:
    c = make_config(cfg)
    rc = lib().bpt_attention_bwd(ctypes.byref(c), _ptr(qkv), _ptr(o), _ptr(lse), _ptr(dout),
                                 _ptr(dqkv), _ptr(ws), ws.numel() * ws.element_size(),
                                 _stream(stream))
    _check(rc, "bpt_attention_bwd")


def make_lm_config(c) -> BptLmConfig:
    """BptLmConfig from an LmConfig (or any object with n, h, vocab,
    vocab_block and flags)."""
    return BptLmConfig(c.n, c.h, c.vocab, c.vocab_block, c.flags)


def bpt_lm_workspace_bytes(cfg, pass_: int) -> int:
    return int(lib().bpt_lm_workspace_bytes(ctypes.byref(make_lm_config(cfg)), int(pass_)))


def bpt_lm_loss_fwd(cfg, x, w, targets, loss, lse, ws, stream=None) -> None:
    """Mean token cross-entropy of x [n, h] through w [V, h] against int32
    targets [n]: writes loss (one fp32 element) and lse [n] (optional)."""
    c = make_lm_config(cfg)
    rc = lib().bpt_lm_loss_fwd(ctypes.byref(c), _ptr(x), _ptr(w), _ptr(targets), _ptr(loss), _ptr(lse),
                               _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))
    _check(rc, "bpt_lm_loss_fwd")


def bpt_lm_loss_bwd(cfg, x, w, targets, lse, dloss, dx, dw, ws, stream=None) -> None:
    """Gradients of dloss * loss: dx [n, h] bf16 and dw [V, h] fp32."""
    c = make_lm_config(cfg)
    rc = lib().bpt_lm_loss_bwd(ctypes.byref(c), _ptr(x), _ptr(w), _ptr(targets), _ptr(lse), float(dloss),
                               _ptr(dx), _ptr(dw), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))
    _check(rc, "bpt_lm_loss_bwd")


BPT_LM_BAD_TARGET_SITE = 950
NOALLOC_SCRATCH_BYTES = 192 * 1024 * 1024


def bpt_attention_bwd_noalloc(cfg, qkv, o, lse, dout, dqkv, stream=None) -> None:
    """bpt_attention_bwd for callers that cannot allocate device memory at
    call time: the scratch (bpt_attention_bwd_workspace_bytes(cfg) =
    24*b*H*s_pad bytes: the fp32 dO.O sums and -LSE*log2(e), and a 16-byte
    bf16 row of both per query) is a fixed array inside the library (at most
    NOALLOC_SCRATCH_BYTES; larger problems raise BptError with BPT_ENOSPC).
    Calls that overlap on the GPU share that array and race: serialise them."""
    c = make_config(cfg)
    rc = lib().bpt_attention_bwd_noalloc(ctypes.byref(c), _ptr(qkv), _ptr(o), _ptr(lse), _ptr(dout),
                                         _ptr(dqkv), _stream(stream))
    _check(rc, "bpt_attention_bwd_noalloc")


def bpt_check_device_range(ptr: int, nbytes: int) -> int:
    """BPT_OK if [ptr, ptr + nbytes) lies inside one device allocation of the
    current device, else BPT_EINVAL (launches nothing)."""
    return int(lib().bpt_check_device_range(ctypes.c_void_p(ptr), int(nbytes)))


def bpt_last_device_error(stream=None):
    """(status, detail) after synchronising the stream; clears the word."""
    d = ctypes.c_int(0)
    rc = lib().bpt_last_device_error(_stream(stream), ctypes.byref(d))
    return int(rc), int(d.value)


BPT_WATCHDOG_SELFTEST_SITE = 900


def bpt_watchdog_selftest(stream=None) -> None:
    """Launch the watchdog self-test: a wait on a barrier nothing signals runs
    out after about 2 s and is recorded as (BPT_ETIMEOUT,
    BPT_WATCHDOG_SELFTEST_SITE), which bpt_last_device_error() then reads."""
    _check(lib().bpt_watchdog_selftest(_stream(stream)), "bpt_watchdog_selftest")


PROF_KINDS = ("gemm", "attn_fwd", "attn_bwd", "norm", "misc")


def bpt_profile_enable(on: bool) -> None:
    _check(lib().bpt_profile_enable(1 if on else 0), "bpt_profile_enable")


def bpt_profile_collect() -> dict:
    """{kind: dict(ms=..., flops=..., bytes=..., launches=...)} since the
    last collect (synchronises on the recorded events)."""
    n = len(PROF_KINDS)
    ms, fl, by = (ctypes.c_double * n)(), (ctypes.c_double * n)(), (ctypes.c_double * n)()
    la = (ctypes.c_int * n)()
    _check(lib().bpt_profile_collect(n, ms, fl, by, la), "bpt_profile_collect")
    return {k: dict(ms=ms[i], flops=fl[i], bytes=by[i], launches=la[i])
            for i, k in enumerate(PROF_KINDS)}


def bpt_profile_list(max_launches: int = 4096) -> list:
    """[(kind, flops, bytes, ms)] of every launch recorded since the last
    collect, in launch order (does not clear the record)."""
    n = max_launches
    kd = (ctypes.c_int * n)()
    fl, by, ms = (ctypes.c_double * n)(), (ctypes.c_double * n)(), (ctypes.c_double * n)()
    got = lib().bpt_profile_list(n, kd, fl, by, ms)
    if got < 0:
        _check(-got, "bpt_profile_list")
    return [(PROF_KINDS[kd[i]], fl[i], by[i], ms[i]) for i in range(got)]


# ------------------------------------------------------------------ helpers

def s_pad(cfg) -> int:
    return (cfg.s + 127) // 128 * 128


def alloc_bytes(n: int, device="cuda"):
    """A 256-byte aligned uint8 device buffer of at least n bytes."""
    import torch
    return torch.empty(max(int(n), 256), dtype=torch.uint8, device=device)


def alloc_grads(weights: dict, device="cuda") -> dict:
    import torch
    return {k: (None if v is None else torch.empty(v.shape, dtype=torch.float32, device=device))
            for k, v in weights.items()}
