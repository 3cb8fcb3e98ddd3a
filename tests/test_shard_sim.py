"""The layer sharded by sequence position over two gloo ranks on CPU (the
sharded schedule a multi-device run would use: K/V all-gathered, partial
dK/dV reduce-scattered, weight gradients all-reduced, zigzag row order)
equals the unsharded fp64 oracle.  No GPU: the library itself runs on one."""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as tdist
import torch.multiprocessing as mp

from oracle import ref, sharded
from oracle.ref import LayerCfg
from tests.oracle_helpers import rand_layer

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

CASES = {
    "gpt causal": LayerCfg(s=16, h=16, n_heads=2, n_kv_heads=2, head_dim=8, ffn_dim=24),
    "llama gqa rope": LayerCfg(s=16, h=16, n_heads=4, n_kv_heads=2, head_dim=4, ffn_dim=24, norm=1, act=2,
                               has_bias=False, rope_base=10000.0),
    "gpt b2 noncausal": LayerCfg(s=8, h=16, n_heads=2, n_kv_heads=1, head_dim=8, ffn_dim=24, b=2,
                                 causal=False, act=1),
}


class LocalComm:
    """One rank alone: the collectives are the identity."""
    rank = 0

    @staticmethod
    def all_gather(a):
        return [np.asarray(a)]

    @staticmethod
    def all_reduce(a):
        return np.array(a, copy=True)


class GlooComm:
    def __init__(self, rank, world):
        self.rank, self.world = rank, world

    def all_gather(self, a):
        t = torch.from_numpy(np.ascontiguousarray(a, np.float64))
        out = [torch.empty_like(t) for _ in range(self.world)]
        tdist.all_gather(out, t)
        return [o.numpy() for o in out]

    def all_reduce(self, a):
        t = torch.from_numpy(np.array(a, np.float64, copy=True))
        tdist.all_reduce(t)
        return t.numpy()


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    tdist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        comm = GlooComm(rank, world)
        for i, (name, cfg) in enumerate(CASES.items()):
            x, W, dy = rand_layer(cfg, seed=70 + i)
            pos = sharded.zigzag_rows(cfg.s, world, rank)
            y = sharded.rank_layer_forward(x[:, pos], pos, W, cfg, comm)
            dx, grads = sharded.rank_layer_backward(x[:, pos], pos, W, dy[:, pos], cfg, comm)
            np.savez(os.path.join(out_dir, f"r{rank}_c{i}.npz"), pos=pos, y=y, dx=dx,
                     **{"g_" + k: v for k, v in grads.items()})
    finally:
        tdist.destroy_process_group()


def _close(got, want, what):
    if np.linalg.norm(want) < 1e-9:
        # the key-bias gradient is zero in exact arithmetic (softmax is
        # shift-invariant along a row); both sides hold rounding noise
        assert np.max(np.abs(got)) <= 1e-12, f"{what}: max |got| {np.max(np.abs(got)):.2e}"
        return
    err = np.linalg.norm(got - want) / np.linalg.norm(want)
    assert err <= 1e-12, f"{what}: relative error {err:.2e}"


def test_two_ranks_equal_the_unsharded_layer(tmp_path):
    world = 2
    mp.spawn(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    for i, (name, cfg) in enumerate(CASES.items()):
        x, W, dy = rand_layer(cfg, seed=70 + i)
        y_ref = ref.layer_forward(x, W, cfg)
        dx_ref, g_ref = ref.layer_backward(x, W, dy, cfg)
        y = np.zeros_like(y_ref)
        dx = np.zeros_like(dx_ref)
        for r in range(world):
            f = np.load(tmp_path / f"r{r}_c{i}.npz")
            y[:, f["pos"]] = f["y"]
            dx[:, f["pos"]] = f["dx"]
            for k, v in g_ref.items():
                _close(f["g_" + k], v, f"{name}: d{k} on rank {r}")
        _close(y, y_ref, f"{name}: y")
        _close(dx, dx_ref, f"{name}: dx")


@pytest.mark.parametrize("name", list(CASES))
def test_one_rank_is_the_unsharded_layer(name):
    cfg = CASES[name]
    x, W, dy = rand_layer(cfg, seed=80)
    pos = sharded.zigzag_rows(cfg.s, 1, 0)
    assert np.array_equal(pos, np.arange(cfg.s))
    _close(sharded.rank_layer_forward(x, pos, W, cfg, LocalComm), ref.layer_forward(x, W, cfg), "y")
    dx, g = sharded.rank_layer_backward(x, pos, W, dy, cfg, LocalComm)
    dx_ref, g_ref = ref.layer_backward(x, W, dy, cfg)
    _close(dx, dx_ref, "dx")
    for k, v in g_ref.items():
        _close(g[k], v, k)


@pytest.mark.parametrize("P", [1, 2, 3, 4, 8])
def test_zigzag_rows_partition_the_sequence_with_equal_causal_work(P):
    s = 2 * P * 5
    rows = [sharded.zigzag_rows(s, P, r) for r in range(P)]
    assert np.array_equal(np.sort(np.concatenate(rows)), np.arange(s))
    # chunk r and chunk 2P-1-r together hold the same number of unmasked
    # (query, key) pairs for every r: s(s+1)/2 split evenly
    work = [sharded.causal_pairs(r) for r in rows]
    assert work == [s * (s + 1) // 2 // P] * P
    # a contiguous split would not be balanced
    if P > 1:
        c = s // P
        contiguous = [sharded.causal_pairs(np.arange(r * c, (r + 1) * c)) for r in range(P)]
        assert len(set(contiguous)) == P


class ThreadComm:
    """Ranks as threads of one process; `broken` plants a mistake in one
    collective: 'gather' hands each rank only its own K/V, 'reduce' skips the
    sum over ranks (each rank keeps its own partial dK/dV and weight
    gradients)."""

    def __init__(self, rank, world, box, barrier, broken=None):
        self.rank, self.world, self.box, self.barrier, self.broken = rank, world, box, barrier, broken

    def _exchange(self, a):
        self.barrier.wait()
        self.box[self.rank] = np.array(a, np.float64, copy=True)
        self.barrier.wait()
        got = [self.box[r] for r in range(self.world)]
        self.barrier.wait()
        return got

    def all_gather(self, a):
        got = self._exchange(a)
        return [got[self.rank]] if self.broken == "gather" else got

    def all_reduce(self, a):
        got = self._exchange(a)
        return got[self.rank] if self.broken == "reduce" else np.sum(got, axis=0)


def _run_threads(cfg, world, broken, seed, backward=True):
    import threading
    x, W, dy = rand_layer(cfg, seed=seed)
    # a rank that fails breaks the barrier for the others instead of leaving
    # them waiting
    box, barrier, out, errs = {}, threading.Barrier(world, timeout=60), {}, []

    def work(r):
        try:
            comm = ThreadComm(r, world, box, barrier, broken)
            pos = sharded.zigzag_rows(cfg.s, world, r)
            y = sharded.rank_layer_forward(x[:, pos], pos, W, cfg, comm)
            dx, g = (sharded.rank_layer_backward(x[:, pos], pos, W, dy[:, pos], cfg, comm) if backward
                     else (np.zeros_like(y), {}))
            out[r] = (pos, y, dx, g)
        except Exception as e:  # noqa: BLE001 - re-raised below
            errs.append(e)
            barrier.abort()

    ts = [threading.Thread(target=work, args=(r,)) for r in range(world)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    if errs:
        raise errs[0]
    y = np.zeros((cfg.b, cfg.s, cfg.h))
    dx = np.zeros_like(y)
    for pos, yr, dxr, _ in out.values():
        y[:, pos] = yr
        dx[:, pos] = dxr
    return (x, W, dy), y, dx, out[0][3]


def _rel(a, b):
    return np.linalg.norm(a - b) / np.linalg.norm(b)


@pytest.mark.parametrize("world", [2, 4])
def test_thread_ranks_equal_the_unsharded_layer(world):
    cfg = CASES["gpt causal"]
    (x, W, dy), y, dx, g0 = _run_threads(cfg, world, None, seed=95)
    _close(y, ref.layer_forward(x, W, cfg), "y")
    dx_ref, g_ref = ref.layer_backward(x, W, dy, cfg)
    _close(dx, dx_ref, "dx")
    for k, v in g_ref.items():
        _close(g0[k], v, k)


def test_planted_exchange_mistakes_are_caught():
    """Without the K/V all-gather the forward is wrong; without the sum over
    ranks the backward is wrong: both exchanges are needed, and the pins
    above would see either one missing."""
    cfg = CASES["gpt causal"]
    (x, W, dy), y, _, _ = _run_threads(cfg, 2, "gather", seed=96, backward=False)
    assert _rel(y, ref.layer_forward(x, W, cfg)) > 1e-3
    (x, W, dy), y, dx, g0 = _run_threads(cfg, 2, "reduce", seed=97)
    _close(y, ref.layer_forward(x, W, cfg), "y")  # the forward needs no sum
    dx_ref, g_ref = ref.layer_backward(x, W, dy, cfg)
    assert _rel(dx, dx_ref) > 1e-3
    assert _rel(g0["wq"], g_ref["wq"]) > 1e-3
