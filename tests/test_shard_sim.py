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
