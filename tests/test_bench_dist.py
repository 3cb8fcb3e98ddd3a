"""The multi-rank host logic of bench.py on CPU: two gloo ranks, as torchrun
would launch them with one rank per GPU.  The layer step shards by batch (each
rank a full replica on its own seeded batch), so the only cross-rank steps
are the barrier-bracketed timing, its max over ranks and the whole-job
aggregate, all checked here without a GPU."""
import json
import os
import socket
import sys

import pytest
import torch.distributed as tdist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    from blockwise_attention_ffn_gb300.presets import C3
    tdist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = bench.dist_setup()
        tdist.barrier()
        ms = 10.0 + 5.0 * rank            # the ranks finish at different times
        slowest = bench.max_over_ranks(ms, ws, "cpu")
        res = {"dist": [ws, r, local], "slowest": slowest,
               "value": bench.job_throughput(1e12, ws, slowest),
               "seed": bench.rank_seed(C3, r), "reports": bench.reports(r)}
        tdist.barrier()
    finally:
        tdist.destroy_process_group()
    with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
        json.dump(res, f)


def test_two_gloo_ranks_time_max_and_aggregate(tmp_path):
    world = 2
    mp.spawn(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    res = [json.load(open(tmp_path / f"r{r}.json")) for r in range(world)]
    assert [r["dist"] for r in res] == [[2, 0, 0], [2, 1, 1]]
    # every rank sees the slowest rank's time
    assert res[0]["slowest"] == res[1]["slowest"] == 15.0
    # whole-job throughput: both ranks' work over the slowest time
    assert res[0]["value"] == pytest.approx(2 * 1e12 / 15e-3 / 1e12)
    # each replica draws its own batch; only rank 0 prints
    assert res[0]["seed"] != res[1]["seed"]
    assert [r["reports"] for r in res] == [True, False]


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import argparse

    import bench
    from blockwise_attention_ffn_gb300.presets import C3
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    args = argparse.Namespace(gpus=2, steps=1, warmup=3, ref_rows=64)
    assert bench.run_reference(args, C3) == 0
    assert capsys.readouterr().out == ""   # rank 1 does no work and prints nothing


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(12.5, 1) == 12.5
    assert bench.job_throughput(2e12, 1, 10.0) == pytest.approx(200.0)


def _failing_worker(rank, world, port, out_dir, mode):
    """Rank 1 fails before the timing barrier -- it exits, or it stalls past
    the group's timeout without joining; rank 0 must get an error from that
    barrier within the (short) timeout instead of waiting."""
    import time
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    bench.init_group("gloo", timeout_s=5)
    if rank == 1:
        if mode == "stall":
            time.sleep(8)    # never joins within the 5 s timeout
        os._exit(3)          # the simulated failure: no barrier, no clean shutdown
    t0 = time.perf_counter()
    try:
        tdist.barrier()
        outcome = "returned"
    except Exception as e:  # noqa: BLE001 - any error is the detection
        outcome = type(e).__name__
    with open(os.path.join(out_dir, "r0.json"), "w") as f:
        json.dump({"outcome": outcome, "seconds": time.perf_counter() - t0}, f)
    os._exit(0)


@pytest.mark.parametrize("mode", ["exit", "stall"])
def test_failed_rank_is_detected_within_the_timeout(tmp_path, mode):
    world = 2
    ctx = mp.get_context("spawn")
    port = _free_port()
    procs = [ctx.Process(target=_failing_worker, args=(r, world, port, str(tmp_path), mode)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert not p.is_alive(), "a rank hung"
    res = json.load(open(tmp_path / "r0.json"))
    assert res["outcome"] != "returned", res
    assert res["seconds"] < 12, res


def test_reference_arm_line_carries_the_contract_keys(monkeypatch, capsys):
    """One rank: the oracle arm prints one JSON line with the keys of the
    bench contract, its own cpu_baseline and an e2e with no copies."""
    import argparse

    import bench
    from blockwise_attention_ffn_gb300.presets import C3
    monkeypatch.setenv("WORLD_SIZE", "1")
    monkeypatch.setenv("RANK", "0")
    args = argparse.Namespace(gpus=1, steps=1, warmup=0, ref_rows=32)
    assert bench.run_reference(args, C3) == 0
    lines = [ln for ln in capsys.readouterr().out.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["value"] > 0
    assert d["config"]["workload"] == C3.name
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
