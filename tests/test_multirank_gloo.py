"""The benchmark's multi-rank control plane with world size 2 on gloo (CPU).

Under torchrun every rank runs an independent replica of the step on its own
GPU.  The ranks share only a barrier and the max / sum of their timings;
there is no data-path collective.  This runs that plumbing in two CPU
processes: the max over ranks of per-rank step times, and the sum of the
parameters each replica processed.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port),
                       "WORLD_SIZE": str(world), "RANK": str(rank), "LOCAL_RANK": str(rank)})
    import bench
    w, r, local = bench.dist_env()
    assert (w, r, local) == (world, rank, rank)
    g = bench.Group(world)
    g.barrier()
    ms = g.max(5.0 + rank)            # slower rank decides the step time
    params = g.sum(1_000_000_000.0)   # every replica processed the whole vector
    g.barrier()
    g.close()
    out.put((rank, ms, params))


@pytest.mark.parametrize("world", [2])
def test_replica_timing_aggregation(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, ms, params in got:
        assert ms == 5.0 + world - 1
        assert params == world * 1e9


def test_reference_arm_only_rank0_prints(capsys, monkeypatch):
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    bench.main(["--impl", "reference", "--steps", "1", "--warmup", "0"])
    assert capsys.readouterr().out == ""


def test_reference_arm_prints_the_contract_line(capsys, monkeypatch):
    """Rank 0 of the reference arm (the oracle on the host cores) prints one
    JSON line with the benchmark contract's keys, on the default workload."""
    import json
    import bench
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    bench.main(["--impl", "reference", "--steps", "1", "--warmup", "0"])
    lines = [ln for ln in capsys.readouterr().out.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "params/s"
    assert d["config"]["workload"] == "flat1b_n8" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
