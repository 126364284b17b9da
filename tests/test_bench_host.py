"""Host-side logic of bench.py for N > 1 ranks (replicas): the timing gather,
max-over-ranks aggregation and the rank-0-only reference arm, on 2 gloo ranks
on the CPU."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        times = bench.gather_floats(10.0 + 5.0 * rank, world)      # rank 1 is the slow one
        value, tmax = bench.aggregate(times, [1e9] * world)
        bench.barrier(world)
        w, r, lr = bench.dist_env()
        out.put((rank, times, value, tmax, (w, r, lr)))
    finally:
        dist.destroy_process_group()


def test_two_rank_gather_takes_the_slowest_rank_and_sums_the_bytes():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, times, value, tmax, env in sorted(res):
        assert times == [10.0, 15.0]                 # every rank sees every rank's time
        assert tmax == 15.0                          # the slowest rank's time
        assert value == pytest.approx(2e9 / 15e-3 / 1e9)   # all ranks' bytes over it
        assert env == (2, rank, rank)


def test_reference_arm_is_rank_zero_only(monkeypatch):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")

    class Args:
        gpus, steps, warmup = 2, 1, 3

    # a non-zero rank exits 0 without touching the oracle
    monkeypatch.setattr(bench, "oracle_sample", lambda *a, **k: pytest.fail("rank 1 did work"))
    assert bench.run_reference(Args()) == 0


def test_single_rank_aggregate():
    value, t = bench.aggregate([4.0], [8e9])
    assert t == 4.0 and value == pytest.approx(2000.0)


def test_reference_arm_prints_the_contract_line(monkeypatch, capsys):
    # the oracle timed on the host cores: one JSON line with the contract's
    # keys (a tiny row sample here, so the test stays fast)
    import json
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    real = bench.oracle_sample
    monkeypatch.setattr(bench, "oracle_sample", lambda rows, seed=4242: real(min(rows, 8), seed))

    class Args:
        gpus, steps, warmup = 1, 2, 3

    assert bench.run_reference(Args()) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC and line["unit"] == "GB/s"
    assert line["higher_is_better"] is True and line["steps"] == 2 and line["warmup"] == 3
    assert line["config"]["workload"] == bench.WORKLOAD
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"] > 0
    assert line["e2e"] == {"value": line["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
