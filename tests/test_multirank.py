"""The N>1 bench path on CPU: replicas with gloo, max-over-ranks timing, rank-0-only output."""
import json
import os
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
from workloads import make_workload  # noqa: E402


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks(10.0 + 5.0 * rank, "cpu")
        dist.barrier()
        out[rank] = got
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        port = 29500 + os.getpid() % 1000
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
        assert all(p.exitcode == 0 for p in procs)
        assert dict(out) == {0: 15.0, 1: 15.0}


def test_max_over_ranks_single_process():
    assert bench.max_over_ranks(3.5, "cpu") == 3.5


def test_ranks_serve_distinct_batches():
    """Weak scaling: each rank's batch is its own seeded draw of the same shapes."""
    a = make_workload(2, seed=0, T=2048)
    b = make_workload(2, seed=1, T=2048)
    assert a.K.shape == b.K.shape and a.q.shape == b.q.shape
    assert not (a.K == b.K).all()


def test_reference_arm_prints_on_rank0_only(monkeypatch, capsys):
    class Args:
        steps, warmup, gpus, config = 1, 3, 2, bench.DEFAULT_CFG
    monkeypatch.setenv("RANK", "1")
    bench.run_reference(Args())
    assert capsys.readouterr().out == ""


@pytest.mark.parametrize("world", [1, 2])
def test_reference_arm_line(monkeypatch, capsys, world):
    """Rank 0's reference line carries the contract's keys (oracle timed on a tiny sample)."""
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setattr(bench, "time_oracle", lambda cfg, reps, warm, **kw: {
        "value": 123.0, "unit": bench.UNIT, "cores": 4, "kind": "oracle", "sample": "stub",
        "mean_step_ms": 0.125})

    class Args:
        steps, warmup, gpus, config = 2, 3, world, bench.DEFAULT_CFG
    bench.run_reference(Args())
    line = json.loads(capsys.readouterr().out.strip())
    assert line["impl"] == "reference" and line["n_gpus"] == world and line["higher_is_better"] is False
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
    # ms_per_step is the time of one timed step (one layer), not a multiple of it
    assert line["ms_per_step"] == 0.125 and line["config"]["layers_per_step"] == 1
    assert line["cpu_baseline"]["cores"] == 4


def test_oracle_timing_runs_on_several_processes():
    """The CPU baseline's oracle timing forks worker processes over the units of one
    layer (tiny configuration) and reports the process count and a one-process figure."""
    res = bench.time_oracle(1, reps=2, warm=1, single_reps=1, workers=2)
    assert res["kind"] == "oracle" and res["value"] > 0 and res["unit"] == bench.UNIT
    assert res["cores"] == 1                    # the tiny configuration has one unit
    assert res["single_thread"]["cores"] == 1 and res["single_thread"]["value"] > 0
