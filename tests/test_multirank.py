"""Multi-rank host logic of bench.py on CPU (gloo, world size 2).

Rows are independent, so N GPUs run N full replicas of the step with no
collective on the data path (weak scaling); the only exchange is the
max-over-ranks of the elapsed time, and the reference arm runs on rank 0
alone."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    elapsed = 0.010 * (rank + 1)  # rank 1 is the slow one
    m = bench.max_over_ranks(elapsed, dist, "cpu")
    agg = bench.aggregate(m, steps=100, world=world)
    out.put((rank, m, agg))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_weak_scaling_aggregate_gloo():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    sys.path.insert(0, ROOT)
    import bench
    b, r = bench.step_bytes()
    for rank, m, agg in res:
        assert m == pytest.approx(0.020)
        # whole-job throughput: both replicas' bytes over the slowest rank's time
        assert agg["gbs"] == pytest.approx(world * b * 100 / 0.020 / 1e9)
        assert agg["rows_per_s"] == pytest.approx(world * r * 100 / 0.020)
        assert agg["ms_per_step"] == pytest.approx(0.2)


def _run_reference(rank, world):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
               DAN_REFERENCE_BUDGET_S="1")
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                           "--gpus", str(world), "--steps", "2", "--warmup", "3"],
                          capture_output=True, text=True, env=env, timeout=300)


def test_reference_arm_runs_on_rank_zero_only():
    r1 = _run_reference(1, 2)
    assert r1.returncode == 0 and r1.stdout.strip() == ""
    r0 = _run_reference(0, 2)
    assert r0.returncode == 0, r0.stderr
    line = json.loads(r0.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0


def test_configuration_ids_cover_every_configuration():
    """The JSON line keys each configuration's fraction of peak by a short id;
    every configuration has exactly one, and no two share it."""
    sys.path.insert(0, ROOT)
    import bench
    names = [c[0] for c in bench.CONFIGS]
    assert sorted(names) == sorted(bench.CONFIG_IDS)
    assert len(set(bench.CONFIG_IDS.values())) == len(names)
