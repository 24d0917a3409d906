"""The N > 1 host path of bench.py on CPU: two gloo ranks.

The decode step does not shard (each rank decodes its own replica of the
batch, no data-path collective), so what the multi-rank run adds is host logic:
all ranks time the same number of steps, the step time is the maximum over
ranks, the whole-job value counts every rank's queries, only rank 0 prints,
and the reference arm runs on rank 0 alone.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, outdir):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        # each rank calibrates a different count; rank 0's wins
        steps = bench.agree_steps(dist, 100 + 37 * rank, "cpu")
        # rank 1 is the slow one in the first field, rank 0 in the second
        ms = bench.max_over_ranks(dist, [1.0 + rank, 5.0 - rank], "cpu")
        value = bench.job_throughput(world, 4, ms[0] / steps)
        with open(os.path.join(outdir, f"r{rank}.json"), "w") as f:
            json.dump({"steps": steps, "ms": ms, "value": value}, f)
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregation(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    got = [json.load(open(tmp_path / f"r{r}.json")) for r in range(world)]
    for g in got:
        assert g["steps"] == 100
        assert g["ms"] == [2.0, 5.0]
        # 2 ranks x 4 queries per step; a step takes 2.0 ms / 100 steps
        assert g["value"] == pytest.approx(2 * 4 / (0.02e-3))


def test_single_process_helpers_are_identity():
    import bench
    assert bench.agree_steps(None, 17, "cpu") == 17
    assert bench.max_over_ranks(None, [1, 2.5], "cpu") == [1.0, 2.5]
    assert bench.job_throughput(1, 64, 0.5) == pytest.approx(128000.0)


def test_reference_arm_under_torchrun_prints_once():
    """Two ranks launched the way the N > 1 runs are: rank 0 alone runs the
    oracle and prints one line; rank 1 exits 0 without work."""
    env = dict(os.environ)
    env.pop("CUDA_VISIBLE_DEVICES", None)
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--workload", "tiny_fp32", "--steps", "2", "--warmup", "1"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference"
    assert line["n_gpus"] == 2
    assert line["steps"] == 2 and line["warmup"] == 1
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
