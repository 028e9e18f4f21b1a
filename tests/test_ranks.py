"""Host logic of the bench's multi-rank run, on CPU with the gloo backend.

The decode shards into independent (batch, KV head) units, so N > 1 runs N
replicas with no data-path collective: the only exchange is the all-reduce
that takes the slowest rank's step time, and the whole-job value is the
units (bytes) of every rank over that time.  These tests run that exchange
as two gloo processes, and the reference arm as two torchrun ranks, of
which only rank 0 works and prints.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        # rank r reports a mean step of 1.5 + r ms; every rank must see the maximum
        ms_max = bench.max_over_ranks(1.5 + rank, dist, "cpu")
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"ms_max": ms_max, "gbs": bench.job_gbs(world, 234881024, ms_max)}, f)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2(tmp_path):
    import torch.multiprocessing as mp
    world, port = 2, _free_port()
    mp.start_processes(_rank_main, args=(world, port, str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    got = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for g in got:
        assert g["ms_max"] == 2.5
        # two replicas of 234,881,024 bytes each in 2.5 ms
        assert g["gbs"] == pytest.approx(2 * 234881024 / 2.5e-3 / 1e9, rel=1e-12)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(0.0926) == 0.0926
    assert bench.job_gbs(1, 234881024, 0.0926) == pytest.approx(2536.5, rel=1e-4)


def test_reference_arm_under_torchrun_world2():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={port}", "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "3"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout            # rank 0 prints, rank 1 exits without work
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["steps"] == 1 and line["warmup"] == 3
    assert line["cpu_baseline"]["kind"] == "oracle" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
