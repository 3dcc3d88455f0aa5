"""The N>1 benchmark path on CPU: two gloo ranks, no GPU.

With --gpus N every rank runs an independent replica on its own batch (the
sequences of a batch are independent, so nothing is exchanged on the data
path); the timing is the slowest rank's, taken with a MAX all-reduce after a
barrier, and the reported value is the units all ranks processed over that
time.  These tests run that host logic in two real processes.
"""
import os
import socket
import tempfile

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, outdir):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    import synth
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, local = bench.dist_env()
        assert (w, r, local) == (world, rank, rank)
        dist.barrier()
        ms_local = 10.0 + 5.0 * rank          # rank 1 is the slow one
        ms = bench.max_over_ranks(ms_local, dist, "cpu")
        shape = synth.WORKLOADS[1]
        lens = synth.lengths(bench.replica_seed(rank), shape)
        np.save(os.path.join(outdir, f"r{rank}.npy"), np.concatenate([[ms], lens.astype(np.float64)]))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_distinct_batches():
    world = 2
    with tempfile.TemporaryDirectory() as d:
        mp.start_processes(_rank_main, args=(world, _free_port(), d), nprocs=world, join=True, start_method="spawn")
        got = [np.load(os.path.join(d, f"r{r}.npy")) for r in range(world)]
    # every rank sees the maximum of the per-rank times
    assert got[0][0] == 15.0 and got[1][0] == 15.0
    # the replicas run different batches (different lengths drawn from their seeds)
    assert not np.array_equal(got[0][1:], got[1][1:])


def test_job_value_counts_every_rank_over_the_slowest_time():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.job_value(2, 65536, 0.5) == pytest.approx(262144.0)
    assert bench.max_over_ranks(3.5, None, "cpu") == 3.5
    assert bench.replica_seed(0) != bench.replica_seed(1)


def test_reference_arm_prints_on_rank_zero_only():
    import json
    import subprocess
    import sys
    base = dict(os.environ, MASTER_ADDR="127.0.0.1", WORLD_SIZE="2")
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1",
           "--warmup", "0", "--workload", "0"]
    r1 = subprocess.run(cmd, env=dict(base, RANK="1", LOCAL_RANK="1"), capture_output=True, text=True, timeout=300)
    assert r1.returncode == 0 and r1.stdout.strip() == ""
    r0 = subprocess.run(cmd, env=dict(base, RANK="0", LOCAL_RANK="0"), capture_output=True, text=True, timeout=300)
    assert r0.returncode == 0
    lines = [l for l in r0.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
