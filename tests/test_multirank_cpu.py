"""Multi-process tier of bench.py on CPU: the replica path's cross-rank steps
(max over ranks of the per-step times, one shared decision to re-run a noisy
round set) as two gloo ranks, and the reference arm launched by torchrun with
two processes (rank 0 alone prints its line; the other rank exits 0)."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r's per-step times: [ms, ms_e2e] and a round-set CV
        times = bench.ranks_max([1.0 + rank, 5.0 - 3 * rank], torch.device("cpu"))
        cv = bench.ranks_max([0.01 if rank == 0 else 0.05], torch.device("cpu"))[0]
        with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
            json.dump({"times": times, "cv": cv}, f)
    finally:
        dist.destroy_process_group()


def test_ranks_max_two_gloo_ranks(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    res = [json.load(open(tmp_path / f"r{r}.json")) for r in range(world)]
    for r in res:
        assert r["times"] == [2.0, 5.0]  # element-wise max, same on every rank
        assert r["cv"] == 0.05           # so both ranks re-run, or neither
    # whole-job throughput from the slowest replica's step time
    assert bench.job_tokens_per_s(8, world, res[0]["times"][0]) == pytest.approx(8000.0)


def test_ranks_max_without_process_group():
    import torch
    assert bench.ranks_max([3, 1.5], torch.device("cpu")) == [3.0, 1.5]
    assert bench.job_tokens_per_s(8, 1, 0.08) == pytest.approx(100000.0)


def test_reference_arm_under_torchrun_two_processes():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()),
           "bench.py", "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "1",
           "--workload", "tiny"]
    p = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [json.loads(l) for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, p.stdout
    r = lines[0]
    assert r["impl"] == "reference" and r["n_gpus"] == 2 and r["steps"] == 2
    assert r["config"]["workload"] == "tiny" and r["value"] > 0
    # the oracle runs on every host core even though torchrun sets OMP_NUM_THREADS=1
    assert r["cpu_baseline"]["cores"] == bench.host_cores()
    assert r["e2e"]["h2d_bytes_per_step"] == 0 and r["e2e"]["value"] == r["value"]
