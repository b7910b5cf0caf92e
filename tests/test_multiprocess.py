"""The N > 1 path of bench.py on the CPU with the gloo backend: one process per
rank (world size 2), the barrier and the max-over-ranks timing, and the
reference arm under torchrun (rank 0 alone prints its line, the other ranks
exit 0 without work). The path has no data-path collective (replicas only), so
this is all the multi-process logic there is."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    r, w, local = bench.dist_setup(world)
    assert (r, w, local) == (rank, world, rank)
    assert dist.get_backend() == "gloo"
    bench.barrier(w)
    # each rank reports its own time; every rank gets the maximum
    got = bench.max_over_ranks(10.0 + 5.0 * rank, w)
    results[rank] = got
    dist.destroy_process_group()


def test_barrier_and_max_over_ranks_on_two_gloo_ranks():
    if torch.cuda.is_available():
        pytest.skip("the CPU (gloo) path; with a GPU bench.py picks NCCL")
    world, port = 2, _free_port()
    with mp.get_context("spawn").Manager() as m:
        results = m.dict()
        mp.spawn(_rank_main, args=(world, port, results), nprocs=world, join=True)
        assert dict(results) == {0: 15.0, 1: 15.0}


def test_reference_arm_under_torchrun_prints_once():
    if torch.cuda.is_available():
        pytest.skip("the CPU (gloo) path")
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--gpus", "2", "--workload", "tiny", "--steps", "1", "--warmup", "3",
           "--ref-seconds", "1"]
    p = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, p.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["unit"] == "us/step"
    assert d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0
