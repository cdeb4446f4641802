"""The multi-process (one rank per GPU) host logic, on the CPU with gloo.

The decode path has no exchange step: N GPUs run N replicas, and the bench
reports the units all ranks processed over the slowest rank's timed region.
These tests run two ranks on the CPU: the barrier and the max-over-ranks
reduction the bench uses, and the reference arm under torchrun (rank 0 alone
works and prints; the other rank exits 0)."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, times: list, out_q) -> None:
    sys.path.insert(0, ROOT)
    import bench
    torch.distributed.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}",
                                         rank=rank, world_size=world)
    try:
        bench.rank_barrier()
        got = bench.max_over_ranks(times[rank], torch.device("cpu"))
        bench.rank_barrier()
        out_q.put((rank, got))
    finally:
        torch.distributed.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    times = [3.5, 7.25]
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, times, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    results = dict(q.get(timeout=10) for _ in range(2))
    assert results == {0: 7.25, 1: 7.25}          # every rank sees the slowest rank's time


def test_max_over_ranks_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(4.5, torch.device("cpu")) == 4.5
    bench.rank_barrier()                            # no process group: a no-op


@pytest.mark.slow
def test_reference_arm_under_torchrun_two_ranks():
    """`python -m torch.distributed.run --nproc-per-node 2 bench.py --impl
    reference`: one JSON line (rank 0), both ranks exit 0."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={_free_port()}", "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3",
           "--workload", "mha", "--num-seqs", "4", "--num-blocks", "512", "--cpu-seconds", "1"]
    res = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0
