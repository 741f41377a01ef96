"""The multi-process host logic of bench.py on CPU: world size 2 over gloo.

On GPUs each rank runs its own layer (replicas, no collective on the data path); the only cross-rank step is the
timing: a barrier around the timed region and the maximum of the ranks' times.
"""
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


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        torch.distributed.barrier()
        out.put((rank, bench.max_over_ranks(10.0 + 5.0 * rank, True, torch.device("cpu"))))
        torch.distributed.barrier()
    finally:
        torch.distributed.destroy_process_group()


def test_step_time_is_the_slowest_ranks_on_every_rank():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == {0: 15.0, 1: 15.0}


def test_single_process_time_is_unchanged():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(12.5, False, torch.device("cpu")) == 12.5


@pytest.mark.parametrize("rank", ["1"])
def test_reference_arm_runs_on_rank_zero_only(rank):
    # under torchrun the other ranks exit 0 without work and print nothing
    env = dict(os.environ, RANK=rank, WORLD_SIZE="2", LOCAL_RANK=rank)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
