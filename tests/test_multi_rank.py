"""The benchmark's multi-GPU host logic on CPU: sequences are independent,
so N GPUs run N replicas with no data-path collective; the ranks only share
a barrier and the max-over-ranks of their timings.  Two gloo ranks on
127.0.0.1 exercise that logic without a GPU."""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    w, r, local = bench.dist_setup()
    assert (w, r, local) == (world, rank, rank)
    bench.barrier(w)
    # each replica's timing; the job's time is the slowest rank's
    t = bench.max_over_ranks(10.0 + rank, w)
    out[rank] = t
    # the reference arm prints on rank 0 only; other ranks return silently
    if rank != 0:
        args = type("A", (), dict(impl="reference", steps=1, warmup=0, config="c2"))()
        assert bench.run_reference(args) is None
    bench.barrier(w)
    dist.destroy_process_group()


def test_two_gloo_ranks_share_barrier_and_max():
    world, port = 2, _free_port()
    manager = mp.Manager()
    out = manager.dict()
    mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
    assert dict(out) == {0: 11.0, 1: 11.0}
