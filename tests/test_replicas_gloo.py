"""The benchmark's multi-GPU bookkeeping (independent replicas, the slowest
rank's time, the job's total throughput), run as two gloo ranks on the CPU."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from static_graph_nn_gb300.replicas import job_throughput, max_over_ranks
    # rank r "measured" 10 + r ms for its 5 steps and 3 + 2r s end to end
    ms, e2e = max_over_ranks([10.0 + rank, 3.0 + 2 * rank])
    out[rank] = (ms, e2e, job_throughput(world, 5, ms * 1e-3))
    dist.barrier()
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    world, port = 2, _free_port()
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    for r in range(world):
        ms, e2e, thr = out[r]
        assert ms == 11.0 and e2e == 5.0
        assert abs(thr - 2 * 5 / 0.011) < 1e-6


def test_single_process_is_identity():
    from static_graph_nn_gb300.replicas import job_throughput, max_over_ranks
    assert max_over_ranks([1.5, 2.5]) == [1.5, 2.5]
    assert job_throughput(1, 20, 2.0) == 10.0
