"""The multi-GPU path is replicas only: each rank runs the whole step on its own
GPU and the ranks only agree on timing.  This checks bench.py's host-side
coordination (rendezvous, barrier, max over ranks, whole-job throughput) with
two gloo ranks on the CPU; no data-path collective exists to test."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, results):
    # CPU ranks (gloo) even on a machine with GPUs: hide them before any CUDA call.
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "CUDA_VISIBLE_DEVICES": ""})
    import bench
    r, w, _ = bench.dist_setup(world)
    assert (r, w) == (rank, world)
    bench.barrier(w)
    elapsed = 1.0 + rank  # the slower rank decides the job's time
    results[rank] = bench.max_over_ranks(elapsed, w)
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    import bench  # noqa: F401  (import errors surface here, not in a child)
    world, port = 2, _free_port()
    with mp.Manager() as mgr:
        results = mgr.dict()
        mp.spawn(_rank, args=(world, port, results), nprocs=world, join=True)
        assert dict(results) == {0: 2.0, 1: 2.0}


def test_whole_job_throughput_is_weak_scaling():
    import bench
    one = bench.whole_job_gbs(10 ** 9, 10, 2.0, 1)
    two = bench.whole_job_gbs(10 ** 9, 10, 2.0, 2)
    assert one == pytest.approx(5.0) and two == pytest.approx(10.0)
