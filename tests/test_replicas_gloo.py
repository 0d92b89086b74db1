"""The N > 1 path of bench.py on CPU: two gloo ranks.

The compressed step does not shard across GPUs here (all W workers live in
one GPU's memory), so `bench.py --gpus N` runs N independent replicas; the
only cross-rank operations are the barriers around the timed region and the
max-over-ranks reduction of the step time.  These tests run that plumbing
with world_size 2 on the gloo backend, plus the whole-job value arithmetic.
"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = bench.dist_env()
        assert (ws, r, local) == (world, rank, rank)
        bench.barrier(None)
        # rank r "measured" (r + 1) ms per step; the job's step time is the max
        ms = bench.reduce_max(float(rank + 1), None)
        bench.barrier(None)
        q.put((rank, ms))
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_barrier():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    got = sorted(q.get(timeout=5) for _ in range(2))
    assert got == [(0, 2.0), (1, 2.0)]


def test_single_process_is_identity():
    import bench
    assert not dist.is_initialized()
    assert bench.reduce_max(3.5) == 3.5
    bench.barrier(None)


def test_whole_job_value():
    """value = (all ranks' parameters) / (max step time): weak scaling."""
    import synth
    wl = synth.workloads()[2]
    ms = 1.87
    for n in (1, 2, 4, 8):
        value = n * wl.d / (ms * 1e-3)
        assert abs(value / n - wl.d / (ms * 1e-3)) < 1e-3 * value


def _layout_worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # the ranks read different amounts of free host memory (one of them
        # read it after another had allocated); all must pick one layout
        seen = 200e9 if rank == 0 else 100e9
        avail = int(bench.reduce_min(seen, None))
        d, W = 1_416_552_448, 8
        q.put((rank, bench.e2e_host_layout(W, 2 * d, 4 * d, world, avail)))
    finally:
        dist.destroy_process_group()


def test_two_ranks_choose_one_host_layout():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_layout_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    got = sorted(q.get(timeout=5) for _ in range(2))
    # 2 ranks x (8 buffers of 2.83 GB + 5.67 GB theta) = 56.7 GB <= 0.6 x 100 GB
    assert got == [(0, (1, 8)), (1, (1, 8))]


def test_host_layout_ladder():
    """The host-buffer leg's layout steps down with the host memory of the
    node: two sets of W buffers, one set, one buffer all workers read, none."""
    import bench
    d, W = 1_416_552_448, 8
    g, th = 2 * d, 4 * d
    assert bench.e2e_host_layout(W, g, th, 1, int(200e9)) == (2, 8)
    assert bench.e2e_host_layout(W, g, th, 4, int(200e9)) == (1, 8)
    assert bench.e2e_host_layout(W, g, th, 8, int(200e9)) == (1, 1)
    assert bench.e2e_host_layout(W, g, th, 8, int(50e9)) is None
    assert bench.host_memory_available() > 0
