"""The host side of a multi-GPU bench run, on CPU: two gloo ranks (one process each, as the
launcher runs them) reduce their timed-region lengths to the slowest rank's, and the whole-job
throughput of the weak-scaling run counts every rank's bytes over that time.  The path shards
into independent replicas, so these reductions are the only communication it has."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    r, w, local = bench.dist_env()
    dist.init_process_group("gloo", rank=r, world_size=w)
    try:
        # rank r measured elapsed = 1 + r seconds and a step of 5 - r ms
        got = bench.max_over_ranks([1.0 + r, 5.0 - r, 10.0 * r], w, "cpu")
        value = bench.weak_scaling_gbs(1e9, w, got[0])
        ref = bench.run_reference(type("A", (), {"steps": 1, "warmup": 0})(), r, w) if r != 0 else "rank0"
        q.put((r, w, local, got, value, ref))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_to_the_slowest_rank():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, (rank, w, local, got, value, ref) in enumerate(out):
        assert (rank, w, local) == (r, world, r)
        assert got == [2.0, 5.0, 10.0]                 # every rank sees the maxima
        assert value == pytest.approx(1.0)             # 2 ranks x 1 GB over the slowest 2 s
    assert out[1][5] is None                           # the reference arm runs on rank 0 only


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks([3.0, 4.0], 1, "cpu") == [3.0, 4.0]
    assert bench.weak_scaling_gbs(6e9, 1, 2.0) == pytest.approx(3.0)
