"""The replicated (N > 1) bench path on CPU: two gloo ranks reduce their
timings by maximum and their work by sum, as the bench's whole-job line does."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r: step 1+r ms, attention 10*(r+1) us, accept 5-r us, e2e 2+3r ms; 64*(r+1) nodes
        times, work = bench.reduce_over_ranks([1.0 + rank, 10.0 * (rank + 1), 5.0 - rank, 2.0 + 3 * rank],
                                              [64.0 * (rank + 1)], torch.device("cpu"))
        out.put((rank, times, work))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_reduce_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, times, work in res:
        assert times == [2.0, 20.0, 5.0, 5.0]      # maximum over the ranks
        assert work == [192.0]                     # sum over the ranks
    # whole-job throughput as the bench reports it: all ranks' nodes over the slowest step
    assert work[0] / (times[0] / 1000.0) == pytest.approx(96000.0)


def test_reduce_over_ranks_single_process_is_identity():
    assert not dist.is_initialized()
    assert bench.reduce_over_ranks([1.5, 2.0], [64], torch.device("cpu")) == ([1.5, 2.0], [64.0])
