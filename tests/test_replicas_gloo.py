"""The replica (data-parallel) host logic across two processes on CPU with gloo:
each rank draws different canvases, and the whole-job time is the slowest rank's."""
import os
import socket

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

from denoising_sampler_step_gb300 import inputs, replicas


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        wl = replicas.rank_workload(inputs.WORKLOADS["tiny"].with_(V=256, L_c=4), rank)
        x = inputs.logits(wl)
        local_ms = [10.0 + rank, 5.0 - rank]        # rank 1 is slower in the first value only
        agg = replicas.max_over_ranks(local_ms)
        q.put((rank, wl.seed, float(x.sum()), agg))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, s0, x0, a0), (r1, s1, x1, a1) = res
    assert s0 != s1 and x0 != x1                    # independent canvases per rank
    assert a0 == a1 == [11.0, 5.0]                  # max over ranks, element-wise
    assert replicas.whole_job_rate(256, 10, 2, 11.0) == pytest.approx(2 * 256 * 10 / 0.011)


def test_single_process_is_identity():
    assert replicas.max_over_ranks([1.5, 2.5]) == [1.5, 2.5]
    assert replicas.rank_workload(inputs.WORKLOADS["canvas256"], 0) == inputs.WORKLOADS["canvas256"]
