"""The vocabulary-parallel host logic (shard bounds, the two gathers in rank order, the
combine and the fixed-order sum) across two processes on CPU with gloo, the per-rank calls
played by the oracle: the sharded step must give the unsharded oracle's step."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from denoising_sampler_step_gb300 import inputs
from denoising_sampler_step_gb300.vocab_parallel import ShardedStep, TorchComm, shard_bounds
from oracle import entropy_accept, row_stats, soft_embed, sum_partials
from oracle.partition_oracle import row_stats_combine, row_stats_partial


class OracleOps:
    """The per-rank calls, on CPU tensors, by the oracle (float64).  The one-read shard calls
    are the same two results: the shard's summaries first, its product against the full-row
    lse second."""

    def workspace(self, shard, W_shard):
        return None

    def shard_begin(self, shard, vocab_offset, W_shard, ws):
        return self.row_stats_partial(shard, vocab_offset)

    def shard_end(self, shard, lse, W_shard, ws):
        return self.soft_embed_shard(shard, lse, W_shard)

    def row_stats_partial(self, shard, vocab_offset):
        p = row_stats_partial(shard.numpy(), vocab_offset)
        return torch.from_numpy(np.stack([p["m"], p["a"].astype(np.float64), p["rest"], p["t"]], axis=1))

    def row_stats_combine(self, states):
        s = states.numpy()
        parts = [{"m": s[r, :, 0], "a": s[r, :, 1].astype(np.int64), "rest": s[r, :, 2], "t": s[r, :, 3]}
                 for r in range(s.shape[0])]
        return {k: torch.from_numpy(np.asarray(v)) for k, v in row_stats_combine(parts).items()}

    def entropy_accept(self, H, kappa, n_req, L_c, budgets, min_accept):
        a = entropy_accept(H.numpy(), kappa.numpy(), n_req, L_c, budgets.numpy(), min_accept=min_accept)
        return {k: torch.from_numpy(np.asarray(v)) for k, v in a.items()}

    def soft_embed_shard(self, shard, lse, W_shard):
        n = shard.shape[1]
        return torch.from_numpy(soft_embed(shard.numpy(), lse.numpy(), 0, n, W_shard.numpy().view(np.uint16), 1.0))

    def sum_partials(self, parts, gamma):
        return torch.from_numpy(sum_partials([p.numpy() for p in parts], gamma))


WL = inputs.WORKLOADS["tiny"].with_(n_req=2, L_c=6, V=301, d=32, seed=5, budget=("uniform", 1.0, 9.0))


def problem():
    x = inputs.logits(WL)
    x[3, :] = -np.inf
    x[3, 290] = 1.0                      # a row whose mass sits in the last shard only
    W = inputs.embedding_bf16(WL)
    return x, W, inputs.budgets(WL)


def reference(x, W, budgets):
    st = row_stats(x)
    acc = entropy_accept(st["H"], st["kappa"], WL.n_req, WL.L_c, budgets, min_accept=1)
    return st, acc, soft_embed(x, st["lse"], 0, WL.V, W, WL.gamma)


def check(out, st, acc, E):
    assert np.array_equal(out["argmax"].numpy(), st["argmax"])
    for k in ("m", "lse", "H", "kappa"):
        assert np.allclose(out[k].numpy(), st[k], rtol=1e-12, atol=1e-12), k
    for k in ("order", "mask", "n_accepted"):
        assert np.array_equal(out[k].numpy(), acc[k]), k
    assert np.allclose(out["E"].numpy(), E, rtol=1e-11, atol=1e-14)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q, two_pass=False):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        x, W, budgets = problem()
        s, e = shard_bounds(WL.V, world)[rank]
        step = ShardedStep(WL.n_req, WL.L_c, WL.gamma, min_accept=1, two_pass=two_pass)
        out = step.rank_step(torch.from_numpy(np.ascontiguousarray(x[:, s:e])), s,
                             torch.from_numpy(W[s:e].view(np.int16)), torch.from_numpy(budgets), TorchComm(),
                             ops=OracleOps())
        q.put((rank, {k: v.numpy() for k, v in out.items()}))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("two_pass", [False, True])
def test_two_gloo_ranks_give_the_unsharded_step(two_pass):
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q, two_pass)) for r in range(world)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=180) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    st, acc, E = reference(*problem())
    for r in range(world):
        check({k: torch.from_numpy(v) for k, v in res[r].items()}, st, acc, E)
    for k in res[0]:                      # every rank holds the same result, bit for bit
        assert np.array_equal(res[0][k], res[1][k], equal_nan=True), k


@pytest.mark.parametrize("T,two_pass", [(1, False), (3, False), (5, False), (3, True)])
def test_local_shards_give_the_unsharded_step(T, two_pass):
    x, W, budgets = problem()
    bounds = shard_bounds(WL.V, T)
    step = ShardedStep(WL.n_req, WL.L_c, WL.gamma, min_accept=1, two_pass=two_pass)
    out = step.local_step([torch.from_numpy(np.ascontiguousarray(x[:, s:e])) for s, e in bounds],
                          [s for s, _ in bounds], [torch.from_numpy(W[s:e].view(np.int16)) for s, e in bounds],
                          torch.from_numpy(budgets), ops=OracleOps())
    check(out, *reference(x, W, budgets))


def test_shard_bounds():
    assert shard_bounds(10, 3) == [(0, 4), (4, 7), (7, 10)]
    assert shard_bounds(262144, 4) == [(0, 65536), (65536, 131072), (131072, 196608), (196608, 262144)]
    with pytest.raises(ValueError):
        shard_bounds(2, 3)
