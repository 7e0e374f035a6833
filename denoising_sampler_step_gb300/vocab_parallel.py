"""Vocabulary-parallel sampler step: each rank holds one contiguous shard of the vocabulary,
both its logit columns and its rows of the embedding table W, and no weight moves
(calvarado04.com, "The fix": the probabilities of a slice multiply the shard's own rows,
the partial embeddings are summed over ranks, and gamma is applied after the sum).

Per step, on every rank (the shard's logits read once):
  1. dg_soft_embed_shard_begin: the product over the shard with the row statistics folded
     in, and a 16-byte summary per row of the shard's logits (the split partials wait in
     the workspace);
  2. all-gather of the summaries (R x 16 bytes per rank), then dg_row_stats_combine in
     rank order: every rank holds the full-row statistics (max, argmax, lse, H, kappa);
  3. dg_entropy_accept on those statistics (the same result on every rank);
  4. dg_soft_embed_shard_end with the global lse and gamma = 1: the shard's partial [R, d];
  5. all-gather of the partials, then dg_sum_partials in rank order with gamma: the same
     E, bit for bit, on every rank and in every run (an all-reduce would leave the order
     of the additions to the library; the partials are small, R x d x 4 bytes).
With two_pass, steps 1 and 4 are dg_row_stats_partial (a read of the shard's logits for the
summaries alone) and dg_soft_embed with the global lse (a second read).

`ops` carries the per-rank calls (the CUDA binding by default) and `comm` the all-gather (a
torch.distributed process group); both are parameters so that the orchestration can be
exercised by multi-process tests on the host.  `local_step` runs all shards in one
process, on one device, with the gathers replaced by stacking.  A shard of an 8-bit table
is the pair (E4M3 codes, fp32 row scales) of its rows; the products then run over the
8-bit table.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


def shard_bounds(V: int, T: int) -> list:
    """Contiguous, disjoint shards [s_r, e_r) covering [0, V), sizes differing by at most one,
    the larger ones first."""
    if T < 1 or V < T:
        raise ValueError("need 1 <= T <= V")
    base, extra = divmod(V, T)
    out, s = [], 0
    for r in range(T):
        e = s + base + (1 if r < extra else 0)
        out.append((s, e))
        s = e
    return out


class CudaOps:
    """The five per-rank calls, through libdgsamp."""

    def __init__(self):
        from . import binding
        self.B = binding

    def row_stats_partial(self, shard, vocab_offset):
        return self.B.dg_row_stats_partial(shard, vocab_offset)

    def row_stats_combine(self, states):
        return self.B.dg_row_stats_combine(states)

    def entropy_accept(self, H, kappa, n_req, L_c, budgets, min_accept):
        return self.B.dg_entropy_accept(H, kappa, n_req, L_c, budgets, min_accept=min_accept)

    def workspace(self, shard, W_shard):
        R, n = shard.shape
        if isinstance(W_shard, tuple):
            return self.B.workspace_e4m3(R, n, W_shard[0].shape[1], shard.device)
        return self.B.workspace(R, n, W_shard.shape[1], shard.device)

    def shard_begin(self, shard, vocab_offset, W_shard, ws):
        return self.B.dg_soft_embed_shard_begin(shard, vocab_offset, W_shard, ws)

    def shard_end(self, shard, lse, W_shard, ws):
        return self.B.dg_soft_embed_shard_end(shard, lse, W_shard, 1.0, ws)

    def soft_embed_shard(self, shard, lse, W_shard):
        if isinstance(W_shard, tuple):  # an 8-bit table: (codes, row scales)
            Q, scale = W_shard
            return self.B.dg_soft_embed_e4m3(shard, lse, 0, shard.shape[1], Q, scale, 1.0)
        return self.B.dg_soft_embed(shard, lse, 0, shard.shape[1], W_shard, 1.0)

    def sum_partials(self, parts, gamma):
        return self.B.dg_sum_partials(parts, gamma)


class TorchComm:
    """All-gather over a torch.distributed process group, rank order = shard order."""

    def __init__(self, group=None):
        import torch.distributed as dist
        self.dist = dist
        self.group = group
        self.world = dist.get_world_size(group)
        self.rank = dist.get_rank(group)

    def all_gather(self, t: torch.Tensor) -> torch.Tensor:
        """[world, *t.shape], rank r's tensor at index r (gathered along dim 0, then viewed)."""
        t = t.contiguous()
        out = torch.empty((self.world * t.shape[0],) + tuple(t.shape[1:]), dtype=t.dtype, device=t.device)
        self.dist.all_gather_into_tensor(out, t, group=self.group)
        return out.view((self.world,) + tuple(t.shape))


@dataclass
class ShardedStep:
    n_req: int
    L_c: int
    gamma: float
    min_accept: int = 0
    two_pass: bool = False

    def rank_step(self, shard: torch.Tensor, vocab_offset: int, W_shard: torch.Tensor, budgets: torch.Tensor,
                  comm, ops=None) -> dict:
        """One step on this rank's shard; returns stats, acceptance and E (identical on all ranks)."""
        ops = CudaOps() if ops is None else ops
        if self.two_pass:
            states = comm.all_gather(ops.row_stats_partial(shard, vocab_offset))
        else:
            ws = ops.workspace(shard, W_shard)
            states = comm.all_gather(ops.shard_begin(shard, vocab_offset, W_shard, ws))
        st = ops.row_stats_combine(states)
        acc = ops.entropy_accept(st["H"], st["kappa"], self.n_req, self.L_c, budgets, self.min_accept)
        part = (ops.soft_embed_shard(shard, st["lse"], W_shard) if self.two_pass
                else ops.shard_end(shard, st["lse"], W_shard, ws))
        parts = comm.all_gather(part)
        E = ops.sum_partials([parts[r] for r in range(parts.shape[0])], self.gamma)
        return dict(st, **acc, E=E)

    def local_step(self, shards: list, offsets: list, W_shards: list, budgets: torch.Tensor, ops=None) -> dict:
        """All shards in one process (one device): the gathers become stacking."""
        ops = CudaOps() if ops is None else ops
        if self.two_pass:
            states = torch.stack([ops.row_stats_partial(s, o) for s, o in zip(shards, offsets)])
        else:
            wss = [ops.workspace(s, w) for s, w in zip(shards, W_shards)]
            states = torch.stack([ops.shard_begin(s, o, w, ws) for s, o, w, ws in zip(shards, offsets, W_shards, wss)])
        st = ops.row_stats_combine(states)
        acc = ops.entropy_accept(st["H"], st["kappa"], self.n_req, self.L_c, budgets, self.min_accept)
        if self.two_pass:
            parts = [ops.soft_embed_shard(s, st["lse"], w) for s, w in zip(shards, W_shards)]
        else:
            parts = [ops.shard_end(s, st["lse"], w, ws) for s, w, ws in zip(shards, W_shards, wss)]
        E = ops.sum_partials(parts, self.gamma)
        return dict(st, **acc, E=E)
