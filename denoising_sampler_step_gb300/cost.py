"""Algorithmic cost model of one sampler step (bytes, FLOPs, wire volume).

The byte and FLOP counts are those of the method, not of any implementation:
each logit is read once, each embedding row once, and the product costs 2 FLOPs
per multiply-add.  The wire-volume formulas restate calvarado04.com, "Why not
just all-gather the weights": the table size V*d*b, the product's FLOPs per rank,
the size of the reduced [L_c x d] tensor, a ring all-reduce's per-rank volume,
and the crossover K*N*L_c <= V/2 against a one-time all-gather.
"""
from __future__ import annotations

from dataclasses import dataclass

BF16_BYTES = 2
F32_BYTES = 4


def embedding_bytes(V: int, d: int, elem_bytes: int = BF16_BYTES) -> int:
    """Size of the token-embedding table W [V, d]."""
    return V * d * elem_bytes


def soft_embed_flops(rows: int, V: int, d: int, tp: int = 1) -> float:
    """FLOPs of P[rows, V/tp] @ W[V/tp, d] on one rank (2 per multiply-add)."""
    return 2.0 * rows * (V / tp) * d


def reduced_tensor_bytes(L_c: int, d: int, elem_bytes: int = BF16_BYTES) -> int:
    """Size of the [L_c, d] partial that the tensor-parallel ranks sum."""
    return L_c * d * elem_bytes


def ring_allreduce_bytes_per_rank(L_c: int, d: int, tp: int, elem_bytes: int = BF16_BYTES) -> float:
    """Bytes each rank sends in a ring all-reduce: 2 (T-1)/T times the tensor size."""
    return 2.0 * (tp - 1) / tp * reduced_tensor_bytes(L_c, d, elem_bytes)


def allgather_crossover_KN(V: int, L_c: int) -> float:
    """K*N below which repeated all-reduces move fewer bytes than one all-gather of W.

    Wire volume 2 K N L_c d <= V d  <=>  K N <= V / (2 L_c)."""
    return V / (2.0 * L_c)


@dataclass(frozen=True)
class StepCost:
    rows: int
    V: int
    d: int
    vocab: int          # width of the vocabulary slice the product covers

    @property
    def logits_bytes(self) -> int:
        return self.rows * self.V * F32_BYTES

    @property
    def w_bytes(self) -> int:
        return embedding_bytes(self.vocab, self.d)

    @property
    def out_bytes(self) -> int:
        return self.rows * self.d * F32_BYTES

    @property
    def flops(self) -> float:
        return 2.0 * self.rows * self.vocab * self.d

    @property
    def stats_bytes(self) -> int:
        """Row-statistics pass: the logits once, plus 5 words per row written."""
        return self.logits_bytes + self.rows * 5 * 4

    @property
    def gemm_bytes(self) -> int:
        """Soft-embed product: the logits of the slice once, W once, E once."""
        return self.rows * self.vocab * F32_BYTES + self.w_bytes + self.out_bytes

    @property
    def step_bytes(self) -> int:
        """One fused step: the logits once, W once, E, and per row the statistics (m, lse, H,
        kappa, argmax), the order entry and the mask byte."""
        return self.gemm_bytes + self.rows * (5 * 4 + 4 + 1)

    @property
    def e4m3_table_bytes(self) -> int:
        """The 8-bit table of the slice: one E4M3 code per entry and one fp32 scale per row."""
        return self.vocab * self.d + self.vocab * F32_BYTES

    @property
    def e4m3_gemm_bytes(self) -> int:
        """Soft-embed product over the 8-bit table: the logits once, the table once, E once."""
        return self.rows * self.vocab * F32_BYTES + self.e4m3_table_bytes + self.out_bytes

    def roofline_seconds(self, hbm_gbs: float, bf16_tflops: float) -> float:
        """Slower of the product's FLOPs at the bf16 peak and the logits + W bytes at HBM bandwidth."""
        t_mem = (self.logits_bytes + self.w_bytes) / (hbm_gbs * 1e9)
        t_cmp = self.flops / (bf16_tflops * 1e12)
        return max(t_mem, t_cmp)
