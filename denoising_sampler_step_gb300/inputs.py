"""Seeded synthetic inputs for the DiffusionGemma denoising-sampler step.

This module only synthesises inputs; it contains none of the sampler's own
arithmetic (no softmax, entropy, ordering or embedding product).  Both the CUDA
path and the CPU oracle take their inputs from here, and nothing else is shared
between them.

Random numbers come from Philox4x64-10 (Salmon, Moraes, Dror, Shaw, "Parallel
random numbers: as easy as 1, 2, 3", SC'11) as implemented by numpy's
``np.random.Philox``.  Every stream is keyed by ``(seed, stream_id)`` where the
stream id packs a tensor tag, an index and a redraw attempt, so that

* a row, a request or a weight block can be redrawn on its own, and
* the result does not depend on how many threads generate it.

Workload shapes and distributions follow the pages' sizes (V = 262,144
vocabulary entries, d = 2,816 hidden size, a 256-position canvas: calvarado04.com,
"Where the shapes stop agreeing" and "Why not just all-gather the weights";
agentlenshq.com, "サンプリングループとエントロピー境界デノイジング").
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field, replace

import numpy as np

# Stream tags (top byte of the 64-bit stream id).
TAG_ROW_Z = 1        # per-row N(0,1) draws of the logits
TAG_ROW_PARAMS = 2   # per-request row scale, boost index and boost size
TAG_W = 3            # per-block N(0,1) draws of the embedding table
TAG_BUDGET = 4       # per-request entropy budgets
TAG_LOOP_NOISE = 5   # per-step, per-row noise of a denoising-loop sequence
TAG_W8 = 6           # per-block draws of an 8-bit (E4M3) embedding table

W_BLOCK_ROWS = 4096  # embedding rows drawn per Philox stream


def stream_id(tag: int, index: int, attempt: int = 0) -> int:
    if not (0 <= tag < 256 and 0 <= attempt < 256 and 0 <= index < (1 << 48)):
        raise ValueError("stream id field out of range")
    return (tag << 56) | (attempt << 48) | index


def philox(seed: int, sid: int) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(key=np.array([seed, sid], dtype=np.uint64)))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round to nearest, ties to even); return the uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> 16) & 1) + np.uint32(0x7FFF)
    return ((u + bias) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def bf16_round(x: float) -> float:
    """A Python float rounded to the nearest bfloat16 value."""
    return float(bf16_bits_to_f32(f32_to_bf16_bits(np.array([x], np.float32)))[0])


def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


@dataclass(frozen=True)
class Workload:
    """One synthetic sampler-step workload.

    ``scale``: per-row logit scale s_i ~ U[scale]; ``boost``: a U[boost] bump added
    at one uniformly random vocab index per row (``boost_over_max``: the bump is
    put on top of the row's maximum instead, which makes rows near one-hot).
    """
    name: str
    n_req: int
    L_c: int
    V: int
    d: int
    scale: tuple
    boost: tuple
    budget: object            # a float, or ("uniform", lo, hi) drawn per request
    slices: int = 1           # vocabulary partitions T (1 = unsliced)
    boost_over_max: bool = False
    seed: int = 0

    @property
    def R(self) -> int:
        return self.n_req * self.L_c

    @property
    def gamma(self) -> float:
        """Normaliser: sqrt(d) rounded to bfloat16 (53.0 at d = 2816, 16.0 at d = 256)."""
        return bf16_round(math.sqrt(self.d))

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# The five workloads of the sampler-step benchmark plus the peaked-row variant.
WORKLOADS = {
    "tiny": Workload("tiny", 1, 16, 4096, 256, (0.5, 4.0), (0.0, 8.0), 2.0, seed=0),
    "canvas256": Workload("canvas256", 1, 256, 262144, 2816, (0.5, 4.0), (0.0, 8.0), 8.0, seed=1),
    "batch8": Workload("batch8", 8, 256, 262144, 2816, (0.25, 8.0), (0.0, 8.0),
                       ("uniform", 2.0, 16.0), seed=2),
    "vocab_tp4": Workload("vocab_tp4", 1, 256, 262144, 2816, (0.5, 4.0), (0.0, 8.0), 8.0,
                          slices=4, seed=3),
    "late_batch32": Workload("late_batch32", 32, 256, 262144, 2816, (4.0, 12.0), (8.0, 20.0), 1.0,
                             seed=4),
    "late_batch32_peaked": Workload("late_batch32_peaked", 32, 256, 262144, 2816, (4.0, 12.0),
                                    (8.0, 20.0), 1.0, boost_over_max=True, seed=4),
}


def request_logits(wl: Workload, q: int, attempt: int = 0, out: np.ndarray | None = None) -> np.ndarray:
    """fp32 logits [L_c, V] of request ``q``: l = s_i * z + bump at one index."""
    L, V = wl.L_c, wl.V
    if out is None:
        out = np.empty((L, V), np.float32)
    pg = philox(wl.seed, stream_id(TAG_ROW_PARAMS, q, attempt))
    s = pg.uniform(wl.scale[0], wl.scale[1], L).astype(np.float32)
    idx = pg.integers(0, V, L)
    bump = pg.uniform(wl.boost[0], wl.boost[1], L).astype(np.float32)

    def one(i: int) -> None:
        g = philox(wl.seed, stream_id(TAG_ROW_Z, q * L + i, attempt))
        row = out[i]
        g.standard_normal(out=row, dtype=np.float32)
        row *= s[i]
        if wl.boost_over_max:
            row[idx[i]] = row.max() + bump[i]
        else:
            row[idx[i]] += bump[i]

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(one, range(L)))
    return out


def logits(wl: Workload, attempts: dict | None = None, ld: int | None = None) -> np.ndarray:
    """fp32 logits [R, ld] (ld >= V; columns V..ld-1 are set to NaN so that reading them shows up)."""
    ld = wl.V if ld is None else ld
    buf = np.empty((wl.R, ld), np.float32)
    if ld > wl.V:
        buf[:, wl.V:] = np.nan
    for q in range(wl.n_req):
        a = 0 if attempts is None else attempts.get(q, 0)
        rows = buf[q * wl.L_c:(q + 1) * wl.L_c]
        if ld == wl.V:
            request_logits(wl, q, a, out=rows)
        else:
            rows[:, :wl.V] = request_logits(wl, q, a)
    return buf


def embedding_bf16(wl: Workload) -> np.ndarray:
    """Token embedding W [V, d] as bfloat16 bit patterns (uint16), W ~ N(0, 0.02^2)."""
    V, d = wl.V, wl.d
    out = np.empty((V, d), np.uint16)
    nblk = (V + W_BLOCK_ROWS - 1) // W_BLOCK_ROWS

    def one(b: int) -> None:
        r0, r1 = b * W_BLOCK_ROWS, min(V, (b + 1) * W_BLOCK_ROWS)
        g = philox(wl.seed, stream_id(TAG_W, b))
        z = g.standard_normal((r1 - r0, d), dtype=np.float32)
        z *= np.float32(0.02)
        out[r0:r1] = f32_to_bf16_bits(z)

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(one, range(nblk)))
    return out


def embedding_e4m3(wl: Workload) -> tuple:
    """An 8-bit embedding table drawn directly: codes Q [V, d] (uint8) and per-row fp32 scales
    [V].  Magnitude codes are uniform over 0x40..0x7E (E4M3 values 2 to 448), signs uniform,
    and one entry per row holds the code of 448 (the row maximum a per-row quantiser
    produces); scales are uniform in [1e-4, 3e-4], so entries lie within about 0.13 of 0."""
    V, d = wl.V, wl.d
    Q = np.empty((V, d), np.uint8)
    scale = np.empty(V, np.float32)
    nblk = (V + W_BLOCK_ROWS - 1) // W_BLOCK_ROWS

    def one(b: int) -> None:
        r0, r1 = b * W_BLOCK_ROWS, min(V, (b + 1) * W_BLOCK_ROWS)
        g = philox(wl.seed, stream_id(TAG_W8, b))
        mag = g.integers(0x40, 0x7F, (r1 - r0, d), dtype=np.uint8)
        sign = g.integers(0, 2, (r1 - r0, d), dtype=np.uint8) << np.uint8(7)
        mag[np.arange(r1 - r0), g.integers(0, d, r1 - r0)] = 0x7E
        Q[r0:r1] = mag | sign
        scale[r0:r1] = g.uniform(1e-4, 3e-4, r1 - r0).astype(np.float32)

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(one, range(nblk)))
    return Q, scale


def budgets(wl: Workload) -> np.ndarray:
    """Per-request entropy budgets in nats (fp32 [n_req])."""
    if isinstance(wl.budget, tuple):
        _, lo, hi = wl.budget
        g = philox(wl.seed, stream_id(TAG_BUDGET, 0))
        return g.uniform(lo, hi, wl.n_req).astype(np.float32)
    return np.full(wl.n_req, wl.budget, np.float32)


def slice_bounds(V: int, T: int) -> list:
    """Contiguous, disjoint, exhaustive vocabulary slices [s_r, e_r) for T partitions."""
    base, extra = divmod(V, T)
    bounds, s = [], 0
    for r in range(T):
        e = s + base + (1 if r < extra else 0)
        bounds.append((s, e))
        s = e
    return bounds


def padded_shard(W_bits: np.ndarray, s: int, e: int, multiple: int = 128, pad_value: str = "zero") -> np.ndarray:
    """Rows [s, e) of W laid out as a shard padded to a multiple of ``multiple`` rows.

    ``pad_value`` is "zero" (what a serving engine stores) or "nan" (bf16 quiet NaN,
    used by tests to prove that padding rows are never read)."""
    rows = e - s
    rows_pad = -(-rows // multiple) * multiple
    out = np.zeros((rows_pad, W_bits.shape[1]), np.uint16)
    out[:rows] = W_bits[s:e]
    if pad_value == "nan":
        out[rows:] = 0x7FC0
    return out


def loop_logits(wl: Workload, step: int, settle: int = 4, noise: float = 1.0, base: np.ndarray | None = None) -> np.ndarray:
    """fp32 logits [R, V] of step ``step`` of a synthetic denoising loop whose predictions
    settle: the workload's logits plus N(0, sigma_t^2) noise per entry, with
    sigma_t = noise * row scale * (1 - step / settle) for step < settle and no noise from
    step ``settle`` on (the logits of every later step are the workload's own)."""
    x = logits(wl) if base is None else base.copy()
    if step >= settle:
        return x
    frac = np.float32(noise * (1.0 - step / settle))

    def one(i: int) -> None:
        g = philox(wl.seed, stream_id(TAG_LOOP_NOISE, i, step))
        row = x[i]
        sd = np.float32(row.std())
        row += g.standard_normal(wl.V, dtype=np.float32) * (frac * sd)

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(one, range(wl.R)))
    return x
