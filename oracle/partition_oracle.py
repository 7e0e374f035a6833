"""CPU oracle for vocabulary-sharded row statistics (float64, plain and slow).

TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the benchmark's
CPU legs may import this module; the product path never calls it and shares no code
with it.

What it computes.  Under vocabulary parallelism each rank holds the logit columns of
its shard [s_r, e_r) (calvarado04.com, "The fix": the vocabulary is split into
contiguous ranges, one per rank, and the softmax stays a distribution over all V
tokens).  A rank summarises its shard per row in four numbers,

    m_r    = max over the shard,  a_r = the global index of its first occurrence,
    rest_r = sum over the shard's entries other than a_r of exp(l - m_r),
    t_r    = sum over the shard of exp(l - m_r) (l - m_r),

and the summaries of all shards, taken in shard order, give the full-row statistics:

    m    = max_r m_r,  a = a_r of the first shard with m_r = m (the lowest global index),
    rest = sum_r exp(m_r - m) rest_r + sum_{r != r*} exp(m_r - m)   (r* the shard of a),
    T    = sum_r exp(m_r - m) (t_r + (m_r - m)(rest_r + 1)),
    lnZ  = log1p(rest), lse = m + lnZ, H = lnZ - T / (1 + rest), kappa = lnZ.

These are the definitions of row_stats (sampler_oracle) regrouped by shard: Z is a sum
over shards of each shard's Z_r rescaled to the common maximum, and so is the sum of
exp(l - m)(l - m).  A shard whose logits are all -inf has m_r = -inf and adds nothing;
a row with no finite logit in any shard has NaN statistics and argmax 0.

Pinned by tests/test_partition_pins.py: the combined summaries of random partitions
(uneven, single-entry and empty shards, maxima tied across a shard boundary) equal the
full-row oracle statistics, which closed forms pin on their own.
"""
from __future__ import annotations

import math

import numpy as np

NO_INDEX = 2**31 - 1   # argmax of a shard with no finite logit


def row_stats_partial(shard: np.ndarray, vocab_offset: int) -> dict:
    """Per-row summary (m, a, rest, t) of the fp32 logit columns of one shard [R, n];
    `vocab_offset` is the global index of the shard's first column."""
    x = np.asarray(shard, dtype=np.float32).astype(np.float64)
    R = x.shape[0]
    out = {"m": np.full(R, -np.inf), "a": np.full(R, NO_INDEX, np.int64), "rest": np.zeros(R),
           "t": np.zeros(R)}
    for i in range(R):
        l = x[i]
        if l.size == 0 or not np.any(np.isfinite(l)):
            continue
        m = l.max()
        j = int(np.argmax(l))
        fin = np.isfinite(l)
        e = np.exp(l[fin] - m)
        d = l[fin] - m
        idx = np.nonzero(fin)[0]
        out["m"][i] = m
        out["a"][i] = vocab_offset + j
        out["rest"][i] = math.fsum(float(v) for v, k in zip(e, idx) if k != j)
        out["t"][i] = math.fsum(float(v) * float(w) for v, w in zip(e, d))
    return out


def row_stats_combine(parts: list) -> dict:
    """Full-row statistics from the shard summaries, given in shard (vocabulary) order."""
    R = len(parts[0]["m"])
    out = {k: np.empty(R) for k in ("m", "lse", "H", "kappa")}
    out["argmax"] = np.zeros(R, np.int64)
    for i in range(R):
        ms = [float(p["m"][i]) for p in parts]
        m = max(ms)
        if m == -math.inf:
            out["m"][i] = -math.inf
            out["lse"][i] = out["H"][i] = out["kappa"][i] = math.nan
            continue
        rstar = ms.index(m)                      # first shard attaining the maximum
        rest_terms, t_terms = [], []
        for r, p in enumerate(parts):
            if ms[r] == -math.inf:
                continue
            s = math.exp(ms[r] - m)
            rest_terms.append(s * float(p["rest"][i]))
            if r != rstar:
                rest_terms.append(s)
            t_terms.append(s * (float(p["t"][i]) + (ms[r] - m) * (float(p["rest"][i]) + 1.0)))
        rest = math.fsum(rest_terms)
        T = math.fsum(t_terms)
        lnZ = math.log1p(rest)
        out["m"][i] = m
        out["argmax"][i] = int(parts[rstar]["a"][i])
        out["lse"][i] = m + lnZ
        out["H"][i] = lnZ - T / (1.0 + rest)
        out["kappa"][i] = lnZ
    return out
