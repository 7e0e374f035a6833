"""CPU oracle for stochastic candidate sampling (float64, plain and slow).

TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the benchmark's
CPU legs may import this module; the product path never calls it and shares no code
with it.

What it computes.  The sampler draws a candidate token at every canvas position
(agentlenshq.com, "サンプリングループとエントロピー境界デノイジング": candidates are sampled
at every position).  The draw is categorical over softmax(l / tau), taken as the
Gumbel-max: candidate = argmax_v (l_v / tau + g_v), g_v = -ln(-ln u_v), which has
exactly the categorical distribution (Gumbel-max property).  The uniforms come from a
counter-based generator, Philox4x32-10 (Salmon, Moraes, Dror and Shaw, "Parallel
random numbers: as easy as 1, 2, 3", SC 2011), written here from that definition:

* a round maps the counter (c0, c1, c2, c3) with key (k0, k1) to
  (hi(M1 c2) ^ c1 ^ k0, lo(M1 c2), hi(M0 c0) ^ c3 ^ k1, lo(M0 c0)) with the 32 x 32 -> 64
  bit products of M0 = 0xD2511F53 and M1 = 0xCD9E8D57; the key is bumped by the Weyl
  constants (0x9E3779B9, 0xBB67AE85) between rounds; ten rounds;
* entry v of row `row` takes word v % 4 of the block with counter
  (v // 4, row, offset mod 2^32, offset // 2^32) and key (seed mod 2^32, seed // 2^32);
* u = ((x >> 9) + 1/2) * 2^-23, a value in (0, 1) that float32 holds exactly (24
  significant bits).

Also returned: ln p_tau(candidate) = l_c / tau - logsumexp_v(l_v / tau), the
candidate's log-probability under the tempered softmax.  Entries at -inf are never
drawn; a row with every entry at -inf gives candidate 0 and a NaN log-probability.

Also: kappa of a drawn candidate, -ln p(c) under the untempered softmax, the confidence
by which a sampling loop orders its positions (most confident first).  For the argmax
it is ln Z, the row statistics' kappa.

Pinned by tests/test_sampling_pins.py: the published known-answer vectors of
Philox4x32-10, a chi-square test of the draw frequencies against the softmax, the
tau -> 0 limit (the argmax), masked entries never drawn, the log-probability against
its closed form, and sum_v exp(-kappa_v) = 1 over every candidate of a row.
"""
from __future__ import annotations

import numpy as np

PHILOX_M0 = 0xD2511F53
PHILOX_M1 = 0xCD9E8D57
PHILOX_W0 = 0x9E3779B9
PHILOX_W1 = 0xBB67AE85
MASK32 = 0xFFFFFFFF


def philox4x32_10(ctr, key):
    """Philox4x32-10 on arrays: ctr is a tuple of four uint32 arrays (broadcastable),
    key a pair of uint32 scalars or arrays.  Returns four uint32 arrays."""
    c0, c1, c2, c3 = (np.asarray(c, dtype=np.uint64) for c in ctr)
    k0 = np.asarray(key[0], dtype=np.uint64)
    k1 = np.asarray(key[1], dtype=np.uint64)
    m0, m1 = np.uint64(PHILOX_M0), np.uint64(PHILOX_M1)
    mask = np.uint64(MASK32)
    for r in range(10):
        p0 = c0 * m0            # 32 x 32 -> 64 bit products, exact in uint64
        p1 = c2 * m1
        hi0, lo0 = p0 >> np.uint64(32), p0 & mask
        hi1, lo1 = p1 >> np.uint64(32), p1 & mask
        c0, c1, c2, c3 = (hi1 ^ c1 ^ k0) & mask, lo1, (hi0 ^ c3 ^ k1) & mask, lo0
        if r < 9:
            k0 = (k0 + np.uint64(PHILOX_W0)) & mask
            k1 = (k1 + np.uint64(PHILOX_W1)) & mask
    return tuple(c.astype(np.uint32) for c in (c0, c1, c2, c3))


def uniforms(R: int, V: int, seed: int, offset: int, row0: int = 0) -> np.ndarray:
    """The uniforms u[row, v] of rows row0 .. row0+R-1 (float64 holding the exact fp32 value)."""
    nq = (V + 3) // 4
    q = np.arange(nq, dtype=np.uint64)[None, :]
    rows = np.arange(row0, row0 + R, dtype=np.uint64)[:, None]
    ctr = (q, rows, np.uint64(offset & MASK32), np.uint64((offset >> 32) & MASK32))
    key = (np.uint64(seed & MASK32), np.uint64((seed >> 32) & MASK32))
    x = np.stack(philox4x32_10(ctr, key), axis=-1).reshape(R, nq * 4)[:, :V]
    return ((x >> np.uint32(9)).astype(np.float64) + 0.5) * 2.0 ** -23


def row_sample(logits: np.ndarray, temperature: float, seed: int, offset: int) -> dict:
    """Gumbel-max candidate per row of the fp32 logits [R, V] at the given temperature,
    with its tempered log-probability and the margin between the best and second-best
    perturbed scores (for tests that compare what is unique)."""
    x = np.asarray(logits, dtype=np.float64)
    R, V = x.shape
    t = float(temperature)
    u = uniforms(R, V, seed, offset)
    g = -np.log(-np.log(u))
    z = x / t
    with np.errstate(invalid="ignore"):
        score = np.where(np.isneginf(x), -np.inf, z + g)
    cand = np.argmax(score, axis=1)
    top = np.take_along_axis(score, cand[:, None], axis=1)[:, 0]
    second = np.where(np.arange(V)[None, :] == cand[:, None], -np.inf, score).max(axis=1) if V > 1 \
        else np.full(R, -np.inf)
    m = z.max(axis=1)
    with np.errstate(invalid="ignore", divide="ignore"):
        lse = m + np.log(np.exp(z - m[:, None]).sum(axis=1))
        log_p = np.take_along_axis(z, cand[:, None], axis=1)[:, 0] - lse
    empty = np.isneginf(m)
    cand = np.where(empty, 0, cand)
    log_p = np.where(empty, np.nan, log_p)
    with np.errstate(invalid="ignore"):
        margin = top - second
    return {"candidate": cand.astype(np.int32), "log_p": log_p, "score": score, "margin": margin}


def candidate_kappa(logits: np.ndarray, candidate) -> np.ndarray:
    """-ln p(candidate_i) under softmax(l_i) (temperature 1), in float64: lse_i - l_{i,c};
    NaN for a row with every entry at -inf."""
    x = np.asarray(logits, dtype=np.float64)
    c = np.asarray(candidate, dtype=np.int64)
    m = x.max(axis=1)
    with np.errstate(invalid="ignore", divide="ignore", over="ignore"):
        lse = m + np.log(np.exp(x - m[:, None]).sum(axis=1))
        k = lse - x[np.arange(x.shape[0]), c]
    return np.where(np.isneginf(m), np.nan, k)
