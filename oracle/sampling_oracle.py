"""CPU oracle for stochastic candidate sampling (float64, plain and slow).

TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the benchmark's
CPU legs may import this module; the product path never calls it and shares no code
with it.

What it computes.  The sampler draws a candidate token at every canvas position
(agentlenshq.com, "サンプリングループとエントロピー境界デノイジング": candidates are sampled
at every position): a categorical draw from softmax(l / tau).  The page fixes the
distribution, not which random numbers drive it; the draw here is a two-level Gumbel-max,
an exact categorical sampler:

* the vocabulary is cut into groups of 16 consecutive entries, g = v // 16 (the last
  group may be shorter); group g has log-mass L_g = logsumexp_{v in g} (l_v / tau);
* the group is g* = argmax_g (L_g + G_g), G_g = -ln(-ln u_g) (lowest g on ties): by the
  Gumbel-max property P(g*) = exp(L_g) / sum_h exp(L_h);
* inside g*, the candidate is argmax_{v in g*} (l_v / tau + G_v) (lowest v on ties):
  P(v | g*) = exp(l_v / tau - L_g*).  So P(v) = softmax(l / tau)_v.

The uniforms come from a counter-based generator, Philox4x32-10 (Salmon, Moraes, Dror and
Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC 2011), written here from that
definition:

* a round maps the counter (c0, c1, c2, c3) with key (k0, k1) to
  (hi(M1 c2) ^ c1 ^ k0, lo(M1 c2), hi(M0 c0) ^ c3 ^ k1, lo(M0 c0)) with the 32 x 32 -> 64
  bit products of M0 = 0xD2511F53 and M1 = 0xCD9E8D57; the key is bumped by the Weyl
  constants (0x9E3779B9, 0xBB67AE85) between rounds; ten rounds;
* entry v of row `row` takes word v % 4 of the block with counter
  (v // 4, row, offset mod 2^32, offset // 2^32); group g takes word g % 4 of the block
  with counter (2^31 + g // 4, row, offset mod 2^32, offset // 2^32); the key is
  (seed mod 2^32, seed // 2^32) for both;
* u = ((x >> 9) + 1/2) * 2^-23, a value in (0, 1) that float32 holds exactly (24
  significant bits).

Also returned: ln p_tau(candidate) = l_c / tau - logsumexp_v(l_v / tau), the
candidate's log-probability under the tempered softmax.  Entries at -inf are never
drawn (a group with every entry at -inf has L_g = -inf); a row with every entry at -inf
gives candidate 0 and a NaN log-probability.

Also: kappa of a drawn candidate, -ln p(c) under the untempered softmax, the confidence
by which a sampling loop orders its positions (most confident first).  For the argmax
it is ln Z, the row statistics' kappa.

Pinned by tests/test_sampling_pins.py: the published known-answer vectors of
Philox4x32-10, chi-square tests of the draw frequencies against the softmax (rows of one
group and of several), the tau -> 0 limit (the argmax), masked entries and masked groups
never drawn, the log-probability against its closed form, and sum_v exp(-kappa_v) = 1
over every candidate of a row.
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


GROUP = 16                # vocabulary entries per group of the first draw level
GROUP_COUNTER = 2**31     # counter word 0 of the group uniforms starts here


def group_uniforms(R: int, G: int, seed: int, offset: int) -> np.ndarray:
    """The group uniforms u[row, g] (float64 holding the exact fp32 value)."""
    nq = (G + 3) // 4
    q = np.arange(nq, dtype=np.uint64)[None, :] + np.uint64(GROUP_COUNTER)
    rows = np.arange(R, dtype=np.uint64)[:, None]
    ctr = (q, rows, np.uint64(offset & MASK32), np.uint64((offset >> 32) & MASK32))
    key = (np.uint64(seed & MASK32), np.uint64((seed >> 32) & MASK32))
    x = np.stack(philox4x32_10(ctr, key), axis=-1).reshape(R, nq * 4)[:, :G]
    return ((x >> np.uint32(9)).astype(np.float64) + 0.5) * 2.0 ** -23


def _top_two(score: np.ndarray):
    """argmax per row (lowest index on ties) and the margin to the runner-up."""
    best = np.argmax(score, axis=1)
    top = np.take_along_axis(score, best[:, None], axis=1)[:, 0]
    if score.shape[1] > 1:
        rest = score.copy()
        np.put_along_axis(rest, best[:, None], -np.inf, axis=1)
        second = rest.max(axis=1)
    else:
        second = np.full(score.shape[0], -np.inf)
    with np.errstate(invalid="ignore"):
        return best, top - second


def row_sample(logits: np.ndarray, temperature: float, seed: int, offset: int) -> dict:
    """Two-level Gumbel-max candidate per row of the fp32 logits [R, V] at the given
    temperature, with its tempered log-probability.  For tests that compare what is unique,
    also the margins of the two decisions (best minus runner-up: group scores, then entry
    scores inside the chosen group), the chosen group and both score arrays."""
    x = np.asarray(logits, dtype=np.float64)
    R, V = x.shape
    t = float(temperature)
    z = x / t
    G = (V + GROUP - 1) // GROUP
    zp = np.full((R, G * GROUP), -np.inf)
    zp[:, :V] = z
    zg = zp.reshape(R, G, GROUP)
    mg = zg.max(axis=2)
    with np.errstate(invalid="ignore", divide="ignore"):
        Lg = mg + np.log(np.exp(zg - mg[:, :, None]).sum(axis=2))
    Lg = np.where(np.isneginf(mg), -np.inf, Lg)
    ug = group_uniforms(R, G, seed, offset)
    with np.errstate(invalid="ignore"):
        gscore = np.where(np.isneginf(Lg), -np.inf, Lg - np.log(-np.log(ug)))
    gstar, gmargin = _top_two(gscore)
    u = uniforms(R, V, seed, offset)
    with np.errstate(invalid="ignore"):
        escore = np.where(np.isneginf(z), -np.inf, z - np.log(-np.log(u)))
    # entries outside the chosen group take no part in the second draw
    inside = (np.arange(V)[None, :] // GROUP) == gstar[:, None]
    escore_in = np.where(inside, escore, -np.inf)
    cand, emargin = _top_two(escore_in)
    m = z.max(axis=1)
    with np.errstate(invalid="ignore", divide="ignore"):
        lse = m + np.log(np.exp(z - m[:, None]).sum(axis=1))
        log_p = np.take_along_axis(z, cand[:, None], axis=1)[:, 0] - lse
    empty = np.isneginf(m)
    cand = np.where(empty, 0, cand)
    log_p = np.where(empty, np.nan, log_p)
    return {"candidate": cand.astype(np.int32), "log_p": log_p, "group": gstar, "group_score": gscore,
            "group_margin": gmargin, "entry_score": escore, "score": escore_in, "margin": emargin}


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
