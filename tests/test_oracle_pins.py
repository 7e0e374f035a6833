"""Pins of the CPU oracle to facts the pages and the mathematics fix.

Each test checks the oracle against something other than itself: a closed form,
an identity computed by a different route, brute force over all orderings or
subsets, or numbers the pages print.  A plausible slip in the oracle (a dropped
term, a sign, an index, a transposed operand, renormalising inside a slice)
fails at least one of them.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

from oracle import entropy_accept, row_stats, soft_embed, sum_partials
from denoising_sampler_step_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
NEG_INF = np.float32(-np.inf)


# ----------------------------------------------------------------------------- row statistics

@pytest.mark.parametrize("V,c", [(4096, 0.0), (4096, 3.7), (262144, -1.25)])
def test_uniform_row_entropy_is_ln_V(V, c):
    st = row_stats(np.full((1, V), c, np.float32))
    assert st["argmax"][0] == 0
    assert abs(st["H"][0] - math.log(V)) < 1e-9
    assert abs(st["kappa"][0] - math.log(V)) < 1e-9
    assert abs(st["conf"][0] - 1.0 / V) < 1e-15
    assert abs(st["lse"][0] - (float(np.float32(c)) + math.log(V))) < 1e-9
    assert st["m"][0] == np.float32(c)


def test_k_way_tie_with_rest_masked():
    row = np.full(64, NEG_INF, np.float32)
    row[[5, 9, 20]] = 1.5
    st = row_stats(row[None])
    assert st["argmax"][0] == 5
    assert abs(st["H"][0] - math.log(3)) < 1e-12
    assert abs(st["kappa"][0] - math.log(3)) < 1e-12
    assert abs(st["lse"][0] - (1.5 + math.log(3))) < 1e-12


def test_one_hot_row():
    row = np.zeros(1000, np.float32)
    row[417] = 1e4
    st = row_stats(row[None])
    assert st["argmax"][0] == 417
    assert st["H"][0] == 0.0 and st["kappa"][0] == 0.0 and st["conf"][0] == 1.0


@pytest.mark.parametrize("t", [0.0, 0.3, -2.0, 5.0])
def test_two_point_row_is_binary_entropy(t):
    row = np.full(10, NEG_INF, np.float32)
    row[2], row[7] = 0.0, t
    t32 = float(np.float32(t))
    q = 1.0 / (1.0 + math.exp(-t32))          # probability of index 7
    H = -(q * math.log(q) + (1 - q) * math.log(1 - q))
    st = row_stats(row[None])
    assert abs(st["H"][0] - H) < 1e-12
    assert st["argmax"][0] == (7 if t32 > 0 else 2)
    assert abs(st["conf"][0] - max(q, 1 - q)) < 1e-12


def test_argmax_takes_lowest_index_on_ties():
    row = np.random.default_rng(0).standard_normal(300).astype(np.float32)
    row[40] = row[210] = 9.0
    st = row_stats(row[None])
    assert st["argmax"][0] == 40
    # the tied twin counts toward kappa: Z >= 2, so conf <= 1/2
    assert st["conf"][0] <= 0.5 and st["kappa"][0] >= math.log(2)


def test_all_masked_row_gives_nan():
    st = row_stats(np.full((1, 16), NEG_INF, np.float32))
    assert np.isnan(st["H"][0]) and np.isnan(st["lse"][0]) and st["argmax"][0] == 0


def _brute_stats(row):
    """Pure-Python row statistics by another route: H = lse - sum_v p_v l_v."""
    vals = [float(x) for x in row]
    m = max(vals)
    lse = m + math.log(math.fsum(math.exp(x - m) for x in vals))
    p = [math.exp(x - lse) for x in vals]
    H = lse - math.fsum(pi * x for pi, x in zip(p, vals))
    return m, vals.index(m), lse, H, -math.log(max(p))


def test_random_rows_against_pure_python():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal((6, 257)) * rng.uniform(0.2, 6, (6, 1))).astype(np.float32)
    st = row_stats(x)
    for i in range(6):
        m, a, lse, H, kap = _brute_stats(x[i])
        assert st["m"][i] == m and st["argmax"][i] == a
        assert abs(st["lse"][i] - lse) < 1e-12
        assert abs(st["H"][i] - H) < 1e-11
        assert abs(st["kappa"][i] - kap) < 1e-11


def test_shift_invariance_and_bounds():
    rng = np.random.default_rng(2)
    x = (rng.standard_normal((4, 4096)) * 3).astype(np.float32)
    a, b = row_stats(x), row_stats(x + np.float32(16.0))   # exact shift in fp32 at these magnitudes
    assert np.array_equal(a["argmax"], b["argmax"])
    assert np.allclose(a["H"], b["H"], atol=1e-10) and np.allclose(a["kappa"], b["kappa"], atol=1e-10)
    assert np.allclose(b["lse"] - a["lse"], 16.0, atol=1e-9)
    assert np.all(a["H"] >= 0) and np.all(a["H"] <= math.log(4096) + 1e-12)


def test_masked_entries_are_skipped():
    rng = np.random.default_rng(3)
    x = rng.standard_normal(50).astype(np.float32)
    y = np.full(80, NEG_INF, np.float32)
    y[15:65] = x
    sx, sy = row_stats(x[None]), row_stats(y[None])
    assert abs(sx["H"][0] - sy["H"][0]) < 1e-12 and abs(sx["lse"][0] - sy["lse"][0]) < 1e-12
    assert sy["argmax"][0] == sx["argmax"][0] + 15


def test_kappa_resolves_near_one_hot_rows():
    # 1/Z rounds to exactly 1 here, but kappa = log1p(rest) still orders the rows
    rows = np.zeros((3, 100), np.float32)
    rows[:, 0] = [60.0, 61.0, 62.0]
    st = row_stats(rows)
    assert np.all(st["conf"] == 1.0)
    assert st["kappa"][0] > st["kappa"][1] > st["kappa"][2] > 0
    assert abs(st["kappa"][1] - 99 * math.exp(-61.0)) < 1e-30


# ----------------------------------------------------------------------------- acceptance

def _worked():
    with open(os.path.join(GOLDEN, "accept_worked_example.json")) as f:
        return json.load(f)


def test_worked_example():
    g = _worked()
    kappa = -np.log(np.array(g["conf"]))
    H = np.array(g["H"])
    for case in g["cases"]:
        out = entropy_accept(H, kappa, 1, g["L_c"], np.array([case["budget"]]))
        assert list(out["order"]) == case["order"], case
        assert list(out["mask"]) == case["mask"], case
        assert out["n_accepted"][0] == case["n_accepted"], case


def _more_confident(kappa, i, j):
    """Position i precedes position j: strictly higher confidence, or equal and lower index."""
    return kappa[i] < kappa[j] or (kappa[i] == kappa[j] and i < j)


def _brute_perm(H, kappa, B):
    L = len(H)
    (order,) = [p for p in itertools.permutations(range(L))
                if all(_more_confident(kappa, p[k], p[k + 1]) for k in range(L - 1))]
    n = 0
    for k in range(1, L + 1):
        if math.fsum(H[list(order[:k])]) <= B:
            n = k
        else:
            break
    return list(order), n


def _brute_subsets(H, kappa, B):
    L = len(H)
    best = ()
    for bits in range(1 << L):
        S = [j for j in range(L) if bits >> j & 1]
        closed = all(i in S for j in S for i in range(L) if _more_confident(kappa, i, j))
        if closed and math.fsum(H[S]) <= B and len(S) > len(best):
            best = tuple(S)
    return sorted(best)


@pytest.mark.parametrize("seed", range(12))
def test_acceptance_brute_force(seed):
    rng = np.random.default_rng(100 + seed)
    L = 6 if seed % 2 else 7
    H = rng.uniform(0, 3, L)
    kappa = rng.choice(rng.uniform(0, 4, 4), L)      # repeated values force tie-breaking
    Hs = np.sort(H)
    for B in [0.0, Hs[0] * 0.5, float(np.sum(H)) * 0.4, float(np.sum(H)) * 0.8, float(np.sum(H)) + 1]:
        out = entropy_accept(H, kappa, 1, L, np.array([B]))
        order, n = _brute_perm(H, kappa, B)
        assert list(out["order"]) == order
        assert out["n_accepted"][0] == n
        assert sorted(np.nonzero(out["mask"])[0]) == _brute_subsets(H, kappa, B)


def test_budget_sweep_hits_every_n():
    rng = np.random.default_rng(7)
    L = 16
    H = rng.uniform(0.1, 2, L)
    kappa = rng.uniform(0, 5, L)
    srt = sorted(range(L), key=lambda j: (kappa[j], j))
    C = np.cumsum(H[srt])
    for n in range(L + 1):
        lo = 0.0 if n == 0 else C[n - 1]
        hi = C[n] if n < L else C[-1] + 1.0
        B = 0.5 * (lo + hi) if n > 0 else 0.5 * C[0]
        out = entropy_accept(H, kappa, 1, L, np.array([B]))
        assert out["n_accepted"][0] == n
        assert set(np.nonzero(out["mask"])[0]) == set(srt[:n])


def test_min_accept_and_requests_are_independent():
    rng = np.random.default_rng(8)
    n_req, L = 3, 8
    H = rng.uniform(1, 2, n_req * L)
    kappa = rng.uniform(0, 5, n_req * L)
    B = np.array([0.5, 100.0, 3.0])
    lit = entropy_accept(H, kappa, n_req, L, B)
    assert list(lit["n_accepted"][:2]) == [0, L]
    forced = entropy_accept(H, kappa, n_req, L, B, min_accept=2)
    assert list(forced["n_accepted"]) == [2, L, max(2, lit["n_accepted"][2])]
    for q in range(n_req):     # each request alone gives the same answer
        one = entropy_accept(H[q * L:(q + 1) * L], kappa[q * L:(q + 1) * L], 1, L, B[q:q + 1])
        assert np.array_equal(one["order"], lit["order"][q * L:(q + 1) * L])
        assert np.array_equal(one["mask"], lit["mask"][q * L:(q + 1) * L])


# ----------------------------------------------------------------------------- soft embedding

def _w(V, d, seed=0):
    rng = np.random.default_rng(seed)
    return inputs.f32_to_bf16_bits((rng.standard_normal((V, d)) * 0.02).astype(np.float32))


def _w64(bits):
    return inputs.bf16_bits_to_f32(bits).astype(np.float64)


def test_one_hot_rows_return_gamma_times_embedding_row():
    V, d, gamma = 300, 24, 16.0
    Wb = _w(V, d)
    x = np.zeros((3, V), np.float32)
    hot = [0, 123, 299]
    x[np.arange(3), hot] = 1e4
    st = row_stats(x)
    E = soft_embed(x, st["lse"], 0, V, Wb, gamma)
    assert np.array_equal(E, gamma * _w64(Wb)[hot])


def test_uniform_rows_return_gamma_times_column_mean():
    V, d, gamma = 512, 16, 53.0
    Wb = _w(V, d, 1)
    x = np.full((2, V), -0.75, np.float32)
    st = row_stats(x)
    E = soft_embed(x, st["lse"], 0, V, Wb, gamma)
    W = _w64(Wb)
    mean = np.array([math.fsum(W[:, c]) / V for c in range(d)])
    assert np.allclose(E, gamma * mean[None], rtol=1e-12, atol=1e-15)


def test_against_pure_python_triple_loop():
    R, V, d, gamma = 3, 7, 5, 2.5
    rng = np.random.default_rng(4)
    x = (rng.standard_normal((R, V)) * 2).astype(np.float32)
    Wb = _w(V, d, 2)
    W = _w64(Wb)
    st = row_stats(x)
    E = soft_embed(x, st["lse"], 0, V, Wb, gamma)
    for i in range(R):
        l = [float(v) for v in x[i]]
        m = max(l)
        Z = math.fsum(math.exp(v - m) for v in l)
        for c in range(d):
            ref = gamma * math.fsum(math.exp(l[v] - m) / Z * W[v, c] for v in range(V))
            assert abs(E[i, c] - ref) <= 1e-13 * max(1.0, abs(ref))


def test_linear_in_gamma_and_permutation_invariant():
    R, V, d = 4, 200, 8
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((R, V)) * 3).astype(np.float32)
    Wb = _w(V, d, 3)
    st = row_stats(x)
    E1 = soft_embed(x, st["lse"], 0, V, Wb, 1.0)
    assert np.allclose(soft_embed(x, st["lse"], 0, V, Wb, 3.0), 3.0 * E1, rtol=1e-14, atol=0)
    perm = rng.permutation(V)
    Ep = soft_embed(x[:, perm], st["lse"], 0, V, Wb[perm], 1.0)
    assert np.allclose(Ep, E1, rtol=1e-12, atol=1e-16)


def test_partition_identity_and_padding_never_read():
    R, V, d, gamma = 5, 4096, 32, 16.0
    rng = np.random.default_rng(6)
    x = (rng.standard_normal((R, V)) * 2).astype(np.float32)
    Wb = _w(V, d, 4)
    st = row_stats(x)
    full = soft_embed(x, st["lse"], 0, V, Wb, gamma)
    for bounds in ([(0, 1000), (1000, 2100), (2100, 3333), (3333, 4096)], inputs.slice_bounds(V, 4)):
        parts = []
        for s, e in bounds:
            shard = inputs.padded_shard(Wb, s, e, 128, pad_value="nan")
            parts.append(soft_embed(x, st["lse"], s, e, shard, 1.0))
        summed = sum_partials(parts, gamma)
        assert np.all(np.isfinite(summed))
        assert np.allclose(summed, full, rtol=1e-12, atol=1e-15)
    # each slice keeps the global normalisation: its row sums of P are the slice's share of mass
    ones = inputs.f32_to_bf16_bits(np.ones((V, 1), np.float32))
    mass = soft_embed(x, st["lse"], 0, V, ones, 1.0)[:, 0]
    assert np.allclose(mass, 1.0, atol=1e-12)
    half = soft_embed(x, st["lse"], 0, V // 2, ones[: V // 2], 1.0)[:, 0]
    assert np.all(half < 1.0)


def test_row_subset_matches_full():
    R, V, d = 6, 300, 8
    rng = np.random.default_rng(9)
    x = (rng.standard_normal((R, V))).astype(np.float32)
    Wb = _w(V, d, 5)
    st = row_stats(x)
    full = soft_embed(x, st["lse"], 0, V, Wb, 2.0)
    sub = soft_embed(x, st["lse"], 0, V, Wb, 2.0, rows=np.array([4, 1]))
    assert np.array_equal(sub, full[[4, 1]])


def test_position_without_distribution_goes_last_and_stops_the_sum():
    H = np.array([0.5, np.nan, 0.2, 0.1])
    kappa = np.array([1.0, np.nan, 0.5, 2.0])
    out = entropy_accept(H, kappa, 1, 4, np.array([100.0]))
    assert list(out["order"]) == [2, 0, 3, 1]
    assert out["n_accepted"][0] == 3 and list(out["mask"]) == [1, 0, 1, 1]
