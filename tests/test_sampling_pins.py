"""Pins of the sampling oracle against facts that do not come from the oracle itself:
the published known-answer vectors of Philox4x32-10, the categorical distribution of
the two-level Gumbel-max draw (chi-square, within one group and across groups), its
zero-temperature limit (the argmax), masked entries and groups, and the closed form of
the log-probability."""
import math

import numpy as np
import pytest

from oracle.sampling_oracle import candidate_kappa, philox4x32_10, row_sample, uniforms


# Known-answer vectors of Philox4x32-10 published with the generator (Random123):
# (counter, key) -> output, every word hexadecimal.
KAT = [
    ((0x00000000, 0x00000000, 0x00000000, 0x00000000), (0x00000000, 0x00000000),
     (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)),
    ((0xFFFFFFFF, 0xFFFFFFFF, 0xFFFFFFFF, 0xFFFFFFFF), (0xFFFFFFFF, 0xFFFFFFFF),
     (0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD)),
    ((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0),
     (0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1)),
]


@pytest.mark.parametrize("ctr,key,out", KAT)
def test_philox_known_answers(ctr, key, out):
    got = philox4x32_10(tuple(np.uint32(c) for c in ctr), tuple(np.uint32(k) for k in key))
    assert tuple(int(w) for w in got) == out


def test_uniforms_are_inside_the_unit_interval_and_exact_in_fp32():
    u = uniforms(64, 1000, seed=7, offset=3)
    assert u.min() > 0.0 and u.max() < 1.0
    assert np.array_equal(u.astype(np.float32).astype(np.float64), u)
    assert abs(u.mean() - 0.5) < 0.01
    # counter layout: entry v of row r is word v % 4 of block (v // 4, r, offset, 0)
    w = philox4x32_10((np.uint32(2), np.uint32(5), np.uint32(3), np.uint32(0)),
                      (np.uint32(7), np.uint32(0)))
    assert u[5, 9] == ((int(w[1]) >> 9) + 0.5) * 2.0 ** -23


def test_same_counter_same_draw_other_offset_other_draw():
    a = uniforms(4, 64, seed=1, offset=0)
    assert np.array_equal(a, uniforms(4, 64, seed=1, offset=0))
    assert not np.array_equal(a, uniforms(4, 64, seed=1, offset=1))
    assert not np.array_equal(a, uniforms(4, 64, seed=2, offset=0))


@pytest.mark.parametrize("temperature", [1.0, 0.5, 2.0])
def test_gumbel_max_draws_follow_the_tempered_softmax(temperature):
    # 40,000 draws of one 6-entry row (each draw a different row counter); chi-square
    # with 5 degrees of freedom, bound far in the tail (false alarm << 1e-6)
    l = np.array([0.3, -1.2, 2.0, 0.0, 1.1, -0.4], dtype=np.float32)
    n = 40000
    out = row_sample(np.tile(l, (n, 1)), temperature, seed=11, offset=5)
    counts = np.bincount(out["candidate"], minlength=6)
    z = l.astype(np.float64) / temperature
    p = np.exp(z - z.max())
    p /= p.sum()
    chi2 = ((counts - n * p) ** 2 / (n * p)).sum()
    assert chi2 < 45.0, (counts, n * p)


def test_zero_temperature_limit_is_the_argmax():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((200, 300)).astype(np.float32)
    out = row_sample(x, 1e-4, seed=1, offset=0)
    assert np.array_equal(out["candidate"], x.argmax(axis=1))


def test_masked_entries_are_never_drawn_and_empty_rows():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((5000, 16)).astype(np.float32)
    x[:, ::3] = -np.inf
    out = row_sample(x, 1.0, seed=9, offset=2)
    assert np.all(out["candidate"] % 3 != 0)
    e = np.full((2, 8), -np.inf, dtype=np.float32)
    o = row_sample(e, 1.0, seed=9, offset=2)
    assert np.all(o["candidate"] == 0) and np.all(np.isnan(o["log_p"]))


def test_log_probability_closed_form():
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((20, 50)) * 3).astype(np.float32)
    t = 0.7
    out = row_sample(x, t, seed=3, offset=0)
    for i in range(20):
        z = [float(v) / t for v in x[i]]
        lse = math.log(math.fsum(math.exp(v - max(z)) for v in z)) + max(z)
        assert abs(out["log_p"][i] - (z[out["candidate"][i]] - lse)) < 1e-12


def test_candidate_kappa_sums_to_one_over_every_candidate():
    """exp(-kappa_v) is p_v: summed over every candidate of a row it is 1; the uniform row
    gives ln V for every candidate; the argmax gives ln Z (its probability is 1/Z)."""
    rng = np.random.default_rng(5)
    V = 37
    x = (rng.standard_normal((3, V)) * [[0.5], [3.0], [9.0]]).astype(np.float32)
    for i in range(3):
        row = np.repeat(x[i:i + 1], V, axis=0)
        k = candidate_kappa(row, np.arange(V))
        assert math.isclose(math.fsum(np.exp(-k)), 1.0, rel_tol=1e-12)
        a = int(np.argmax(x[i]))
        Z = math.fsum(math.exp(float(v) - float(x[i, a])) for v in x[i])
        assert math.isclose(float(k[a]), math.log(Z), rel_tol=1e-12)
    u = np.zeros((1, V), np.float32)
    assert np.allclose(candidate_kappa(np.repeat(u, V, axis=0), np.arange(V)), math.log(V), rtol=1e-14)
    empty = np.full((1, 4), -np.inf, np.float32)
    assert np.isnan(candidate_kappa(empty, [0])[0])


@pytest.mark.parametrize("temperature", [1.0, 0.6])
def test_draws_across_groups_follow_the_tempered_softmax(temperature):
    # 60,000 draws of one 40-entry row: three groups (16, 16, 8), both levels at work;
    # chi-square with 39 degrees of freedom, bound far in the tail (false alarm << 1e-6)
    rng = np.random.default_rng(21)
    l = (rng.standard_normal(40) * 1.3).astype(np.float32)
    l[33] = 2.5                                   # the short last group holds the most mass
    n = 60000
    out = row_sample(np.tile(l, (n, 1)), temperature, seed=12, offset=1)
    counts = np.bincount(out["candidate"], minlength=40)
    z = l.astype(np.float64) / temperature
    p = np.exp(z - z.max())
    p /= p.sum()
    chi2 = ((counts - n * p) ** 2 / (n * p)).sum()
    assert chi2 < 110.0, (chi2, counts, n * p)
    # the group choice alone follows the group masses
    gc = np.bincount(out["group"], minlength=3)
    pg = np.array([p[:16].sum(), p[16:32].sum(), p[32:].sum()])
    assert ((gc - n * pg) ** 2 / (n * pg)).sum() < 40.0


def test_masked_groups_are_never_chosen():
    rng = np.random.default_rng(6)
    x = rng.standard_normal((3000, 64)).astype(np.float32)
    x[:, 16:32] = -np.inf                          # group 1 entirely masked
    x[:, 50] = -np.inf
    out = row_sample(x, 1.0, seed=4, offset=0)
    assert np.all(out["group"] != 1) and np.all(out["candidate"] != 50)
    assert np.all(out["candidate"] // 16 == out["group"])
