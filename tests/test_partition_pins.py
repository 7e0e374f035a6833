"""Pins of the vocabulary-sharded statistics oracle: the combined shard summaries of any
partition give the full-row statistics (themselves pinned by closed forms)."""
import math

import numpy as np
import pytest

from oracle import row_stats
from oracle.partition_oracle import NO_INDEX, row_stats_combine, row_stats_partial


def partition(x, bounds):
    return [row_stats_partial(x[:, s:e], s) for s, e in zip(bounds[:-1], bounds[1:])]


def check_equal(c, full, rows=None):
    idx = np.arange(len(full["m"])) if rows is None else rows
    assert np.array_equal(c["argmax"][idx], full["argmax"][idx])
    for k in ("m", "lse", "H", "kappa"):
        a, b = c[k][idx], full[k][idx]
        assert np.array_equal(np.isnan(a), np.isnan(b)), k
        fin = ~np.isnan(b)
        assert np.allclose(a[fin], b[fin], rtol=1e-12, atol=1e-12), k


@pytest.mark.parametrize("seed", range(4))
def test_random_partitions_give_the_full_row_statistics(seed):
    rng = np.random.default_rng(seed)
    V = 301
    x = (rng.standard_normal((5, V)) * rng.uniform(0.3, 6.0, (5, 1))).astype(np.float32)
    x[1, 17] += 20.0                                        # a peaked row
    cuts = np.sort(rng.choice(np.arange(1, V), size=rng.integers(1, 7), replace=False))
    bounds = [0] + list(cuts) + [V]
    check_equal(row_stats_combine(partition(x, bounds)), row_stats(x))
    # one shard: the summary alone is the row
    check_equal(row_stats_combine(partition(x, [0, V])), row_stats(x))


def test_single_entry_and_empty_shards():
    rng = np.random.default_rng(9)
    V = 40
    x = rng.standard_normal((3, V)).astype(np.float32)
    x[0, 10:20] = -np.inf                                   # shard [10, 20) empty for row 0
    x[2, :] = -np.inf                                       # no distribution at all
    bounds = [0, 1, 10, 20, 21, 40]
    parts = partition(x, bounds)
    assert parts[2]["m"][0] == -np.inf and parts[2]["a"][0] == NO_INDEX
    c = row_stats_combine(parts)
    check_equal(c, row_stats(x))
    assert math.isnan(c["H"][2]) and c["argmax"][2] == 0


def test_maximum_tied_across_a_shard_boundary_takes_the_lowest_index():
    x = np.zeros((2, 12), np.float32)
    x[0, [3, 9]] = 5.0                                      # tie between shards 0 and 1
    x[1, [7, 8]] = 5.0                                      # tie inside shard 1
    c = row_stats_combine(partition(x, [0, 6, 12]))
    assert list(c["argmax"]) == [3, 7]
    check_equal(c, row_stats(x))
    # the regrouping keeps kappa's precision near one-hot: rest is never formed as Z - 1
    y = np.full((1, 64), -30.0, np.float32)
    y[0, 40] = 0.0
    cy = row_stats_combine(partition(y, [0, 16, 32, 48, 64]))
    assert math.isclose(cy["kappa"][0], math.log1p(63 * math.exp(-30.0)), rel_tol=1e-12)
