"""Pins of the loop oracle: acceptance over eligible positions against the acceptance
rule on the compacted subset and against brute force; the loop update against
hand-worked step sequences."""
import itertools

import numpy as np
import pytest

from oracle import entropy_accept
from oracle.loop_oracle import entropy_accept_eligible, loop_update, new_loop_state


def draw(L_c, n_req, seed):
    rng = np.random.default_rng(seed)
    H = rng.uniform(0.0, 3.0, n_req * L_c)
    kappa = rng.uniform(0.0, 5.0, n_req * L_c)
    budgets = rng.uniform(1.0, 12.0, n_req)
    return H, kappa, budgets


@pytest.mark.parametrize("seed", range(5))
def test_all_eligible_is_the_plain_rule(seed):
    H, kappa, budgets = draw(40, 3, seed)
    a = entropy_accept_eligible(H, kappa, np.ones(120, np.uint8), 3, 40, budgets, min_accept=2)
    b = entropy_accept(H, kappa, 3, 40, budgets, min_accept=2)
    for k in a:
        assert np.array_equal(a[k], b[k]), k


@pytest.mark.parametrize("seed", range(5))
def test_eligible_subset_is_the_plain_rule_on_the_compacted_positions(seed):
    L_c, n_req = 30, 2
    H, kappa, budgets = draw(L_c, n_req, seed)
    rng = np.random.default_rng(100 + seed)
    el = (rng.random(n_req * L_c) < 0.6).astype(np.uint8)
    a = entropy_accept_eligible(H, kappa, el, n_req, L_c, budgets, min_accept=1)
    for q in range(n_req):
        idx = [j for j in range(L_c) if el[q * L_c + j]]
        b = entropy_accept(H[q * L_c:][idx], kappa[q * L_c:][idx], 1, len(idx), budgets[q:q + 1], min_accept=1)
        order_q = a["order"][q * L_c:(q + 1) * L_c]
        assert list(order_q[:len(idx)]) == [idx[j] for j in b["order"]]
        assert list(order_q[len(idx):]) == [j for j in range(L_c) if not el[q * L_c + j]]
        assert a["n_accepted"][q] == b["n_accepted"][0]
        for j in range(L_c):
            if not el[q * L_c + j]:
                assert a["mask"][q * L_c + j] == 0


@pytest.mark.parametrize("seed", range(20))
def test_eligible_acceptance_brute_force(seed):
    L_c = 9
    H, kappa, budgets = draw(L_c, 1, 200 + seed)
    rng = np.random.default_rng(300 + seed)
    el = (rng.random(L_c) < 0.7).astype(np.uint8)
    a = entropy_accept_eligible(H, kappa, el, 1, L_c, budgets)
    elig = [j for j in range(L_c) if el[j]]
    rank = sorted(elig, key=lambda j: (kappa[j], j))
    best = 0
    for r in range(len(elig) + 1):
        for sub in itertools.combinations(elig, r):
            # downward closed in confidence order: the sub-set is a prefix of `rank`
            if set(sub) == set(rank[:r]) and sum(H[j] for j in sub) <= budgets[0]:
                best = max(best, r)
    assert a["n_accepted"][0] == best
    assert {j for j in range(L_c) if a["mask"][j]} == set(rank[:best])


def test_loop_update_hand_worked_sequence():
    # one request of 4 positions; stable for 2 steps and mean H < 0.5 converges; limit 6
    st = new_loop_state(1, 4, canvas0=[9, 9, 9, 9])
    c = np.array([3, 1, 4, 1])
    low = np.full(4, 0.1)
    m0 = np.array([1, 0, 0, 0], np.uint8)
    st = loop_update(st, c, low, m0, 1, 4, 2, 0.5, 6)       # first step: nothing to compare with
    assert (st["stable"][0], st["steps"][0], st["converged"][0]) == (0, 1, 0)
    assert list(st["canvas"]) == [3, 9, 9, 9] and list(st["eligible"]) == [0, 1, 1, 1]
    st = loop_update(st, c, low, np.zeros(4, np.uint8), 1, 4, 2, 0.5, 6)
    assert (st["stable"][0], st["converged"][0]) == (1, 0)
    st = loop_update(st, c, low, np.zeros(4, np.uint8), 1, 4, 2, 0.5, 6)
    assert (st["stable"][0], st["converged"][0]) == (2, 1)   # stable twice, mean H 0.1
    c2 = np.array([3, 1, 5, 1])                              # one position changes: reset
    st = loop_update(st, c2, low, np.array([0, 1, 1, 0], np.uint8), 1, 4, 2, 0.5, 6)
    assert (st["stable"][0], st["converged"][0]) == (0, 0)
    assert list(st["canvas"]) == [3, 1, 5, 9] and list(st["eligible"]) == [0, 0, 0, 1]


def test_loop_update_entropy_threshold_and_step_limit():
    st = new_loop_state(2, 3)
    c = np.array([1, 2, 3, 1, 2, 3])
    H = np.array([0.5, 0.5, 0.5, 2.0, 2.0, 2.0])   # request 0 mean 0.5, request 1 mean 2.0
    none = np.zeros(6, np.uint8)
    for step in range(1, 5):
        st = loop_update(st, c, H, none, 2, 3, 1, 0.5, 4)
        # request 0: mean H equals the threshold, which is not below it; request 1 is far above
        assert st["converged"][0] == (1 if step >= 4 else 0)
        assert st["converged"][1] == (1 if step >= 4 else 0)
    st = new_loop_state(1, 3)
    for step in range(1, 3):
        st = loop_update(st, c[:3], H[:3], none[:3], 1, 3, 1, 0.5000001, 10)
    assert st["converged"][0] == 1   # stable once and mean H 0.5 < 0.5000001


def test_stability_is_judged_on_the_argmax_and_the_canvas_takes_the_candidates():
    """Sampled candidates that change every step while the argmax predictions stay put:
    the stable count grows; the kept positions take the sampled tokens."""
    st = new_loop_state(1, 3, canvas0=[0, 0, 0])
    am = np.array([7, 8, 9])
    H = np.full(3, 0.1)
    draws = [np.array([1, 2, 3]), np.array([4, 5, 6]), np.array([1, 5, 9])]
    masks = [np.array([1, 0, 0], np.uint8), np.array([0, 1, 0], np.uint8), np.zeros(3, np.uint8)]
    for t in range(3):
        st = loop_update(st, draws[t], H, masks[t], 1, 3, 2, 0.5, 10, argmax=am)
        assert st["stable"][0] == t and list(st["prev"]) == [7, 8, 9]
    assert list(st["canvas"]) == [1, 5, 0] and st["converged"][0] == 1
    # the same candidates with no argmax given: judged on the candidates, never stable
    st2 = new_loop_state(1, 3)
    for t in range(3):
        st2 = loop_update(st2, draws[t], H, masks[t], 1, 3, 2, 0.5, 10)
    assert st2["stable"][0] == 0 and st2["converged"][0] == 0
