"""CPU oracle for the denoising-loop state (plain Python/numpy, float64 where it sums).

TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the benchmark's
CPU legs may import this module; the product path never calls it and shares no code
with it.

What it computes (agentlenshq.com, "サンプリングループとエントロピー境界デノイジング"):
the loop samples a candidate at every position, keeps tokens from most to least
confident while the cumulative entropy stays within the budget, and a canvas has
converged when the argmax predictions have been stable for several steps and the mean
entropy per token is below a threshold, or when the step limit is reached.  Where the
page is silent the readings are:

* a kept (accepted) position keeps its token and is no longer offered for acceptance
  (it is not eligible) until the canvas commits;
* "stable for several steps": every position's argmax prediction equals the previous
  step's, counted in consecutive steps (the page speaks of the argmax predictions; the
  canvas may take sampled candidates, which need not be stable);
* "mean entropy per token": the mean of H over all L_c positions of the canvas.

Pinned by tests/test_loop_pins.py: acceptance over the eligible positions equals the
acceptance of the compacted eligible subset and brute force over subsets; the loop
update against hand-worked step sequences.
"""
from __future__ import annotations

import math

import numpy as np


def entropy_accept_eligible(H, kappa, eligible, n_req: int, L_c: int, budgets, min_accept: int = 0) -> dict:
    """Entropy-bound acceptance restricted to eligible positions.

    For request q: the eligible positions are ordered from most to least confident
    (kappa ascending, ties by the lower position, positions without a distribution --
    NaN statistics -- after every other eligible one); the ineligible positions follow,
    in position order.  C_k sums H over the first k eligible positions; n is the largest
    k with C_k <= B_q (taking stops at the first that would pass it), raised to
    min(min_accept, number eligible); mask[order_j] = 1 for j < n.  Ineligible positions
    are never kept and carry no entropy into the sum."""
    H = np.asarray(H, np.float64)
    kappa = np.asarray(kappa, np.float64)
    el = np.asarray(eligible).astype(bool)
    R = n_req * L_c
    order = np.empty(R, np.int64)
    mask = np.zeros(R, np.uint8)
    n_acc = np.empty(n_req, np.int64)
    for q in range(n_req):
        base = q * L_c
        elig = [j for j in range(L_c) if el[base + j]]
        rest = [j for j in range(L_c) if not el[base + j]]
        pos = sorted(elig, key=lambda j: (bool(math.isnan(kappa[base + j])), kappa[base + j], j)) + rest
        B = float(budgets[q])
        running, n = 0.0, 0
        for k, j in enumerate(pos[:len(elig)]):
            running += H[base + j]
            if running <= B:
                n = k + 1
            else:
                break
        n = max(n, min(int(min_accept), len(elig)))
        for k, j in enumerate(pos):
            order[base + k] = j
            if k < n:
                mask[base + j] = 1
        n_acc[q] = n
    return {"order": order, "mask": mask, "n_accepted": n_acc}


def new_loop_state(n_req: int, L_c: int, canvas0=None) -> dict:
    """The state a canvas starts from: no previous argmax (-1), no stable step, no step
    taken, every position eligible, the canvas as given (zeros if not)."""
    R = n_req * L_c
    return {"canvas": np.zeros(R, np.int64) if canvas0 is None else np.array(canvas0, np.int64),
            "eligible": np.ones(R, np.uint8), "prev": np.full(R, -1, np.int64),
            "stable": np.zeros(n_req, np.int64), "steps": np.zeros(n_req, np.int64),
            "converged": np.zeros(n_req, np.uint8)}


def loop_update(state: dict, candidate, H, mask, n_req: int, L_c: int, stable_steps: int,
                entropy_threshold: float, step_limit: int, argmax=None) -> dict:
    """One step of the loop state, per request q (positions q*L_c .. q*L_c + L_c - 1):
      canvas[pos] = candidate[pos] and eligible[pos] = 0 where mask[pos] (kept tokens);
      stable[q] = stable[q] + 1 if every argmax prediction equals prev at its position,
                  else 0 (argmax defaults to the candidates: an argmax loop);
      prev = argmax;  steps[q] += 1;
      mean_H = (sum of H over the request's positions, in position order) / L_c;
      converged[q] = (stable[q] >= stable_steps and mean_H < entropy_threshold)
                     or steps[q] >= step_limit.
    Returns a new state dict."""
    cand = np.asarray(candidate, np.int64)
    am = cand if argmax is None else np.asarray(argmax, np.int64)
    H = np.asarray(H, np.float64)
    m = np.asarray(mask).astype(bool)
    s = {k: v.copy() for k, v in state.items()}
    for q in range(n_req):
        sl = slice(q * L_c, (q + 1) * L_c)
        same = bool(np.all(am[sl] == s["prev"][sl]))
        s["stable"][q] = s["stable"][q] + 1 if same else 0
        s["steps"][q] += 1
        mean_H = math.fsum(float(h) for h in H[sl]) / L_c
        s["converged"][q] = 1 if ((s["stable"][q] >= stable_steps and mean_H < entropy_threshold)
                                  or s["steps"][q] >= step_limit) else 0
    s["canvas"] = np.where(m, cand, s["canvas"])
    s["eligible"] = np.where(m, 0, s["eligible"]).astype(np.uint8)
    s["prev"] = am.copy()
    return s
