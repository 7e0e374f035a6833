"""Guarded synthetic workloads for the parity tests (test infrastructure).

The seeded generator draws the inputs; this helper then runs the CPU oracle on
them and redraws (with the next Philox attempt of the same request) any request
whose decisions sit too close to a floating-point tie, so that the exact checks
test the kernels and not the rounding:

* every running entropy C_k of a request is at least BUDGET_MARGIN nats away from
  its budget (the margin the sampler-step benchmark asks for), and
* any two positions of a request differ in kappa = -ln(confidence) by more than
  KAPPA_REL * max(kappa) (fp32 statistics keep five to six decimal digits of kappa).
"""
from __future__ import annotations

import numpy as np

from denoising_sampler_step_gb300 import inputs
from oracle import row_stats

BUDGET_MARGIN = 1e-4
KAPPA_REL = 1e-5
MAX_ATTEMPTS = 40


def request_ok(H: np.ndarray, kappa: np.ndarray, B: float) -> bool:
    if not np.all(np.isfinite(kappa)):
        return True
    srt = np.argsort(kappa, kind="stable")
    ks = kappa[srt]
    gaps = np.diff(ks)
    if gaps.size and np.any(gaps <= KAPPA_REL * np.maximum(ks[1:], 1e-300)):
        return False
    C = np.cumsum(H[srt])
    return bool(np.all(np.abs(C - B) >= BUDGET_MARGIN))


def guarded(wl: inputs.Workload, ld: int | None = None, budgets: np.ndarray | None = None):
    """Returns (logits [R, ld] fp32, budgets [n_req], oracle stats dict, attempts dict)."""
    B = inputs.budgets(wl) if budgets is None else budgets
    attempts = {}
    x = inputs.logits(wl, ld=ld)
    st = row_stats(x[:, :wl.V])
    for q in range(wl.n_req):
        sl = slice(q * wl.L_c, (q + 1) * wl.L_c)
        a = 0
        while not request_ok(st["H"][sl], st["kappa"][sl], float(B[q])):
            a += 1
            if a >= MAX_ATTEMPTS:
                raise RuntimeError(f"request {q} of {wl.name}: no guarded draw in {MAX_ATTEMPTS} attempts")
            rows = inputs.request_logits(wl, q, a)
            x[sl, :wl.V] = rows
            sub = row_stats(rows)
            for k in st:
                st[k][sl] = sub[k]
        if a:
            attempts[q] = a
    return x, B, st, attempts
