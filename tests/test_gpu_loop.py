"""Parity of the denoising-loop calls (through the C ABI) with the loop oracle.

Bars: order, mask, n_accepted and every field of the loop state bit-exact.  Where the
decisions rest on floating point (a running entropy against its budget, the mean
entropy against the threshold, two kappas), the test asserts that the oracle's values
keep a margin from the decision boundary larger than the fp32 statistics' error, so
that an equality failure is a kernel error and not rounding.
"""
import numpy as np
import pytest
import torch

from denoising_sampler_step_gb300 import inputs
from oracle import row_stats, soft_embed
from oracle.loop_oracle import entropy_accept_eligible, loop_update, new_loop_state
from tests.test_gpu_parity import check_stats, dev, rel_l2, w_dev

pytestmark = pytest.mark.gpu

BUDGET_MARGIN = 1e-4   # nats, as the guarded step workloads
KAPPA_REL = 1e-5
MEAN_H_MARGIN = 1e-3   # nats: the mean of fp32 entropies within 1e-4 of fp64 ones

STATE_KEYS = {"canvas": "canvas", "eligible": "eligible", "prev_argmax": "prev", "stable": "stable",
              "steps": "steps", "converged": "converged"}


@pytest.fixture(scope="module")
def B():
    from denoising_sampler_step_gb300 import build
    build.build()
    from denoising_sampler_step_gb300 import binding
    return binding


def compare_state(g: dict, o: dict, where: str) -> None:
    for gk, ok in STATE_KEYS.items():
        a = g[gk].cpu().numpy().astype(np.int64)
        assert np.array_equal(a, o[ok].astype(np.int64)), (where, gk)


def decision_margins_ok(H, kappa, eligible, n_req, L_c, budgets) -> bool:
    for q in range(n_req):
        sl = slice(q * L_c, (q + 1) * L_c)
        el = np.asarray(eligible[sl]).astype(bool)
        k = np.asarray(kappa[sl], np.float64)[el]
        h = np.asarray(H[sl], np.float64)[el]
        if not np.all(np.isfinite(k)):
            continue
        o = np.argsort(k, kind="stable")
        ks = k[o]
        gaps = np.diff(ks)
        if gaps.size and np.any(gaps <= KAPPA_REL * np.maximum(ks[1:], 1e-300)):
            return False
        if np.any(np.abs(np.cumsum(h[o]) - float(budgets[q])) < BUDGET_MARGIN):
            return False
    return True


# --------------------------------------------------------------------------- acceptance over eligible positions

@pytest.mark.parametrize("L_c,n_req", [(1, 3), (5, 2), (33, 4), (256, 3), (1000, 1), (1024, 2)])
@pytest.mark.parametrize("density", [0.0, 0.3, 0.9, 1.0])
def test_accept_eligible_matches_oracle(B, L_c, n_req, density):
    rng = np.random.default_rng(1000 * L_c + int(density * 10))
    R = L_c * n_req
    H = rng.uniform(0, 3, R).astype(np.float32)
    kappa = rng.uniform(0, 6, R).astype(np.float32)
    kappa[::7] = kappa[0]                      # exact ties: lower position first
    el = (rng.random(R) < density).astype(np.uint8)
    budgets = rng.uniform(0, 1.5 * L_c * max(density, 0.1), n_req).astype(np.float32)
    for min_acc in (0, 3):
        g = B.dg_entropy_accept_eligible(dev(H), dev(kappa), dev(el), n_req, L_c, dev(budgets), min_accept=min_acc)
        o = entropy_accept_eligible(H, kappa, el, n_req, L_c, budgets, min_accept=min_acc)
        for k in ("order", "mask", "n_accepted"):
            assert np.array_equal(g[k].cpu().numpy(), o[k]), (k, min_acc)


def test_accept_eligible_nan_positions_and_full_eligibility(B):
    """A position without a distribution sorts last among the eligible ones; with every
    position eligible the call is the plain acceptance."""
    L = 64
    rng = np.random.default_rng(7)
    H = rng.uniform(0.1, 1, L).astype(np.float32)
    kappa = rng.uniform(0, 5, L).astype(np.float32)
    H[5] = kappa[5] = np.nan
    H[9] = kappa[9] = np.nan
    el = np.ones(L, np.uint8)
    el[9] = 0                                  # an ineligible NaN position
    el[20:30] = 0
    bud = np.array([1e9], np.float32)
    g = B.dg_entropy_accept_eligible(dev(H), dev(kappa), dev(el), 1, L, dev(bud))
    o = entropy_accept_eligible(H, kappa, el, 1, L, bud)
    n_el = int(el.sum())
    assert g["order"][n_el - 1].item() == 5 and g["n_accepted"][0].item() == n_el - 1
    for k in ("order", "mask", "n_accepted"):
        assert np.array_equal(g[k].cpu().numpy(), o[k]), k
    H2, k2 = H.copy(), kappa.copy()
    H2[[5, 9]] = 0.5
    k2[[5, 9]] = 2.5
    one = np.ones(L, np.uint8)
    a = B.dg_entropy_accept_eligible(dev(H2), dev(k2), dev(one), 1, L, dev(np.array([7.0], np.float32)))
    b = B.dg_entropy_accept(dev(H2), dev(k2), 1, L, dev(np.array([7.0], np.float32)))
    for k in ("order", "mask", "n_accepted"):
        assert torch.equal(a[k], b[k]), k


# --------------------------------------------------------------------------- loop-state update

@pytest.mark.parametrize("L_c,n_req", [(1, 3), (37, 3), (256, 2), (1024, 2)])
def test_loop_update_matches_oracle_over_steps(B, L_c, n_req):
    rng = np.random.default_rng(L_c)
    R = L_c * n_req
    stable_steps, step_limit, thr = 2, 9, 1.0
    canvas0 = rng.integers(0, 1000, R)
    o = new_loop_state(n_req, L_c, canvas0=canvas0)
    g = B.new_loop_state(n_req, L_c, "cuda", canvas0=torch.from_numpy(canvas0))
    # request q's entropies sit below the threshold for even q, above it for odd q
    lo = np.where(np.arange(n_req) % 2 == 0, 0.1, 1.1).repeat(L_c)
    cand = rng.integers(0, 50, R).astype(np.int32)
    for t in range(11):
        p_change = [0.5, 0.2, 0.05, 0.0, 0.0, 0.0, 0.3, 0.0, 0.0, 0.0, 0.0][t]
        flip = rng.random(R) < p_change
        cand = np.where(flip, rng.integers(0, 50, R), cand).astype(np.int32)
        H = (lo + rng.uniform(0.0, 0.8, R)).astype(np.float32)
        for q in range(n_req):
            mean = H[q * L_c:(q + 1) * L_c].astype(np.float64).mean()
            assert abs(mean - thr) >= MEAN_H_MARGIN, "redraw: mean entropy on the threshold"
        mask = ((rng.random(R) < 0.2) & (o["eligible"] == 1)).astype(np.uint8)
        B.dg_loop_update(dev(cand), dev(H), dev(mask), n_req, L_c, g, stable_steps, thr, step_limit)
        o = loop_update(o, cand, H, mask, n_req, L_c, stable_steps, thr, step_limit)
        torch.cuda.synchronize()
        compare_state(g, o, f"step {t}")
    B.dg_get_device_status()
    # the sequence reaches every branch: a reset of the stable count, convergence by
    # stability and low entropy (even requests), and by the step limit (odd ones)
    assert o["converged"].all()


def test_loop_update_mean_entropy_is_summed_in_fp64(B):
    """1023 entropies of 1 and one of 1 - 2^-24, threshold 1: the fp64 mean is 1 - 2^-34,
    below the threshold, while any fp32 sum rounds to 1024 and a mean of exactly 1."""
    L = 1024
    H = np.ones(L, np.float32)
    H[0] = np.float32(1.0 - 2.0 ** -24)
    o = new_loop_state(1, L)
    g = B.new_loop_state(1, L, "cuda")
    c = np.zeros(L, np.int32)
    none = np.zeros(L, np.uint8)
    for _ in range(2):
        B.dg_loop_update(dev(c), dev(H), dev(none), 1, L, g, 1, 1.0, 100)
        o = loop_update(o, c, H, none, 1, L, 1, 1.0, 100)
    torch.cuda.synchronize()
    assert o["converged"][0] == 1
    compare_state(g, o, "fp64 mean")


# --------------------------------------------------------------------------- the loop step

LOOP_WL = inputs.WORKLOADS["tiny"].with_(n_req=4, L_c=64, V=40000, d=256, seed=31, budget=("uniform", 4.0, 24.0))
STABLE_STEPS, STEP_LIMIT, N_STEPS = 2, 8, 9


def loop_threshold(base_stats, wl) -> float:
    """A threshold between the requests' mean entropies, so that some converge by
    stability and low entropy and the others only at the step limit."""
    mh = sorted(float(base_stats["H"][q * wl.L_c:(q + 1) * wl.L_c].mean()) for q in range(wl.n_req))
    return (mh[1] + mh[2]) / 2


def test_loop_step_chain_matches_oracle(B):
    """N_STEPS loop steps on logits that settle after four steps: at every step the
    statistics within the step tolerances, and the acceptance over the eligible
    positions, the kept tokens and the whole loop state bit-exact against the oracle
    chain (oracle statistics, oracle acceptance, oracle update) run independently."""
    from denoising_sampler_step_gb300.step import SamplerLoop
    wl = LOOP_WL
    base = inputs.logits(wl)
    thr = loop_threshold(row_stats(base), wl)
    budgets = inputs.budgets(wl)
    Wb = inputs.embedding_bf16(wl)
    lp = SamplerLoop(w_dev(Wb), wl.n_req, wl.L_c, wl.V, wl.gamma, STABLE_STEPS, thr, STEP_LIMIT, min_accept=1)
    bud = dev(budgets)
    o = new_loop_state(wl.n_req, wl.L_c)
    seen_converged = set()
    for t in range(N_STEPS):
        x = inputs.loop_logits(wl, t, base=base)
        st = row_stats(x)
        assert decision_margins_ok(st["H"], st["kappa"], o["eligible"], wl.n_req, wl.L_c, budgets), t
        for q in range(wl.n_req):
            assert abs(st["H"][q * wl.L_c:(q + 1) * wl.L_c].mean() - thr) >= MEAN_H_MARGIN, (t, q)
        out = lp(dev(x), bud)
        torch.cuda.synchronize()
        check_stats(out, st)
        acc = entropy_accept_eligible(st["H"], st["kappa"], o["eligible"], wl.n_req, wl.L_c, budgets, min_accept=1)
        for k in ("order", "mask", "n_accepted"):
            assert np.array_equal(out[k].cpu().numpy(), acc[k]), (t, k)
        o = loop_update(o, st["argmax"], st["H"], acc["mask"], wl.n_req, wl.L_c, STABLE_STEPS, thr, STEP_LIMIT)
        compare_state(lp.state, o, f"step {t}")
        seen_converged |= {(q, int(o["steps"][q])) for q in range(wl.n_req) if o["converged"][q]}
    B.dg_get_device_status()
    rows = np.array([0, 17, 130, wl.R - 1])
    ref = soft_embed(x, st["lse"], 0, wl.V, Wb, wl.gamma, rows=rows)
    assert rel_l2(out["E"].cpu().numpy()[rows], ref).max() <= 1e-2
    # some request converged before the step limit, and every one by it
    assert any(n < STEP_LIMIT for _, n in seen_converged)
    assert o["converged"].all()


def test_loop_steps_in_a_cuda_graph_match_eager_steps(B):
    """Four loop steps captured in one CUDA graph: replayed from the starting state they
    leave the same state and outputs, bit for bit, as four eager calls."""
    from denoising_sampler_step_gb300.step import SamplerLoop
    wl = LOOP_WL.with_(n_req=2, V=30000)
    x = dev(inputs.logits(wl))
    bud = dev(inputs.budgets(wl))
    lp = SamplerLoop(w_dev(inputs.embedding_bf16(wl)), wl.n_req, wl.L_c, wl.V, wl.gamma, 1, 9.0, 3, min_accept=1)
    for _ in range(4):
        lp(x, bud)
    torch.cuda.synchronize()
    eager = {k: v.clone() for k, v in list(lp.out.items()) + list(lp.state.items())}
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        lp.reset()
        lp(x, bud)                             # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(cap)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cap):
        for _ in range(4):
            lp(x, bud)
    lp.reset()
    for v in lp.out.values():
        v.zero_()
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    B.dg_get_device_status()
    now = dict(list(lp.out.items()) + list(lp.state.items()))
    for k, v in eager.items():
        assert torch.equal(now[k], v), k
    assert lp.state["steps"].tolist() == [4, 4] and lp.state["converged"].tolist() == [1, 1]


def test_loop_update_judges_stability_on_the_argmax(B):
    """Candidates (drawn tokens) that change every step, argmax predictions that settle:
    the canvas takes the candidates, the stable count follows the argmax."""
    rng = np.random.default_rng(11)
    n_req, L_c = 3, 50
    R = n_req * L_c
    o = new_loop_state(n_req, L_c)
    g = B.new_loop_state(n_req, L_c, "cuda")
    am = rng.integers(0, 100, R).astype(np.int32)
    for t in range(8):
        if t < 3:
            am = np.where(rng.random(R) < 0.3, rng.integers(0, 100, R), am).astype(np.int32)
        cand = rng.integers(0, 100, R).astype(np.int32)
        H = rng.uniform(0.0, 0.4, R).astype(np.float32)
        mask = ((rng.random(R) < 0.3) & (o["eligible"] == 1)).astype(np.uint8)
        B.dg_loop_update(dev(cand), dev(H), dev(mask), n_req, L_c, g, 3, 1.0, 20, argmax=dev(am))
        o = loop_update(o, cand, H, mask, n_req, L_c, 3, 1.0, 20, argmax=am)
        torch.cuda.synchronize()
        compare_state(g, o, f"step {t}")
    assert o["converged"].all() and (o["stable"] >= 3).all()


SAMPLE_MARGIN = 1e-4   # top-two perturbed scores: the GPU's fp32 scores are within 1e-5
SAMPLED_WL = LOOP_WL.with_(seed=45)


def sampled_chain_inputs(wl, steps, temperature, seed):
    """The oracle chain of a sampling loop, with the margins its exact comparison needs."""
    from oracle import candidate_kappa, row_sample
    base = inputs.logits(wl)
    budgets = inputs.budgets(wl)
    thr = loop_threshold(row_stats(base), wl)
    o = new_loop_state(wl.n_req, wl.L_c)
    chain = []
    for t in range(steps):
        x = inputs.loop_logits(wl, t, base=base)
        st = row_stats(x)
        sm = row_sample(x, temperature, seed, t)
        kc = candidate_kappa(x, sm["candidate"])
        assert np.all((sm["margin"] > SAMPLE_MARGIN) & (sm["group_margin"] > SAMPLE_MARGIN)), ("near-tie draw", t)
        assert decision_margins_ok(st["H"], kc, o["eligible"], wl.n_req, wl.L_c, budgets), t
        for q in range(wl.n_req):
            assert abs(st["H"][q * wl.L_c:(q + 1) * wl.L_c].mean() - thr) >= MEAN_H_MARGIN, (t, q)
        acc = entropy_accept_eligible(st["H"], kc, o["eligible"], wl.n_req, wl.L_c, budgets, min_accept=1)
        o = loop_update(o, sm["candidate"], st["H"], acc["mask"], wl.n_req, wl.L_c, STABLE_STEPS, thr, STEP_LIMIT,
                        argmax=st["argmax"])
        chain.append((x, st, sm, kc, acc, o))
    return budgets, thr, chain


@pytest.mark.parametrize("temperature,two_pass", [(1.0, False), (0.7, False), (0.7, True)])
def test_sampled_loop_chain_matches_oracle(B, temperature, two_pass):
    """A sampling loop (Philox offset = step): at every step the statistics and the draw
    (folded into the single pass, or with two passes the fused statistics + draw pass before
    the product), the acceptance by -ln p of the drawn token over the eligible positions,
    the canvas of drawn tokens and the argmax-judged state, bit-exact against the oracle
    chain."""
    from denoising_sampler_step_gb300.step import SamplerLoop
    wl, seed = SAMPLED_WL, 2024
    budgets, thr, chain = sampled_chain_inputs(wl, N_STEPS, temperature, seed)
    Wb = inputs.embedding_bf16(wl)
    lp = SamplerLoop(w_dev(Wb), wl.n_req, wl.L_c, wl.V, wl.gamma, STABLE_STEPS, thr, STEP_LIMIT,
                     temperature=temperature, seed=seed, min_accept=1, two_pass=two_pass)
    bud = dev(budgets)
    for t, (x, st, sm, kc, acc, o) in enumerate(chain):
        out = lp(dev(x), bud)
        torch.cuda.synchronize()
        check_stats(out, dict(st, kappa=kc))   # kappa: -ln p of the drawn token
        assert np.array_equal(out["candidate"].cpu().numpy(), sm["candidate"]), t
        for key in ("order", "mask", "n_accepted"):
            assert np.array_equal(out[key].cpu().numpy(), acc[key]), (t, key)
        compare_state(lp.state, o, f"step {t}")
    B.dg_get_device_status()
    assert chain[-1][5]["converged"].all()
    # the chain keeps drawn tokens that are not the argmax of their step
    assert any(np.any((sm["candidate"] != st["argmax"]) & (acc["mask"] == 1)) for _, st, sm, _, acc, _ in chain)


def test_sampled_loop_steps_in_a_cuda_graph_match_eager_steps(B):
    """Four loop steps at temperature 1 (the draw folded into the single pass) captured in
    one CUDA graph: replayed from the starting state they give the eager steps' state,
    draws and outputs bit for bit (the graph keeps the offsets it was captured with)."""
    from denoising_sampler_step_gb300.step import SamplerLoop
    wl = LOOP_WL.with_(n_req=2, V=30000)
    x = dev(inputs.logits(wl))
    bud = dev(inputs.budgets(wl))
    lp = SamplerLoop(w_dev(inputs.embedding_bf16(wl)), wl.n_req, wl.L_c, wl.V, wl.gamma, 1, 9.0, 3,
                     temperature=1.0, seed=5, min_accept=1)
    for _ in range(4):
        lp(x, bud)
    torch.cuda.synchronize()
    eager = {k: v.clone() for k, v in list(lp.out.items()) + list(lp.state.items())}
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        lp.reset()
        lp(x, bud)
    torch.cuda.current_stream().wait_stream(cap)
    torch.cuda.synchronize()
    lp.reset()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cap):
        for _ in range(4):
            lp(x, bud)
    lp.reset()
    for v in lp.out.values():
        v.zero_()
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    B.dg_get_device_status()
    now = dict(list(lp.out.items()) + list(lp.state.items()))
    for k, v in eager.items():
        assert torch.equal(now[k].view(torch.int32) if now[k].dtype == torch.float32 else now[k],
                           v.view(torch.int32) if v.dtype == torch.float32 else v), k
