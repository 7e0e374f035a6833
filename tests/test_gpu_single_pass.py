"""The single-pass step (the product folds the row statistics, the logits are read once)
against the oracle, against the two-pass step, and on the rows it must redo (a split
whose maximum lies far from its reference)."""
import os

import numpy as np
import pytest
import torch

from denoising_sampler_step_gb300 import inputs
from oracle import entropy_accept, row_stats, soft_embed
from tests.test_gpu_parity import E_TOL, check_stats, dev, rel_l2, sampled_rows, w_dev
from tests.workloads import guarded

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from denoising_sampler_step_gb300 import build
    build.build()
    from denoising_sampler_step_gb300 import binding
    return binding


def run_step(B, x, wl, Wd, budgets, V=None, two_pass=False):
    out = B.dg_sampler_step(dev(x), wl.n_req, wl.L_c, Wd, wl.gamma, dev(budgets), V=V, two_pass=two_pass)
    torch.cuda.synchronize()
    B.dg_get_device_status()
    return out


@pytest.mark.parametrize("V,d,L_c,n_req", [(4096, 256, 16, 1), (40001, 256, 64, 2), (70000, 640, 100, 3)])
def test_single_pass_matches_oracle_and_two_pass(B, V, d, L_c, n_req):
    wl = inputs.WORKLOADS["tiny"].with_(V=V, d=d, L_c=L_c, n_req=n_req, seed=V + d, budget=("uniform", 1.0, 12.0))
    ld = (V + 3) // 4 * 4
    x, budgets, ost, _ = guarded(wl, ld=ld)
    Wb = inputs.embedding_bf16(wl)
    Wd = w_dev(Wb)
    one = run_step(B, x, wl, Wd, budgets, V=V)
    check_stats(one, ost)
    acc = entropy_accept(ost["H"], ost["kappa"], wl.n_req, wl.L_c, budgets)
    for k in ("order", "mask", "n_accepted"):
        assert np.array_equal(one[k].cpu().numpy(), acc[k]), k
    E = one["E"].cpu().numpy()
    assert rel_l2(E, soft_embed(x[:, :V], ost["lse"], 0, V, Wb, wl.gamma)).max() <= E_TOL
    two = run_step(B, x, wl, Wd, budgets, V=V, two_pass=True)
    assert torch.equal(one["argmax"], two["argmax"])
    for k in ("order", "mask", "n_accepted"):
        assert torch.equal(one[k], two[k]), k
    # the two passes round different bf16 probabilities (exp(l - c) against exp(l - lse)),
    # so they agree to the tolerance, not to the rounding
    assert rel_l2(E, two["E"].cpu().numpy().astype(np.float64)).max() <= E_TOL


def test_single_pass_redoes_rows_far_from_their_reference(B):
    """Rows whose probabilities against a split's reference could overflow (a one-hot row,
    a logit 90 nats above the rest) go through the redo pass; rows whose splits start
    masked, shifted rows and rows with nothing finite stay in the product: all must give the
    oracle's statistics and embedding."""
    wl = inputs.WORKLOADS["tiny"].with_(V=40000, d=256, L_c=16, n_req=1, seed=3, budget=5.0)
    x = inputs.logits(wl)
    x[0, 12345] = 1.0e4                     # one-hot: overflow against any reference
    x[1, 30000] = 90.0                      # 90 nats above the rest
    x[2, :8192] = -np.inf                   # the first splits start masked
    x[3, :] = -np.inf                       # no distribution
    x[4, :] -= 300.0                        # far below the default reference
    Wb = inputs.embedding_bf16(wl)
    out = run_step(B, x, wl, w_dev(Wb), np.array([5.0], np.float32))
    ost = row_stats(x)
    check_stats(out, ost)
    assert out["argmax"][0].item() == 12345 and out["argmax"][1].item() == 30000
    E = out["E"].cpu().numpy()
    rows = np.array([0, 1, 2, 4, 5, 15])
    assert rel_l2(E[rows], soft_embed(x, ost["lse"], 0, wl.V, Wb, wl.gamma, rows=rows)).max() <= E_TOL
    assert np.all(np.isnan(E[3]))           # a row without a distribution, as in the two-pass step


@pytest.mark.slow
def test_single_pass_canvas256_full_size(B):
    wl = inputs.WORKLOADS["canvas256"]
    x, budgets, ost, _ = guarded(wl)
    Wb = inputs.embedding_bf16(wl)
    out = run_step(B, x, wl, w_dev(Wb), budgets)
    check_stats(out, ost)
    acc = entropy_accept(ost["H"], ost["kappa"], wl.n_req, wl.L_c, budgets)
    for k in ("order", "mask", "n_accepted"):
        assert np.array_equal(out[k].cpu().numpy(), acc[k]), k
    rows = np.arange(wl.R)   # every row
    ref = soft_embed(x, ost["lse"], 0, wl.V, Wb, wl.gamma, rows=rows)
    assert rel_l2(out["E"].cpu().numpy()[rows], ref).max() <= E_TOL


def test_single_pass_largest_canvas(B):
    """1024 positions per request (the acceptance's limit): statistics and E against the
    oracle; the acceptance against the oracle's rule applied to the step's own fp32
    statistics (1024 kappas cannot all be kept 1e-5 apart, so the order is decided on the
    same fp32 values on both sides)."""
    wl = inputs.WORKLOADS["tiny"].with_(V=8192, d=256, L_c=1024, n_req=2, seed=99, budget=("uniform", 5.0, 60.0))
    x = inputs.logits(wl)
    budgets = inputs.budgets(wl)
    Wb = inputs.embedding_bf16(wl)
    out = run_step(B, x, wl, w_dev(Wb), budgets)
    ost = row_stats(x)
    check_stats(out, ost)
    H = out["H"].cpu().numpy().astype(np.float64)
    kappa = out["kappa"].cpu().numpy().astype(np.float64)
    acc = entropy_accept(H, kappa, wl.n_req, wl.L_c, budgets)
    for q in range(wl.n_req):                # the budget decision keeps a margin over the sum order
        sl = slice(q * wl.L_c, (q + 1) * wl.L_c)
        C = np.cumsum(H[sl][acc["order"][sl]])
        assert np.all(np.abs(C - budgets[q]) > 1e-9)
    for k in ("order", "mask", "n_accepted"):
        assert np.array_equal(out[k].cpu().numpy(), acc[k]), k
    rows = np.array([0, 511, 1023, 1024, 2047])
    ref = soft_embed(x, ost["lse"], 0, wl.V, Wb, wl.gamma, rows=rows)
    assert rel_l2(out["E"].cpu().numpy()[rows], ref).max() <= E_TOL


@pytest.mark.parametrize("temperature", [1.0, 0.7, 1.6])
def test_single_pass_draw(B, temperature):
    """A sampling loop step folds the draw into the product: the candidates against the
    two-level oracle draw from softmax(l / T) (unique where both decisions lead by 1e-3),
    kappa = -ln p of the drawn token under softmax(l); rows far from their reference
    (one-hot, 90 nats up, masked starts, shifted) take the fallback folds.  At T = 1 the
    groups' log-masses come from the product's own exponentials, at other T from their own."""
    from oracle import candidate_kappa, row_sample
    from tests.test_gpu_parity import check_sample
    wl = inputs.WORKLOADS["tiny"].with_(V=40000, d=256, L_c=24, n_req=2, seed=17, budget=5.0)
    x = inputs.logits(wl)
    x[0, 12345] = 1.0e4
    x[1, 30000] = 90.0
    x[2, :8192] = -np.inf
    x[4, :] -= 300.0
    x[5, :] = -np.inf
    x[5, [100, 20000]] = 2.0
    Wb = inputs.embedding_bf16(wl)
    Wd = w_dev(Wb)
    state = B.new_loop_state(wl.n_req, wl.L_c, "cuda")
    out = B.dg_sampler_loop_step(dev(x), wl.n_req, wl.L_c, Wd, wl.gamma, dev(inputs.budgets(wl)), state, 2, 1.0, 10,
                                 temperature=temperature, seed=31, offset=4)
    torch.cuda.synchronize()
    B.dg_get_device_status()
    o = row_sample(x, temperature, 31, 4)
    g = {"candidate": out["candidate"], "log_p": torch.from_numpy(o["log_p"].astype(np.float32))}
    check_sample(g, o)
    cand = out["candidate"].cpu().numpy()
    assert cand[0] == 12345 and cand[1] == 30000 and cand[5] in (100, 20000)
    ref = candidate_kappa(x, cand)
    k = out["kappa"].cpu().numpy().astype(np.float64)
    assert np.all(np.abs(k - ref) <= 1e-5 * np.maximum(1.0, ref))
    check_stats({kk: out[kk] for kk in ("m", "lse", "H", "argmax")} | {"kappa": out["kappa"]},
                dict(row_stats(x), kappa=ref))


@pytest.mark.slow
def test_two_pass_canvas256_full_size(B):
    """The two-pass step (statistics before the product) at full size, as the DG_STEP_TWO_PASS
    flag selects it."""
    wl = inputs.WORKLOADS["canvas256"]
    x, budgets, ost, _ = guarded(wl)
    Wb = inputs.embedding_bf16(wl)
    out = run_step(B, x, wl, w_dev(Wb), budgets, two_pass=True)
    check_stats(out, ost)
    acc = entropy_accept(ost["H"], ost["kappa"], wl.n_req, wl.L_c, budgets)
    for k in ("order", "mask", "n_accepted"):
        assert np.array_equal(out[k].cpu().numpy(), acc[k]), k
    rows = np.arange(wl.R)   # every row
    ref = soft_embed(x, ost["lse"], 0, wl.V, Wb, wl.gamma, rows=rows)
    assert rel_l2(out["E"].cpu().numpy()[rows], ref).max() <= E_TOL


def test_single_pass_many_small_requests(B):
    """600 rows as 300 requests of 2 positions: the reduce kernel's acceptance CTAs (one per
    request) far outnumber its reduce CTAs' rows per request."""
    wl = inputs.WORKLOADS["tiny"].with_(n_req=300, L_c=2, seed=11, budget=("uniform", 0.5, 8.0))
    x, budgets, ost, _ = guarded(wl)
    Wb = inputs.embedding_bf16(wl)
    out = run_step(B, x, wl, w_dev(Wb), budgets)
    check_stats(out, ost)
    acc = entropy_accept(ost["H"], ost["kappa"], wl.n_req, wl.L_c, budgets)
    for k in ("order", "mask", "n_accepted"):
        assert np.array_equal(out[k].cpu().numpy(), acc[k]), k
    ref = soft_embed(x, ost["lse"], 0, wl.V, Wb, wl.gamma, rows=np.arange(wl.R))
    assert rel_l2(out["E"].cpu().numpy(), ref).max() <= E_TOL


def test_single_pass_repeats_bit_for_bit_on_a_dirty_workspace(B):
    """Steps on one workspace that starts filled with 0xff bytes, with a plain product on the
    same workspace between them, give the same bits: nothing depends on its prior contents."""
    wl = inputs.WORKLOADS["tiny"].with_(n_req=4, seed=5, budget=("uniform", 0.5, 6.0))
    x, budgets, _, _ = guarded(wl)
    Wb = inputs.embedding_bf16(wl)
    xd, Wd, bd = dev(x), w_dev(Wb), dev(budgets)
    ws = B.workspace(wl.R, wl.V, wl.d, xd.device)
    ws.fill_(255)
    first = B.dg_sampler_step(xd, wl.n_req, wl.L_c, Wd, wl.gamma, bd, ws=ws)
    for _ in range(3):
        B.dg_soft_embed(xd, first["lse"], 0, wl.V, Wd, 1.0, ws=ws)
        again = B.dg_sampler_step(xd, wl.n_req, wl.L_c, Wd, wl.gamma, bd, ws=ws)
        torch.cuda.synchronize()
        for k in ("E", "lse", "H", "kappa", "argmax", "order", "mask", "n_accepted"):
            assert torch.equal(first[k], again[k]), k
    B.dg_get_device_status()
