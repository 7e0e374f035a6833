"""The 8-bit embedding table on the GPU (through the C ABI) against the oracle: the per-row
E4M3 quantiser bit for bit, the block-scaled product within the soft-embedding tolerance
(ragged tiles, slices that start and end off a block, column tails), and the step with the
8-bit table in both of its forms (statistics first, and the single pass with its redo rows)."""
import os

import numpy as np
import pytest
import torch

from denoising_sampler_step_gb300 import inputs
from oracle import entropy_accept, row_stats
from oracle.quant_oracle import dequantize_rows_e4m3, quantize_rows_e4m3, soft_embed_e4m3
from tests.test_gpu_parity import E_TOL, check_stats, dev, rel_l2, sampled_rows, w_dev
from tests.workloads import guarded

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from denoising_sampler_step_gb300 import build
    build.build()
    from denoising_sampler_step_gb300 import binding
    return binding


def q_dev(Q, pad_rows=0, fill=0x7F):
    """Codes on the device in rows padded to a multiple of 16 bytes (padding NaN codes: never
    read), plus `pad_rows` rows of NaN codes after the table."""
    V, d = Q.shape
    ldq = (d + 15) // 16 * 16
    buf = np.full((V + pad_rows, ldq), fill, np.uint8)
    buf[:V, :d] = Q
    return dev(buf)[:, :d]


def s_dev(scale, pad_rows=0):
    return dev(np.concatenate([scale, np.full(pad_rows, np.nan, np.float32)]).astype(np.float32))


# --------------------------------------------------------------------------- quantiser

@pytest.mark.parametrize("V,d,ldw", [(3000, 2816, 2816), (777, 257, 258), (64, 16, 16)])
def test_quantiser_is_bit_exact(B, V, d, ldw):
    wl = inputs.WORKLOADS["tiny"].with_(V=V, d=d, seed=d)
    bits = inputs.embedding_bf16(wl)
    bits[1] = 0                                                   # a zero row
    bits[2, ::2] = 0x8000                                         # negative zeros
    bits[3, 5] = inputs.f32_to_bf16_bits(np.array([-0.75], np.float32))[0]   # a negative row maximum
    bits[4] = inputs.f32_to_bf16_bits(np.linspace(-1e-3, 1e-3, d).astype(np.float32))  # codes down to subnormal
    Qo, so = quantize_rows_e4m3(bits)
    buf = np.zeros((V, ldw), np.uint16)
    buf[:, :d] = bits
    Wd = w_dev(buf)[:, :d]
    Q, scale = B.dg_quantize_e4m3(Wd)
    torch.cuda.synchronize()
    assert np.array_equal(scale.cpu().numpy().view(np.uint32), so.view(np.uint32))
    Qg = Q.cpu().numpy()
    bad = np.argwhere(Qg != Qo)
    assert bad.size == 0, (bad[:5], Qg[tuple(bad[0])], Qo[tuple(bad[0])])


# --------------------------------------------------------------------------- product

@pytest.mark.parametrize("V,d,R,s,e", [
    (4096, 256, 128, 0, 4096),        # one column tile, one row block
    (40001, 640, 300, 0, 40001),      # a 480-column tile and a tail of 160, ragged rows, ragged vocabulary
    (40001, 1000, 256, 3, 39990),     # a slice off the block grid at both ends (scalar scale loads), tail of 40
    (20000, 2816, 64, 0, 20000),      # the model's hidden size: five full tiles and a tail of 416
])
def test_product_matches_oracle(B, V, d, R, s, e):
    wl = inputs.WORKLOADS["tiny"].with_(V=V, d=d, L_c=R, n_req=1, seed=V + d)
    ld = (V + 3) // 4 * 4
    x = inputs.logits(wl, ld=ld)
    Q, scale = inputs.embedding_e4m3(wl)
    st = row_stats(x[:, :V])
    Qd, sd = q_dev(Q[s:e], pad_rows=7), s_dev(scale[s:e], pad_rows=7)
    out = B.dg_soft_embed_e4m3(dev(x), dev(st["lse"].astype(np.float32)), s, e, Qd, sd, wl.gamma)
    torch.cuda.synchronize()
    B.dg_get_device_status()
    ref = soft_embed_e4m3(x[:, :V], st["lse"], s, e, Q[s:e], scale[s:e], wl.gamma)
    err = rel_l2(out.cpu().numpy(), ref)
    assert err.max() <= E_TOL, float(err.max())


def test_product_matches_the_bf16_product_on_a_shared_table(B):
    """A table that both formats hold exactly (power-of-two row scales): the 8-bit and the bf16
    products round the probabilities differently, so they agree to the tolerance."""
    wl = inputs.WORKLOADS["tiny"].with_(V=30000, d=512, L_c=256, n_req=1, seed=21)
    x = inputs.logits(wl)
    Q, _ = inputs.embedding_e4m3(wl)
    scale = np.full(wl.V, 2.0 ** -12, np.float32)
    W = dequantize_rows_e4m3(Q, scale).astype(np.float32)
    bits = inputs.f32_to_bf16_bits(W)
    assert np.array_equal(inputs.bf16_bits_to_f32(bits), W)
    lse = B.dg_row_stats(dev(x))["lse"]
    e8 = B.dg_soft_embed_e4m3(dev(x), lse, 0, wl.V, q_dev(Q), s_dev(scale), 1.0).cpu().numpy()
    e16 = B.dg_soft_embed(dev(x), lse, 0, wl.V, w_dev(bits), 1.0).cpu().numpy()
    assert rel_l2(e8, e16.astype(np.float64)).max() <= E_TOL


def test_product_blocks_with_wide_scale_ranges(B):
    """Rows whose probabilities and row scales span many decades inside one 32-entry block:
    the per-(row, block) exponent and the high/low split must keep the large entries exact to
    about eight bits and not lose the small ones that matter."""
    wl = inputs.WORKLOADS["tiny"].with_(V=8192, d=480, L_c=128, n_req=1, seed=4)
    x = inputs.logits(wl)
    x[0, :] = -np.inf
    x[0, 100:132] = np.linspace(0.0, -25.0, 32)                # one block, 25 nats of range
    x[1, ::2] -= 30.0                                         # alternate entries 30 nats down
    Q, scale = inputs.embedding_e4m3(wl)
    scale[100:132] = np.logspace(2, -6, 32).astype(np.float32)    # row scales falling over eight decades
    st = row_stats(x)
    out = B.dg_soft_embed_e4m3(dev(x), dev(st["lse"].astype(np.float32)), 0, wl.V, q_dev(Q), s_dev(scale), 1.0)
    ref = soft_embed_e4m3(x, st["lse"], 0, wl.V, Q, scale, 1.0)
    err = rel_l2(out.cpu().numpy(), ref)
    assert err.max() <= E_TOL, float(err.max())
    assert err[0] <= 5e-3


# --------------------------------------------------------------------------- step

def run_step(B, x, wl, Qd, sd, budgets, V=None, two_pass=False):
    out = B.dg_sampler_step_e4m3(dev(x), wl.n_req, wl.L_c, Qd, sd, wl.gamma, dev(budgets), V=V, two_pass=two_pass)
    torch.cuda.synchronize()
    B.dg_get_device_status()
    return out


@pytest.mark.parametrize("single", [True, False])
def test_step_matches_oracle(B, single):
    wl = inputs.WORKLOADS["tiny"].with_(V=40001, d=1000, L_c=64, n_req=3, seed=8, budget=("uniform", 1.0, 12.0))
    x, budgets, ost, _ = guarded(wl, ld=40004)
    Q, scale = inputs.embedding_e4m3(wl)
    Qd, sd = q_dev(Q), s_dev(scale)
    out = run_step(B, x, wl, Qd, sd, budgets, V=wl.V, two_pass=not single)
    check_stats(out, ost)
    acc = entropy_accept(ost["H"], ost["kappa"], wl.n_req, wl.L_c, budgets)
    for k in ("order", "mask", "n_accepted"):
        assert np.array_equal(out[k].cpu().numpy(), acc[k]), k
    ref = soft_embed_e4m3(x[:, :wl.V], ost["lse"], 0, wl.V, Q, scale, wl.gamma)
    assert rel_l2(out["E"].cpu().numpy(), ref).max() <= E_TOL


def test_single_pass_redo_rows(B):
    """Rows the single pass must redo (one-hot, a logit 90 nats above the rest) go through the
    8-bit redo kernel; rows that start masked or sit far below the reference stay in the
    product; a row without a distribution gives NaN as with the bf16 table."""
    wl = inputs.WORKLOADS["tiny"].with_(V=40000, d=640, L_c=16, n_req=1, seed=3, budget=5.0)
    x = inputs.logits(wl)
    x[0, 12345] = 1.0e4
    x[1, 30000] = 90.0
    x[2, :8192] = -np.inf
    x[3, :] = -np.inf
    x[4, :] -= 300.0
    Q, scale = inputs.embedding_e4m3(wl)
    out = run_step(B, x, wl, q_dev(Q), s_dev(scale), np.array([5.0], np.float32))
    ost = row_stats(x)
    check_stats(out, ost)
    E = out["E"].cpu().numpy()
    rows = np.array([0, 1, 2, 4, 5, 15])
    ref = soft_embed_e4m3(x, ost["lse"], 0, wl.V, Q, scale, wl.gamma, rows=rows)
    assert rel_l2(E[rows], ref).max() <= E_TOL
    assert np.all(np.isnan(E[3]))


@pytest.mark.slow
def test_step_canvas256_full_size(B):
    """The 256-position canvas over the full vocabulary (V = 262,144, d = 2816) with the 8-bit
    table: statistics and acceptance on every row, E on sampled rows."""
    wl = inputs.WORKLOADS["canvas256"]
    x, budgets, ost, _ = guarded(wl)
    Q, scale = inputs.embedding_e4m3(wl)
    out = run_step(B, x, wl, q_dev(Q), s_dev(scale), budgets)
    check_stats(out, ost)
    acc = entropy_accept(ost["H"], ost["kappa"], wl.n_req, wl.L_c, budgets)
    for k in ("order", "mask", "n_accepted"):
        assert np.array_equal(out[k].cpu().numpy(), acc[k]), k
    rows = np.arange(wl.R)   # every row
    ref = soft_embed_e4m3(x, ost["lse"], 0, wl.V, Q, scale, wl.gamma, rows=rows)
    assert rel_l2(out["E"].cpu().numpy()[rows], ref).max() <= E_TOL


@pytest.mark.parametrize("temperature", [0.0, 1.0, 0.7])
def test_loop_over_the_8bit_table_matches_the_oracle_chain(B, temperature):
    """Denoising-loop steps over the 8-bit table (argmax, and drawn candidates with the draw
    folded into the single pass): statistics, candidates, acceptance and the whole loop
    state bit-exact against the oracle chain (whose decisions keep their margins), E against
    the 8-bit oracle."""
    from oracle.loop_oracle import entropy_accept_eligible, loop_update, new_loop_state
    from tests.test_gpu_loop import (LOOP_WL, SAMPLED_WL, STABLE_STEPS, STEP_LIMIT, compare_state,
                                     decision_margins_ok, loop_threshold, sampled_chain_inputs)
    steps, seed = 6, 2024
    if temperature > 0:
        wl = SAMPLED_WL
        budgets, thr, chain = sampled_chain_inputs(wl, steps, temperature, seed)
    else:
        wl = LOOP_WL
        base = inputs.logits(wl)
        budgets = inputs.budgets(wl)
        thr = loop_threshold(row_stats(base), wl)
        o = new_loop_state(wl.n_req, wl.L_c)
        chain = []
        for t in range(steps):
            x = inputs.loop_logits(wl, t, base=base)
            st = row_stats(x)
            assert decision_margins_ok(st["H"], st["kappa"], o["eligible"], wl.n_req, wl.L_c, budgets), t
            acc = entropy_accept_eligible(st["H"], st["kappa"], o["eligible"], wl.n_req, wl.L_c, budgets,
                                          min_accept=1)
            o = loop_update(o, st["argmax"], st["H"], acc["mask"], wl.n_req, wl.L_c, STABLE_STEPS, thr, STEP_LIMIT)
            chain.append((x, st, {"candidate": st["argmax"]}, st["kappa"], acc, o))
    Q, scale = quantize_rows_e4m3(inputs.embedding_bf16(wl))
    Qd, sd = q_dev(Q), s_dev(scale)
    state = B.new_loop_state(wl.n_req, wl.L_c, "cuda")
    bud = dev(budgets)
    for t, (x, st, sm, kc, acc, o) in enumerate(chain):
        out = B.dg_sampler_loop_step_e4m3(dev(x), wl.n_req, wl.L_c, Qd, sd, wl.gamma, bud, state, STABLE_STEPS, thr,
                                          STEP_LIMIT, min_accept=1, temperature=temperature, seed=seed, offset=t)
        torch.cuda.synchronize()
        check_stats(out, dict(st, kappa=kc))
        if temperature > 0:
            assert np.array_equal(out["candidate"].cpu().numpy(), sm["candidate"]), t
        for key in ("order", "mask", "n_accepted"):
            assert np.array_equal(out[key].cpu().numpy(), acc[key]), (t, key)
        compare_state(state, o, f"step {t}")
    B.dg_get_device_status()
    rows = np.array([0, 17, 130, wl.R - 1])
    ref = soft_embed_e4m3(x, st["lse"], 0, wl.V, Q, scale, wl.gamma, rows=rows)
    assert rel_l2(out["E"].cpu().numpy()[rows], ref).max() <= E_TOL


def test_resident_step_and_loop_hold_an_8bit_table(B):
    """SamplerStep and SamplerLoop given an 8-bit table run the same calls as the C ABI's
    8-bit entry points: identical outputs (the product's reduce is deterministic) and, over
    three loop steps, identical state."""
    from denoising_sampler_step_gb300.step import SamplerLoop, SamplerStep
    wl = inputs.WORKLOADS["tiny"].with_(V=20000, d=512, L_c=64, n_req=2, seed=13, budget=6.0)
    x = dev(inputs.logits(wl))
    Q, scale = inputs.embedding_e4m3(wl)
    Qd, sd = q_dev(Q), s_dev(scale)
    bud = dev(inputs.budgets(wl))
    st = SamplerStep(Qd, wl.n_req, wl.L_c, wl.V, wl.gamma, scale=sd)
    a = {k: v.clone() for k, v in st(x, bud).items()}
    b = B.dg_sampler_step_e4m3(x, wl.n_req, wl.L_c, Qd, sd, wl.gamma, bud)
    torch.cuda.synchronize()
    for k in a:
        assert torch.equal(a[k], b[k]), k
    lp = SamplerLoop(Qd, wl.n_req, wl.L_c, wl.V, wl.gamma, 2, 1.0, 8, temperature=1.0, seed=5, scale=sd)
    state = B.new_loop_state(wl.n_req, wl.L_c, "cuda")
    for t in range(3):
        o1 = lp(x, bud)
        o2 = B.dg_sampler_loop_step_e4m3(x, wl.n_req, wl.L_c, Qd, sd, wl.gamma, bud, state, 2, 1.0, 8,
                                         temperature=1.0, seed=5, offset=t)
        torch.cuda.synchronize()
        assert torch.equal(o1["candidate"], o2["candidate"]) and torch.equal(o1["E"], o2["E"]), t
        for k in state:
            assert torch.equal(lp.state[k], state[k]), (t, k)
    B.dg_get_device_status()
