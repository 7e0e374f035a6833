"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Bars: argmax, order, mask and n_accepted bit-exact; entropy within 1e-4 nats;
soft embeddings within a per-row relative L2 error of 1e-2 (the sampler-step
benchmark's tolerances).  lse within 1e-4 and kappa within 1e-5 * max(1, kappa)
(the library's fp32 statistics against fp64), and within 5e-6 relative where
kappa < 1 (rows near one-hot, whose order rests on it).
"""
import math

import numpy as np
import pytest
import torch

from denoising_sampler_step_gb300 import inputs
from oracle import entropy_accept, row_stats, soft_embed, sum_partials
from tests.workloads import guarded

pytestmark = pytest.mark.gpu

H_TOL = 1e-4
E_TOL = 1e-2


@pytest.fixture(scope="module")
def B():
    from denoising_sampler_step_gb300 import build
    build.build()
    from denoising_sampler_step_gb300 import binding
    return binding


def dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def w_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def check_stats(g, o, rows=None):
    idx = np.arange(len(o["H"])) if rows is None else rows
    am = g["argmax"].cpu().numpy()[idx]
    assert np.array_equal(am, o["argmax"][idx]), "argmax"
    m = g["m"].cpu().numpy()[idx].astype(np.float64)
    fin = np.isfinite(o["lse"][idx])
    assert np.array_equal(m[fin], o["m"][idx][fin])
    for k, tol in (("H", H_TOL), ("lse", 1e-4)):
        v = g[k].cpu().numpy()[idx].astype(np.float64)
        assert np.array_equal(np.isnan(v), np.isnan(o[k][idx])), k
        err = np.abs(v[fin] - o[k][idx][fin])
        assert err.size == 0 or err.max() <= tol, (k, float(err.max()))
    kp = g["kappa"].cpu().numpy()[idx].astype(np.float64)
    ref = o["kappa"][idx]
    err = np.abs(kp[fin] - ref[fin]) / np.maximum(1.0, ref[fin])
    assert err.size == 0 or err.max() <= 1e-5, float(err.max())
    rel = np.abs(kp[fin] - ref[fin]) / np.maximum(ref[fin], 1e-30)
    # near one-hot (kappa < 1) the order rests on kappa's relative precision; below 1e-30 the
    # terms of rest fall under fp32's normal range (flushed to zero), so only an absolute
    # bound holds there
    small = (ref[fin] < 1.0) & (ref[fin] >= 1e-30)
    assert not np.any(small) or rel[small].max() <= 5e-6, ("kappa near one-hot", float(rel[small].max()))
    tiny = ref[fin] < 1e-30
    assert not np.any(tiny) or np.abs(kp[fin] - ref[fin])[tiny].max() <= 1e-33


def rel_l2(E, ref):
    E = np.asarray(E, np.float64)
    num = np.linalg.norm(E - ref, axis=1)
    den = np.maximum(np.linalg.norm(ref, axis=1), 1e-30)
    return num / den


# --------------------------------------------------------------------------- row statistics

@pytest.mark.parametrize("V,ld", [(4096, 4096), (4093, 4096), (1000, 1000), (40000, 40004), (70001, 70004),
                                  (262144, 262144)])
def test_row_stats_shapes(B, V, ld):
    wl = inputs.WORKLOADS["tiny"].with_(V=V, L_c=9, seed=V)
    x = inputs.logits(wl, ld=ld)
    g = B.dg_row_stats(dev(x), V=V)
    check_stats(g, row_stats(x[:, :V]))


def test_row_stats_special_rows(B):
    V = 50000
    rng = np.random.default_rng(0)
    x = (rng.standard_normal((8, V)) * 2).astype(np.float32)
    x[0] = 1.25                                 # uniform: H = ln V, argmax 0
    x[1, :] = -np.inf
    x[1, [7, 77, 40000]] = 3.0                  # 3-way tie, rest masked: H = ln 3, argmax 7
    x[2, 12345] = 1e4                           # one-hot
    x[3, 100:200] = -np.inf                     # masked vocabulary
    x[4, [10, 49999]] = 50.0                    # tie at the top across pieces: lowest index
    x[5] = -np.inf                              # empty row: NaN statistics
    x[6, 31] = x[6].max() + 30.0                # nearly one-hot (kappa ~ V e^-30)
    x[7, 49999] = 60.0                          # max in the last entry
    g = B.dg_row_stats(dev(x))
    o = row_stats(x)
    check_stats(g, o)
    assert abs(g["H"][0].item() - math.log(V)) < H_TOL and g["argmax"][1].item() == 7
    assert abs(g["H"][1].item() - math.log(3)) < H_TOL
    assert g["argmax"][4].item() == 10 and g["argmax"][5].item() == 0 and math.isnan(g["H"][5].item())


def test_row_stats_deterministic(B):
    x = dev(inputs.logits(inputs.WORKLOADS["tiny"].with_(V=262144, L_c=16, seed=5)))
    a = B.dg_row_stats(x)
    b = B.dg_row_stats(x)
    for k in a:
        assert torch.equal(a[k], b[k]), k


# --------------------------------------------------------------------------- acceptance

@pytest.mark.parametrize("L_c,n_req", [(1, 3), (5, 2), (16, 1), (33, 4), (256, 3), (1000, 1), (1024, 2)])
def test_accept_matches_oracle_on_same_inputs(B, L_c, n_req):
    rng = np.random.default_rng(L_c)
    R = L_c * n_req
    H = rng.uniform(0, 3, R).astype(np.float32)
    kappa = rng.uniform(0, 6, R).astype(np.float32)
    kappa[::7] = kappa[0]                      # exact ties: lower position first
    budgets = rng.uniform(0, 1.5 * L_c, n_req).astype(np.float32)
    for min_acc in (0, 3):
        g = B.dg_entropy_accept(dev(H), dev(kappa), n_req, L_c, dev(budgets), min_accept=min_acc)
        o = entropy_accept(H, kappa, n_req, L_c, budgets, min_accept=min_acc)
        assert np.array_equal(g["order"].cpu().numpy(), o["order"])
        assert np.array_equal(g["mask"].cpu().numpy(), o["mask"])
        assert np.array_equal(g["n_accepted"].cpu().numpy(), o["n_accepted"])


def test_accept_budget_sweep_and_nan(B):
    L = 64
    rng = np.random.default_rng(3)
    H = rng.uniform(0.1, 1, L).astype(np.float32)
    kappa = rng.uniform(0, 5, L).astype(np.float32)
    srt = np.lexsort((np.arange(L), kappa.astype(np.float64)))
    C = np.cumsum(H[srt].astype(np.float64))
    budgets = np.array([C[0] / 2] + [(C[k] + C[k + 1]) / 2 for k in range(L - 1)] + [C[-1] + 1], np.float32)
    nq = len(budgets)
    g = B.dg_entropy_accept(dev(np.tile(H, nq)), dev(np.tile(kappa, nq)), nq, L, dev(budgets))
    assert list(g["n_accepted"].cpu().numpy()) == list(range(L + 1))
    # a position without a distribution (all -inf logits) sorts last and stops the running sum
    Hn, kn = H.copy(), kappa.copy()
    Hn[5] = np.nan
    kn[5] = np.nan
    bud = np.array([1e9], np.float32)
    g = B.dg_entropy_accept(dev(Hn), dev(kn), 1, L, dev(bud))
    o = entropy_accept(Hn, kn, 1, L, bud)
    assert g["order"][L - 1].item() == 5 and g["n_accepted"][0].item() == L - 1
    assert np.array_equal(g["order"].cpu().numpy(), o["order"])
    assert np.array_equal(g["mask"].cpu().numpy(), o["mask"])


# --------------------------------------------------------------------------- soft embedding

def embed_case(B, R, V, d, seed, ldl=None):
    wl = inputs.Workload("case", 1, R, V, d, (0.5, 4.0), (0.0, 8.0), 2.0, seed=seed)
    x = inputs.logits(wl, ld=ldl)
    Wb = inputs.embedding_bf16(wl)
    xd = dev(x)
    st = B.dg_row_stats(xd, V=V)
    Wd = w_dev(Wb)
    gamma = wl.gamma
    E = B.dg_soft_embed(xd, st["lse"], 0, V, Wd, gamma)
    ost = row_stats(x[:, :V])
    ref = soft_embed(x[:, :V], ost["lse"], 0, V, Wb, gamma)
    return E.cpu().numpy(), ref, (x, Wb, st, xd, Wd, gamma)


@pytest.mark.parametrize("R,V,d", [(16, 4096, 256), (130, 4096, 256), (16, 4096, 200), (5, 1000, 40),
                                   (256, 8192, 512), (300, 2048, 768)])
def test_soft_embed_shapes(B, R, V, d):
    E, ref, _ = embed_case(B, R, V, d, seed=R + V + d)
    assert np.all(np.isfinite(E))
    assert rel_l2(E, ref).max() <= E_TOL


@pytest.mark.parametrize("d,ldw", [(960, 960), (1000, 1000), (1000, 1024), (600, 608), (2816, 2880)])
def test_soft_embed_w_load_paths_with_nan_pitch_padding(B, d, ldw):
    """Every way the product loads W: one 4-D load of a CTA's four atoms per block, a 3-D
    load per half where the fourth atom would pass the row pitch (d = 960: the second tile),
    64-column 2-D boxes where the pitch does not hold whole atoms (d = 1000, 600), and 4-D
    loads that read the pitch's padding columns (ldw > d), which hold NaN here and must not
    reach E.  The plain product and the single-pass step, 256 rows (one row block)."""
    R, V = 256, 8192
    wl = inputs.Workload("case", 1, R, V, d, (0.5, 4.0), (0.0, 8.0), 2.0, seed=d + ldw)
    x = inputs.logits(wl)
    Wb = inputs.embedding_bf16(wl)
    pitch = np.full((V, ldw), 0x7FC0, np.uint16)
    pitch[:, :d] = Wb
    Wd = w_dev(pitch)[:, :d]
    assert Wd.stride(0) == ldw
    xd = dev(x)
    st = B.dg_row_stats(xd, V=V)
    E = B.dg_soft_embed(xd, st["lse"], 0, V, Wd, wl.gamma).cpu().numpy()
    ref = soft_embed(x, row_stats(x)["lse"], 0, V, Wb, wl.gamma)
    assert np.all(np.isfinite(E))
    assert rel_l2(E, ref).max() <= E_TOL
    g = B.dg_sampler_step(xd, 1, R, Wd, wl.gamma, dev(np.full(1, 1e9, np.float32)))
    Es = g["E"].cpu().numpy()
    assert np.all(np.isfinite(Es))
    assert rel_l2(Es, ref).max() <= E_TOL


def test_soft_embed_ragged_slices_with_nan_padding(B):
    R, V, d = 40, 4096, 256
    full, ref_full, (x, Wb, st, xd, _, gamma) = embed_case(B, R, V, d, seed=11, ldl=4100)
    bounds = [(0, 1000), (1000, 2100), (2100, 3333), (3333, 4096)]
    parts, oparts = [], []
    ost = row_stats(x[:, :V])
    for s, e in bounds:
        shard = inputs.padded_shard(Wb, s, e, 128, pad_value="nan")
        parts.append(B.dg_soft_embed(xd, st["lse"], s, e, w_dev(shard), 1.0))
        oparts.append(soft_embed(x[:, :V], ost["lse"], s, e, shard, 1.0))
    summed = B.dg_sum_partials(parts, gamma).cpu().numpy()
    assert np.all(np.isfinite(summed))
    ref = sum_partials(oparts, gamma)
    assert rel_l2(summed, ref).max() <= E_TOL
    assert rel_l2(summed, ref_full).max() <= E_TOL
    for g, o in zip(parts, oparts):
        assert rel_l2(g.cpu().numpy(), o).max() <= E_TOL


def test_soft_embed_one_slice_is_the_unsliced_call(B):
    """At one partition the sliced call over [0, V) is the unsliced product, bit for bit."""
    R, V, d = 64, 4096, 256
    E, _, (x, Wb, st, xd, Wd, gamma) = embed_case(B, R, V, d, seed=12)
    again = B.dg_soft_embed(xd, st["lse"], 0, V, Wd, gamma).cpu().numpy()
    assert np.array_equal(E, again)       # deterministic split-K order
    part = B.dg_soft_embed(xd, st["lse"], 0, V, Wd, 1.0)
    one = B.dg_sum_partials([part], gamma).cpu().numpy()
    assert np.array_equal(one, E)


def test_soft_embed_one_hot_and_uniform(B):
    V = 4096
    wl = inputs.WORKLOADS["tiny"]
    Wb = inputs.embedding_bf16(wl)
    W = inputs.bf16_bits_to_f32(Wb).astype(np.float64)
    x = np.zeros((3, V), np.float32)
    x[0, 77] = 1e4
    x[1, 4095] = 1e4
    x[2] = 0.5
    xd = dev(x)
    st = B.dg_row_stats(xd)
    E = B.dg_soft_embed(xd, st["lse"], 0, V, w_dev(Wb), 16.0).cpu().numpy()
    assert np.array_equal(E[0], (16.0 * W[77]).astype(np.float32))
    assert np.array_equal(E[1], (16.0 * W[4095]).astype(np.float32))
    assert rel_l2(E[2:], 16.0 * W.mean(0, keepdims=True)).max() <= 1e-3


def test_empty_slice_writes_zeros(B):
    x = dev(np.zeros((4, 64), np.float32))
    st = B.dg_row_stats(x)
    W = w_dev(np.zeros((128, 64), np.uint16))
    E = B.dg_soft_embed(x, st["lse"], 10, 10, W, 1.0)
    assert torch.count_nonzero(E).item() == 0


# --------------------------------------------------------------------------- fused step

def step_and_compare(B, wl, sample_rows=None):
    x, budgets, ost, _ = guarded(wl)
    Wb = inputs.embedding_bf16(wl)
    xd, Wd = dev(x), w_dev(Wb)
    out = B.dg_sampler_step(xd, wl.n_req, wl.L_c, Wd, wl.gamma, dev(budgets))
    torch.cuda.synchronize()
    B.dg_get_device_status()
    check_stats(out, ost)
    oacc = entropy_accept(ost["H"], ost["kappa"], wl.n_req, wl.L_c, budgets)
    for k in ("order", "mask", "n_accepted"):
        assert np.array_equal(out[k].cpu().numpy(), oacc[k]), k
    rows = np.arange(wl.R) if sample_rows is None else sample_rows
    ref = soft_embed(x, ost["lse"], 0, wl.V, Wb, wl.gamma, rows=rows)
    err = rel_l2(out["E"].cpu().numpy()[rows], ref)
    assert err.max() <= E_TOL, float(err.max())
    assert torch.isfinite(out["E"]).all()
    return out


def test_step_tiny(B):
    step_and_compare(B, inputs.WORKLOADS["tiny"])


def test_step_tiny_many_requests(B):
    wl = inputs.WORKLOADS["tiny"].with_(n_req=6, budget=("uniform", 0.5, 6.0))
    step_and_compare(B, wl)


def sampled_rows(R, n, seed):
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([[0, R - 1], rng.choice(R, n, replace=False)]))


@pytest.mark.slow
def test_step_canvas256_full_size(B):
    """The headline workload at full size: every one of the 256 rows' E against the oracle."""
    wl = inputs.WORKLOADS["canvas256"]
    step_and_compare(B, wl)


@pytest.mark.slow
def test_vocab_tp4_partition_full_size(B):
    wl = inputs.WORKLOADS["vocab_tp4"]
    x, budgets, ost, _ = guarded(wl)
    Wb = inputs.embedding_bf16(wl)
    xd = dev(x)
    st = B.dg_row_stats(xd)
    check_stats(st, ost)
    full = B.dg_soft_embed(xd, st["lse"], 0, wl.V, w_dev(Wb), wl.gamma)
    parts = []
    for s, e in inputs.slice_bounds(wl.V, wl.slices):
        shard = inputs.padded_shard(Wb, s, e, 128, pad_value="zero")
        parts.append(B.dg_soft_embed(xd, st["lse"], s, e, w_dev(shard), 1.0))
    summed = B.dg_sum_partials(parts, wl.gamma).cpu().numpy()
    rows = np.arange(wl.R)   # every row
    ref = soft_embed(x, ost["lse"], 0, wl.V, Wb, wl.gamma, rows=rows)
    assert rel_l2(summed[rows], ref).max() <= E_TOL
    # the partition identity on every row: the sum of slices is the unsliced product up to
    # the order of the fp32 additions (the probabilities are the same bf16 values)
    dev_rows = rel_l2(summed, full.cpu().numpy().astype(np.float64))
    assert dev_rows.max() <= 1e-3, float(dev_rows.max())


@pytest.mark.slow
def test_step_batch8_full_size(B):
    wl = inputs.WORKLOADS["batch8"]
    step_and_compare(B, wl, sample_rows=sampled_rows(wl.R, 30, 2))


@pytest.mark.slow
@pytest.mark.parametrize("name", ["late_batch32", "late_batch32_peaked"])
def test_step_late_batch32_full_size(B, name):
    """8192 rows: statistics and acceptance on every row, the embedding on sampled rows."""
    wl = inputs.WORKLOADS[name]
    step_and_compare(B, wl, sample_rows=sampled_rows(wl.R, 30, 4))


def test_step_captured_in_a_cuda_graph_matches_the_eager_step(B):
    """Every call is capturable (no allocation, synchronisation or host copy inside); the
    replayed graph, programmatic-launch edges included, gives bit-identical results."""
    from denoising_sampler_step_gb300.step import SamplerStep
    wl = inputs.WORKLOADS["tiny"].with_(V=40000, L_c=64, n_req=2, d=256, seed=21)
    x = dev(inputs.logits(wl))
    Wd = w_dev(inputs.embedding_bf16(wl))
    bud = dev(inputs.budgets(wl))
    st = SamplerStep(Wd, wl.n_req, wl.L_c, wl.V, wl.gamma, device="cuda")
    eager = {k: v.clone() for k, v in st(x, bud).items()}
    torch.cuda.synchronize()
    for v in st.out.values():
        v.zero_()
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        st(x, bud)
    torch.cuda.current_stream().wait_stream(cap)
    torch.cuda.synchronize()
    for v in st.out.values():
        v.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cap):
        st(x, bud)
    g.replay()
    torch.cuda.synchronize()
    B.dg_get_device_status()
    for k, v in eager.items():
        assert torch.equal(st.out[k], v), k


# --------------------------------------------------------------------------- failure detection

def test_wait_timeout_is_reported_and_the_context_stays_usable(B):
    """A device wait that can never complete gives up after its bound; the host reads
    DG_ERR_TIMEOUT once, the word is cleared, and the next kernel runs correctly."""
    B.dg_get_device_status()  # nothing pending
    B.dg_check_wait_timeout(20000)  # 20 ms
    with pytest.raises(B.DgError) as err:
        B.dg_get_device_status()
    assert err.value.status == 4
    B.dg_get_device_status()  # cleared
    wl = inputs.WORKLOADS["tiny"].with_(V=4096, L_c=9, seed=11)
    x = inputs.logits(wl)
    check_stats(B.dg_row_stats(dev(x)), row_stats(x))
    B.dg_get_device_status()


# --------------------------------------------------------------------------- stochastic candidates

def check_sample(g, o, tol=1e-3):
    """The candidate is unique where both of the oracle's decisions (the group, then the
    entry inside it) lead their runner-up by more than `tol`; elsewhere the GPU's group must
    score within `tol` of the best group and its entry within `tol` of the best entry of
    that group."""
    cand = g["candidate"].cpu().numpy()
    lp = g["log_p"].cpu().numpy().astype(np.float64)
    rows = np.arange(len(cand))
    fin = np.isfinite(o["log_p"])
    clear = (o["group_margin"] > tol) & (o["margin"] > tol)
    assert np.array_equal(cand[clear], o["candidate"][clear])
    gs = o["group_score"]
    grp = cand // 16
    top_g = gs[rows, o["group"]]
    assert np.all(gs[rows[fin], grp[fin]] >= top_g[fin] - tol)
    es = o["entry_score"]
    for i in rows[fin & ~clear]:
        lo, hi = 16 * grp[i], min(16 * grp[i] + 16, es.shape[1])
        assert es[i, cand[i]] >= es[i, lo:hi].max() - tol, i
    assert np.array_equal(np.isnan(lp), ~fin)
    assert np.all(np.abs(lp[fin] - o["log_p"][fin]) <= 1e-4 * np.maximum(1.0, np.abs(o["log_p"][fin])))


@pytest.mark.parametrize("V,ld,temperature", [(4096, 4096, 1.0), (4093, 4096, 0.5), (1000, 1000, 2.0),
                                              (70001, 70004, 1.0), (262144, 262144, 0.7)])
def test_row_sample_matches_oracle(B, V, ld, temperature):
    from oracle import row_sample
    wl = inputs.WORKLOADS["tiny"].with_(V=V, L_c=12, seed=V + 3)
    x = inputs.logits(wl, ld=ld)
    g = B.dg_row_sample(dev(x), temperature, seed=1234, offset=7, V=V)
    check_sample(g, row_sample(x[:, :V], temperature, 1234, 7))


def test_row_sample_special_rows_and_determinism(B):
    from oracle import row_sample
    V = 50000
    rng = np.random.default_rng(8)
    x = (rng.standard_normal((6, V)) * 2).astype(np.float32)
    x[1, :] = -np.inf
    x[1, [7, 77, 40000]] = 3.0       # three allowed entries
    x[2, 12345] = 1e4                # one-hot: always drawn
    x[3, ::2] = -np.inf              # half masked
    x[4] = -np.inf                   # empty: candidate 0, NaN log_p
    xd = dev(x)
    g = B.dg_row_sample(xd, 1.0, seed=99, offset=3)
    check_sample(g, row_sample(x, 1.0, 99, 3))
    c = g["candidate"].cpu().numpy()
    assert c[1] in (7, 77, 40000) and c[2] == 12345 and c[3] % 2 == 1 and c[4] == 0
    h = B.dg_row_sample(xd, 1.0, seed=99, offset=3)
    for k in g:  # bit patterns (NaN compares unequal to itself)
        assert torch.equal(g[k].view(torch.int32), h[k].view(torch.int32)), k
    o = B.dg_row_sample(dev(np.tile(x[0], (64, 1))), 1.0, seed=99, offset=4)
    assert len(set(o["candidate"].cpu().numpy().tolist())) > 1  # other counters, other draws


@pytest.mark.parametrize("V,ld,temperature", [(4096, 4096, 1.0), (4093, 4096, 0.5), (70001, 70004, 1.0),
                                              (262144, 262144, 0.7)])
def test_row_stats_sample_is_the_two_passes_in_one(B, V, ld, temperature):
    """The fused pass: statistics as dg_row_stats (the same max and argmax; sums folded in
    another order), the draw and its log-probability bit-identical to dg_row_sample, both
    against the oracle; kappa is -ln p of the drawn token (ln Z where it is the argmax)."""
    from oracle import candidate_kappa, row_sample
    wl = inputs.WORKLOADS["tiny"].with_(V=V, L_c=12, seed=V + 5)
    x = inputs.logits(wl, ld=ld)
    xd = dev(x)
    f = B.dg_row_stats_sample(xd, temperature, seed=77, offset=2, V=V)
    s = B.dg_row_stats(xd, V=V)
    r = B.dg_row_sample(xd, temperature, seed=77, offset=2, V=V)
    for k in ("m", "argmax"):
        assert torch.equal(f[k].view(torch.int32), s[k].view(torch.int32)), k
    for k in ("lse", "H"):
        assert torch.allclose(f[k], s[k], rtol=2e-6, atol=2e-6), k
    for k in ("candidate", "log_p"):
        assert torch.equal(f[k].view(torch.int32), r[k].view(torch.int32)), k
    ost = row_stats(x[:, :V])
    check_stats({k: s[k] for k in s}, ost)
    check_stats({k: (f[k] if k != "kappa" else s[k]) for k in s}, ost)
    check_sample(f, row_sample(x[:, :V], temperature, 77, 2))
    cand = f["candidate"].cpu().numpy()
    kc = f["kappa"].cpu().numpy().astype(np.float64)
    ref = candidate_kappa(x[:, :V], cand)
    assert np.all(np.abs(kc - ref) <= 1e-5 * np.maximum(1.0, ref))
    at_argmax = cand == f["argmax"].cpu().numpy()
    assert np.allclose(f["kappa"].cpu().numpy()[at_argmax], s["kappa"].cpu().numpy()[at_argmax], rtol=2e-6, atol=1e-7)


def test_row_stats_sample_special_rows(B):
    from oracle import candidate_kappa, row_sample
    V = 50000
    rng = np.random.default_rng(9)
    x = (rng.standard_normal((5, V)) * 2).astype(np.float32)
    x[1, :] = -np.inf
    x[1, [7, 77, 40000]] = 3.0
    x[2, 12345] = 1e4
    x[4] = -np.inf
    xd = dev(x)
    f = B.dg_row_stats_sample(xd, 1.0, seed=5, offset=0)
    check_sample(f, row_sample(x, 1.0, 5, 0))
    s = B.dg_row_stats(xd)
    for k in ("m", "argmax"):
        assert torch.equal(f[k].view(torch.int32), s[k].view(torch.int32)), k
    for k in ("lse", "H"):
        assert torch.allclose(f[k], s[k], rtol=2e-6, atol=2e-6, equal_nan=True), k
    kc = f["kappa"].cpu().numpy().astype(np.float64)
    ref = candidate_kappa(x, f["candidate"].cpu().numpy())
    assert np.array_equal(np.isnan(kc), np.isnan(ref))
    fin = np.isfinite(ref)
    assert np.all(np.abs(kc[fin] - ref[fin]) <= 1e-5 * np.maximum(1.0, ref[fin]))
    assert f["candidate"][2].item() == 12345 and f["kappa"][2].item() == 0.0
