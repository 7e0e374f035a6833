"""Parity of the vocabulary-sharded path on one device (through the C ABI): the shard
summaries, their combination, and the whole sharded step emulated with all shards on
one GPU, against the oracle and the unsharded calls."""
import numpy as np
import pytest
import torch

from denoising_sampler_step_gb300 import inputs
from denoising_sampler_step_gb300.vocab_parallel import ShardedStep, shard_bounds
from oracle import entropy_accept, row_stats, soft_embed
from oracle.partition_oracle import row_stats_partial
from tests.test_gpu_parity import E_TOL, check_stats, dev, rel_l2, w_dev
from tests.workloads import guarded

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from denoising_sampler_step_gb300 import build
    build.build()
    from denoising_sampler_step_gb300 import binding
    return binding


def shard_tensor(x, s, e):
    """Columns [s, e) in their own buffer, rows padded to a multiple of 4 with NaN (never read)."""
    n = e - s
    ld = (n + 3) // 4 * 4
    buf = np.full((x.shape[0], ld), np.nan, np.float32)
    buf[:, :n] = x[:, s:e]
    return dev(buf)[:, :n]


def test_one_shard_is_the_row_statistics_bit_for_bit(B):
    wl = inputs.WORKLOADS["tiny"].with_(V=40000, L_c=24, seed=12)
    xd = dev(inputs.logits(wl))
    st = B.dg_row_stats(xd)
    c = B.dg_row_stats_combine(B.dg_row_stats_partial(xd, 0)[None])
    for k in ("m", "lse", "H", "kappa", "argmax"):
        assert torch.equal(c[k].view(torch.int32), st[k].view(torch.int32)), k


@pytest.mark.parametrize("V,T", [(4096, 2), (40001, 4), (70003, 7)])
def test_shard_summaries_and_their_combination(B, V, T):
    wl = inputs.WORKLOADS["tiny"].with_(V=V, L_c=20, seed=V + T)
    x = inputs.logits(wl)
    x[2, :] = -np.inf
    x[2, V - 1] = 0.5                                  # mass only in the last shard
    x[3, :] = -np.inf                                  # no distribution
    x[4, [5, V - 3]] = x[4].max() + 3.0                # a maximum tied across shards
    bounds = shard_bounds(V, T)
    parts = [B.dg_row_stats_partial(shard_tensor(x, s, e), s) for s, e in bounds]
    for (s, e), p in zip(bounds, parts):
        o = row_stats_partial(x[:, s:e], s)
        g = p.cpu().numpy()
        assert np.array_equal(g[:, 1].view(np.int32), o["a"].astype(np.int32))
        assert np.array_equal(g[:, 0], o["m"].astype(np.float32))
        fin = np.isfinite(o["m"])
        for col, k in ((2, "rest"), (3, "t")):
            err = np.abs(g[fin, col] - o[k][fin]) / np.maximum(1.0, np.abs(o[k][fin]))
            assert err.max() <= 1e-5, k
    c = B.dg_row_stats_combine(torch.stack(parts))
    check_stats(c, row_stats(x))
    assert c["argmax"][4].item() == 5 and c["argmax"][2].item() == V - 1


@pytest.mark.parametrize("two_pass", [False, True])
def test_sharded_step_on_one_device(B, two_pass):
    """Four uneven shards in one process, each read once (the shard calls) or twice:
    statistics, acceptance and E against the oracle; E against the unsharded product (the
    partition identity)."""
    wl = inputs.WORKLOADS["tiny"].with_(n_req=3, L_c=32, V=40001, d=256, seed=77, budget=("uniform", 2.0, 20.0))
    x, budgets, ost, _ = guarded(wl, ld=40004)       # the unsharded calls need ldl % 4 == 0
    Wb = inputs.embedding_bf16(wl)
    Wd = w_dev(Wb)
    bounds = shard_bounds(wl.V, 4)
    step = ShardedStep(wl.n_req, wl.L_c, wl.gamma, two_pass=two_pass)
    out = step.local_step([shard_tensor(x, s, e) for s, e in bounds], [s for s, _ in bounds],
                          [Wd[s:e] for s, e in bounds], dev(budgets))
    torch.cuda.synchronize()
    B.dg_get_device_status()
    check_stats(out, ost)
    acc = entropy_accept(ost["H"], ost["kappa"], wl.n_req, wl.L_c, budgets)
    for k in ("order", "mask", "n_accepted"):
        assert np.array_equal(out[k].cpu().numpy(), acc[k]), k
    E = out["E"].cpu().numpy()
    assert rel_l2(E, soft_embed(x[:, :wl.V], ost["lse"], 0, wl.V, Wb, wl.gamma)).max() <= E_TOL
    xd = dev(x)
    full = B.dg_soft_embed(xd, B.dg_row_stats(xd, V=wl.V)["lse"], 0, wl.V, Wd, wl.gamma).cpu().numpy()
    # two passes: the same bf16 probabilities as the unsharded product, only the fp32 additions
    # reassociated; one read: probabilities exp(l - c) rounded before their scale, so the two
    # agree to the bf16 rounding (the tolerance), as the single-pass step and the two-pass one do
    assert rel_l2(E, full.astype(np.float64)).max() <= (1e-3 if two_pass else E_TOL)


@pytest.mark.slow
def test_sharded_statistics_full_size(B):
    """The vocab_tp4 workload (V = 262,144, four shards): every row against the oracle."""
    wl = inputs.WORKLOADS["vocab_tp4"]
    x = inputs.logits(wl)
    bounds = shard_bounds(wl.V, 4)
    c = B.dg_row_stats_combine(torch.stack([B.dg_row_stats_partial(shard_tensor(x, s, e), s) for s, e in bounds]))
    check_stats(c, row_stats(x))


def test_sharded_step_over_an_8bit_table(B):
    """Four uneven shards of an 8-bit table (codes and row scales per shard) in one process:
    statistics and acceptance against the oracle, E against the 8-bit oracle over the whole
    table (the partition identity)."""
    from oracle.quant_oracle import soft_embed_e4m3
    wl = inputs.WORKLOADS["tiny"].with_(n_req=2, L_c=32, V=40001, d=512, seed=78, budget=("uniform", 2.0, 20.0))
    x, budgets, ost, _ = guarded(wl, ld=40004)
    Q, scale = inputs.embedding_e4m3(wl)
    bounds = shard_bounds(wl.V, 4)

    def q_shard(s, e):
        ldq = (wl.d + 15) // 16 * 16
        buf = np.zeros((e - s, ldq), np.uint8)
        buf[:, :wl.d] = Q[s:e]
        return dev(buf)[:, :wl.d], dev(scale[s:e])

    step = ShardedStep(wl.n_req, wl.L_c, wl.gamma)
    out = step.local_step([shard_tensor(x, s, e) for s, e in bounds], [s for s, _ in bounds],
                          [q_shard(s, e) for s, e in bounds], dev(budgets))
    torch.cuda.synchronize()
    B.dg_get_device_status()
    check_stats(out, ost)
    acc = entropy_accept(ost["H"], ost["kappa"], wl.n_req, wl.L_c, budgets)
    for k in ("order", "mask", "n_accepted"):
        assert np.array_equal(out[k].cpu().numpy(), acc[k]), k
    ref = soft_embed_e4m3(x[:, :wl.V], ost["lse"], 0, wl.V, Q, scale, wl.gamma)
    assert rel_l2(out["E"].cpu().numpy(), ref).max() <= E_TOL


def test_rank_step_over_a_one_rank_nccl_group(B):
    """rank_step with its gathers over a real NCCL process group of one rank (the whole
    vocabulary is the rank's shard): statistics, acceptance and E against the oracle.  The
    same code runs one rank per GPU when there are several."""
    import socket
    import torch.distributed as dist
    from denoising_sampler_step_gb300.vocab_parallel import TorchComm
    if dist.is_initialized():
        pytest.skip("a process group is already set up in this process")
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1)
    try:
        wl = inputs.WORKLOADS["tiny"].with_(n_req=2, L_c=32, V=40000, d=512, seed=79, budget=("uniform", 2.0, 20.0))
        x, budgets, ost, _ = guarded(wl)
        Wb = inputs.embedding_bf16(wl)
        out = ShardedStep(wl.n_req, wl.L_c, wl.gamma).rank_step(dev(x), 0, w_dev(Wb), dev(budgets), TorchComm())
        torch.cuda.synchronize()
        B.dg_get_device_status()
        check_stats(out, ost)
        acc = entropy_accept(ost["H"], ost["kappa"], wl.n_req, wl.L_c, budgets)
        for k in ("order", "mask", "n_accepted"):
            assert np.array_equal(out[k].cpu().numpy(), acc[k]), k
        ref = soft_embed(x, ost["lse"], 0, wl.V, Wb, wl.gamma)
        assert rel_l2(out["E"].cpu().numpy(), ref).max() <= E_TOL
    finally:
        dist.destroy_process_group()


def test_shard_calls_summaries_and_redo_rows(B):
    """The one-read shard calls on three uneven shards: each shard's summaries against the
    oracle's (m and the argmax exact, rest and t to 1e-5), the combined statistics against the
    whole-row oracle, and E against the oracle, with rows whose probabilities against a split's
    reference could overflow (the second call recomputes them), rows whose mass lies in one
    shard only and a row without a distribution."""
    wl = inputs.WORKLOADS["tiny"].with_(n_req=1, L_c=24, V=40000, d=256, seed=81, budget=5.0)
    x = inputs.logits(wl)
    x[0, 12345] = 1.0e4                     # one-hot: overflow against any reference
    x[1, 30000] = 90.0                      # 90 nats above the rest, in the last shard
    x[2, :20000] = -np.inf                  # no mass in the first shard
    x[3, :] = -np.inf                       # no distribution
    x[4, :] -= 300.0                        # far below the default reference
    Wb = inputs.embedding_bf16(wl)
    bounds = shard_bounds(wl.V, 3)
    states, parts = [], []
    shards = [shard_tensor(x, s, e) for s, e in bounds]
    wss = [B.workspace(wl.R, e - s, wl.d, shards[0].device) for s, e in bounds]
    for (s, e), sh, ws in zip(bounds, shards, wss):
        st = B.dg_soft_embed_shard_begin(sh, s, w_dev(Wb[s:e]), ws)
        o = row_stats_partial(x[:, s:e], s)
        g = st.cpu().numpy()
        assert np.array_equal(g[:, 1].view(np.int32), o["a"].astype(np.int32))
        assert np.array_equal(g[:, 0], o["m"].astype(np.float32))
        fin = np.isfinite(o["m"])
        for col, k in ((2, "rest"), (3, "t")):
            err = np.abs(g[fin, col] - o[k][fin]) / np.maximum(1.0, np.abs(o[k][fin]))
            assert err.max() <= 1e-5, k
        states.append(st)
    c = B.dg_row_stats_combine(torch.stack(states))
    ost = row_stats(x)
    check_stats(c, ost)
    for (s, e), sh, ws in zip(bounds, shards, wss):
        parts.append(B.dg_soft_embed_shard_end(sh, c["lse"], w_dev(Wb[s:e]), 1.0, ws))
    E = B.dg_sum_partials(parts, wl.gamma).cpu().numpy()
    torch.cuda.synchronize()
    B.dg_get_device_status()
    rows = np.array([0, 1, 2, 4, 5, 23])
    assert rel_l2(E[rows], soft_embed(x, ost["lse"], 0, wl.V, Wb, wl.gamma, rows=rows)).max() <= E_TOL
    assert np.all(np.isnan(E[3]))


def test_shard_calls_reject_an_empty_shard(B):
    from denoising_sampler_step_gb300.binding import DgError
    x = dev(np.zeros((4, 8), np.float32))
    W = w_dev(np.zeros((8, 64), np.uint16))
    ws = B.workspace(4, 8, 64, x.device)
    with pytest.raises(DgError) as ei:
        B.dg_soft_embed_shard_begin(x[:, :0], 0, W, ws)
    assert ei.value.status == 1
