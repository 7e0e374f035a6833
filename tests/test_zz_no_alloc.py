"""dg_soft_embed_no_alloc against dg_soft_embed, through the C ABI.

Callers that cannot allocate device memory (a plugin handed only its buffers, a
server under a fixed memory budget) use dg_soft_embed_no_alloc, which keeps its
partial tiles in a fixed array inside the library instead of a caller workspace.
Its results must match dg_soft_embed within the soft-embedding tolerance, on two
calls in a row (the array keeps the first call's data, which the second must not
see).  This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import numpy as np
import pytest
import torch

from denoising_sampler_step_gb300 import inputs

pytestmark = pytest.mark.gpu

E_TOL = 1e-2   # per-row relative L2 error, as for every soft-embedding check


@pytest.fixture(scope="module")
def B():
    from denoising_sampler_step_gb300 import build
    build.build()
    from denoising_sampler_step_gb300 import binding
    return binding


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return np.linalg.norm(a - b, axis=1) / np.maximum(np.linalg.norm(b, axis=1), 1e-30)


def case(B, R, V, d, seed, s=0, e=None):
    e = V if e is None else e
    wl = inputs.Workload("no_alloc", 1, R, V, d, (0.5, 4.0), (0.0, 8.0), 2.0, seed=seed)
    x = torch.from_numpy(inputs.logits(wl)).cuda()
    Wb = inputs.padded_shard(inputs.embedding_bf16(wl), s, e, 128, pad_value="nan")
    W = torch.from_numpy(Wb.view(np.int16)).cuda().view(torch.bfloat16)
    st = B.dg_row_stats(x)
    return x, st["lse"], W, wl.gamma


def test_no_alloc_matches_workspace_call_twice(B):
    shapes = [(256, 65536, 2816, 0, None), (130, 4096, 256, 1000, 3333)]
    for k, (R, V, d, s, e) in enumerate(shapes):
        e = V if e is None else e
        x, lse, W, gamma = case(B, R, V, d, seed=70 + k, s=s, e=e)
        ref = B.dg_soft_embed(x, lse, s, e, W, gamma).cpu().numpy()
        out = torch.full((R, d), float("nan"), dtype=torch.float32, device="cuda")
        B.dg_soft_embed_no_alloc(x, lse, s, e, W, gamma, out)
        B.dg_get_device_status()
        got = out.cpu().numpy()
        assert np.all(np.isfinite(got)), k
        err = rel_l2(got, ref)
        assert err.max() <= E_TOL, (k, float(err.max()))


def test_no_alloc_small_case_matches_the_oracle(B):
    """A ragged slice on a small table against the CPU oracle itself, at the same bound."""
    from oracle import row_stats, soft_embed
    R, V, d, s, e = 130, 4096, 256, 1000, 3333
    wl = inputs.Workload("no_alloc", 1, R, V, d, (0.5, 4.0), (0.0, 8.0), 2.0, seed=77)
    x = inputs.logits(wl)
    Wb = inputs.embedding_bf16(wl)
    shard = inputs.padded_shard(Wb, s, e, 128, pad_value="nan")
    st = row_stats(x)
    xd = torch.from_numpy(x).cuda()
    lse = torch.from_numpy(st["lse"].astype(np.float32)).cuda()
    W = torch.from_numpy(shard.view(np.int16)).cuda().view(torch.bfloat16)
    out = torch.full((R, d), float("nan"), dtype=torch.float32, device="cuda")
    for _ in range(2):
        B.dg_soft_embed_no_alloc(xd, lse, s, e, W, wl.gamma, out)
        B.dg_get_device_status()
        ref = soft_embed(x, st["lse"], s, e, shard, wl.gamma)
        err = rel_l2(out.cpu().numpy(), ref)
        assert err.max() <= E_TOL, float(err.max())


def one_split_bytes(R, d):
    """Partial tiles of one vocabulary split: rows in whole 256-row tiles, columns in whole
    pairs of 512-column tiles, fp32 (the size rule the header states)."""
    return -(-R // 256) * 256 * (-(-d // 1024) * 1024) * 4


SCRATCH_BYTES = 16 << 20


def test_no_alloc_lowers_the_split_count_to_fit(B):
    """1024 rows at d = 2816: the workspace call plans several splits (their tiles need more
    than the fixed 16 MiB) while one split's tiles (12 MiB) fit, so the call must run with
    fewer splits than planned; the result still matches the workspace call, twice."""
    R, V, d = 1024, 262144, 2816
    assert one_split_bytes(R, d) <= SCRATCH_BYTES < 2 * one_split_bytes(R, d)
    assert B.dg_soft_embed_workspace_size(R, V, d) >= 2 * one_split_bytes(R, d)   # several splits planned
    x, lse, W, gamma = case(B, R, V, d, seed=91)
    ref = B.dg_soft_embed(x, lse, 0, V, W, gamma).cpu().numpy()
    out = torch.full((R, d), float("nan"), dtype=torch.float32, device="cuda")
    for _ in range(2):
        B.dg_soft_embed_no_alloc(x, lse, 0, V, W, gamma, out)
        B.dg_get_device_status()
        got = out.cpu().numpy()
        assert np.all(np.isfinite(got))
        assert rel_l2(got, ref).max() <= E_TOL


@pytest.mark.parametrize("R,d,fits", [(8192, 2816, False), (1400, 2816, False), (1100, 2816, True),
                                      (2048, 1200, True), (2304, 1200, False)])
def test_no_alloc_size_rule(B, R, d, fits):
    """d = 1,200 takes three 512-column tiles, padded to a pair of pairs (2,048 columns):
    2,048 rows fill the 16 MiB exactly, 2,304 do not fit."""
    from denoising_sampler_step_gb300.binding import DgError
    assert (one_split_bytes(R, d) <= SCRATCH_BYTES) == fits
    x = torch.zeros((R, 64), dtype=torch.float32, device="cuda")
    lse = torch.zeros(R, dtype=torch.float32, device="cuda")
    W = torch.zeros((64, d), dtype=torch.bfloat16, device="cuda")
    out = torch.full((R, d), float("nan"), dtype=torch.float32, device="cuda")
    if fits:
        # all logits 0 against lse = 0: every probability is 1, E = gamma * (sum of 64 zero rows)
        B.dg_soft_embed_no_alloc(x, lse, 0, 64, W, 1.0, out)
        B.dg_get_device_status()
        assert torch.count_nonzero(out).item() == 0
    else:
        with pytest.raises(DgError) as ei:
            B.dg_soft_embed_no_alloc(x, lse, 0, 64, W, 1.0, out)
        assert ei.value.status == 2 and "fixed scratch" in str(ei.value)
