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


def test_no_alloc_rejects_shapes_beyond_its_scratch(B):
    from denoising_sampler_step_gb300.binding import DgError
    R, d = 8192, 2816
    x = torch.zeros((R, 64), dtype=torch.float32, device="cuda")
    lse = torch.zeros(R, dtype=torch.float32, device="cuda")
    W = torch.zeros((64, d), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((R, d), dtype=torch.float32, device="cuda")
    with pytest.raises(DgError) as ei:
        B.dg_soft_embed_no_alloc(x, lse, 0, 64, W, 1.0, out)
    assert ei.value.status == 2 and "fixed scratch" in str(ei.value)
