"""The cost model against the numbers the pages print, and the input generator's contract."""
import json
import math
import os

import numpy as np

from denoising_sampler_step_gb300 import cost, inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_cost_model_matches_printed_numbers():
    with open(os.path.join(GOLDEN, "cost_model.json")) as f:
        g = json.load(f)
    V, d, L, T = g["V"], g["d"], g["L_c"], g["T"]
    assert cost.embedding_bytes(V, d) == g["embedding_bytes"]
    assert round(cost.embedding_bytes(V, d) / 2**30, 2) == g["embedding_gib_approx"]
    assert round(cost.soft_embed_flops(L, V, d) / 1e9) == g["full_product_gflop_per_rank_allgather"]
    assert round(cost.soft_embed_flops(L, V, d, tp=T) / 1e9, 1) == g["sharded_product_gflop_per_rank"]
    assert round(cost.reduced_tensor_bytes(L, d) / 2**20, 2) == g["reduced_tensor_mib_approx"]
    assert round(cost.ring_allreduce_bytes_per_rank(L, d, T) / 2**20, 2) == g["ring_mib_per_rank_approx"]
    assert cost.allgather_crossover_KN(V, L) == g["crossover_KN"]


def test_step_cost_and_roofline():
    c = cost.StepCost(rows=256, V=262144, d=2816, vocab=262144)
    assert c.logits_bytes == 268435456 and c.w_bytes == 1476395008
    assert abs(c.flops - 377.96e9) < 0.01e9
    t = c.roofline_seconds(6690.1, 1915.0)
    assert abs(t * 1e6 - 260.8) < 0.1          # HBM-bound at one canvas


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1 + 2**-8, 1 + 3 * 2**-8, -2.5, 53.066, 16.0], np.float32)
    b = inputs.f32_to_bf16_bits(x)
    assert list(b[:4]) == [0x3F80, 0x3F80, 0x3F82, 0xC020]
    back = inputs.bf16_bits_to_f32(b)
    assert back[4] == 53.0 and back[5] == 16.0
    assert inputs.WORKLOADS["canvas256"].gamma == 53.0 and inputs.WORKLOADS["tiny"].gamma == 16.0


def test_generator_is_seeded_and_redraws_one_request():
    wl = inputs.WORKLOADS["tiny"].with_(n_req=3, L_c=4, V=64)
    a, b = inputs.logits(wl), inputs.logits(wl)
    assert np.array_equal(a, b)
    c = inputs.logits(wl, attempts={1: 1})
    assert np.array_equal(a[:4], c[:4]) and np.array_equal(a[8:], c[8:])
    assert not np.array_equal(a[4:8], c[4:8])
    assert inputs.logits(wl, ld=72)[:, 64:].shape == (12, 8)


def test_generator_distributions():
    wl = inputs.WORKLOADS["tiny"]
    W = inputs.bf16_bits_to_f32(inputs.embedding_bf16(wl))
    assert W.shape == (4096, 256) and abs(W.std() - 0.02) < 1e-3
    x = inputs.logits(wl)
    assert x.shape == (16, 4096) and x.dtype == np.float32
    b = inputs.budgets(inputs.WORKLOADS["batch8"])
    assert b.shape == (8,) and np.all((b >= 2) & (b <= 16))
    pk = inputs.logits(inputs.WORKLOADS["late_batch32_peaked"].with_(n_req=1, L_c=4, V=1024))
    top2 = np.sort(pk, axis=1)[:, -2:]
    assert np.all(top2[:, 1] - top2[:, 0] >= 8.0 - 1e-4)


def test_slice_bounds_are_a_partition():
    for V, T in [(262144, 4), (4096, 3), (10, 4)]:
        b = inputs.slice_bounds(V, T)
        assert b[0][0] == 0 and b[-1][1] == V
        assert all(b[i][1] == b[i + 1][0] for i in range(T - 1))
    Wb = np.arange(40, dtype=np.uint16).reshape(10, 4)
    sh = inputs.padded_shard(Wb, 3, 8, 4, pad_value="nan")
    assert sh.shape == (8, 4) and np.array_equal(sh[:5], Wb[3:8]) and np.all(sh[5:] == 0x7FC0)
