"""Pins of the 8-bit-table oracle (oracle/quant_oracle.py) to facts fixed elsewhere: the
E4M3 format's definition (hand-derived values and ties), PyTorch's float8_e4m3fn
conversions, brute force on small tables, and the bf16 oracle on tables that both formats
hold exactly."""
import json
import math
import os

import numpy as np
import pytest
import torch

from denoising_sampler_step_gb300 import inputs
from oracle import row_stats, soft_embed
from oracle.quant_oracle import (E4M3_VALUES, dequantize_rows_e4m3, e4m3_decode, e4m3_round,
                                 quantize_rows_e4m3, soft_embed_e4m3)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def fixture():
    with open(os.path.join(GOLDEN, "e4m3_format.json")) as f:
        return json.load(f)


def test_decode_matches_the_format_definition():
    g = fixture()
    for code, value, _ in g["values"]:
        got = e4m3_decode(np.array([int(code, 16)], np.uint8))[0]
        assert got == value and math.copysign(1.0, got) == math.copysign(1.0, value), code
    for code in g["nan_codes"]:
        assert np.isnan(e4m3_decode(np.array([int(code, 16)], np.uint8))[0])
    assert np.sum(np.isfinite(E4M3_VALUES)) == 254


def test_decode_matches_torch_float8_e4m3fn():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(e4m3_decode(codes), ref, equal_nan=True)


def test_round_ties_and_saturation():
    for x, code, _ in fixture()["rounding"]:
        assert e4m3_round(np.array([x]))[0] == int(code, 16), x


def test_round_trips_every_finite_code():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    assert np.array_equal(e4m3_round(e4m3_decode(codes)), codes)


def test_round_matches_torch_within_range():
    g = np.random.default_rng(7)
    x = np.concatenate([g.standard_normal(200000) * 60.0,                 # normal range
                        g.uniform(-0.02, 0.02, 100000),                   # subnormals
                        (np.arange(-447, 448) + 0.5),                     # midpoints at large magnitudes
                        np.ldexp(np.arange(-64, 64) + 0.5, -9)])          # midpoints among subnormals
    x = x[np.abs(x) <= 448].astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = e4m3_round(x.astype(np.float64))
    # torch keeps the sign of a value that rounds to zero; so does the oracle
    assert np.array_equal(ours, ref)


def test_quantize_by_brute_force():
    g = np.random.default_rng(3)
    W = (g.standard_normal((6, 40)) * 0.03).astype(np.float32)
    W[2] = 0.0                                                            # a zero row
    W[4, 7] = -0.5                                                        # the row maximum is negative
    bits = inputs.f32_to_bf16_bits(W)
    Q, scale = quantize_rows_e4m3(bits)
    Wb = inputs.bf16_bits_to_f32(bits)
    for v in range(W.shape[0]):
        amax = np.float32(max(abs(float(t)) for t in Wb[v]))
        s = np.float32(amax / np.float32(448.0))
        assert scale[v] == s
        for j in range(W.shape[1]):
            if s == 0:
                assert Q[v, j] == 0
                continue
            x = float(np.float32(Wb[v, j] / s))
            # the nearest finite value by exhaustive search, ties to the even code
            best = min((c for c in range(256) if np.isfinite(E4M3_VALUES[c])),
                       key=lambda c: (abs(E4M3_VALUES[c] - x), c % 2, c))
            if E4M3_VALUES[best] == 0 and x != 0:                         # a signed zero keeps x's sign
                best = 0x80 if x < 0 else 0x00
            assert Q[v, j] == best, (v, j, x)
    assert Q[4, 7] == 0xFE and np.all(Q[2] == 0) and scale[2] == 0


def test_quantize_error_bound_and_row_maximum():
    wl = inputs.WORKLOADS["tiny"].with_(V=300, d=96)
    bits = inputs.embedding_bf16(wl)
    Q, scale = quantize_rows_e4m3(bits)
    W = inputs.bf16_bits_to_f32(bits).astype(np.float64)
    deq = dequantize_rows_e4m3(Q, scale)
    x = np.abs(W) / scale[:, None]
    # half a spacing: 2^-4 |x| in the normal range, 2^-10 among the subnormals
    bound = np.maximum(x * 2.0 ** -4, 2.0 ** -10) * scale[:, None]
    assert np.all(np.abs(deq - W) <= bound * (1 + 1e-6))
    a = np.argmax(np.abs(W), axis=1)
    assert np.all(np.isin(Q[np.arange(len(a)), a], (0x7E, 0xFE)))


def test_soft_embed_by_brute_force():
    g = np.random.default_rng(11)
    R, V, d, s, e = 3, 23, 5, 4, 19
    x = (g.standard_normal((R, V)) * 2).astype(np.float32)
    x[1, 6] = -np.inf
    Q = g.integers(0, 256, (e - s + 3, d), dtype=np.uint8)
    Q[Q == 0x7F] = 0x11
    Q[Q == 0xFF] = 0x91
    Q[e - s:] = 0x7F                                                      # NaN padding: never read
    scale = g.uniform(0.001, 0.01, e - s + 3).astype(np.float32)
    lse = row_stats(x)["lse"]
    got = soft_embed_e4m3(x, lse, s, e, Q, scale, 0.75)
    for i in range(R):
        for j in range(d):
            acc = 0.0
            for v in range(s, e):
                c = int(Q[v - s, j])
                sign = -1.0 if c & 0x80 else 1.0
                ex, m = (c >> 3) & 15, c & 7
                val = sign * (m * 2.0 ** -9 if ex == 0 else (1 + m / 8) * 2.0 ** (ex - 7))
                acc += math.exp(float(x[i, v]) - lse[i]) * float(scale[v - s]) * val
            assert abs(got[i, j] - 0.75 * acc) <= 1e-12 * max(1.0, abs(acc))


def test_soft_embed_equals_the_bf16_oracle_on_a_shared_table():
    """A table scale * e4m3(Q) with a power-of-two scale is exactly a bf16 table (E4M3 values
    have four significant bits): both oracles must agree."""
    wl = inputs.WORKLOADS["tiny"].with_(V=5000, d=48, L_c=4, n_req=1)
    x = inputs.logits(wl)
    g = np.random.default_rng(5)
    Q = g.integers(0, 256, (wl.V, wl.d), dtype=np.uint8)
    Q[(Q & 0x7F) == 0x7F] = 0x3C
    scale = np.full(wl.V, 2.0 ** -10, np.float32)
    W = dequantize_rows_e4m3(Q, scale).astype(np.float32)
    bits = inputs.f32_to_bf16_bits(W)
    assert np.array_equal(inputs.bf16_bits_to_f32(bits), W)
    lse = row_stats(x)["lse"]
    a = soft_embed_e4m3(x, lse, 100, 4900, Q[100:4900], scale[100:4900], 1.3)
    b = soft_embed(x, lse, 100, 4900, bits[100:4900], 1.3)
    assert np.allclose(a, b, rtol=1e-12, atol=1e-15)


def test_soft_embed_partition_identity():
    wl = inputs.WORKLOADS["tiny"].with_(V=3001, d=32, L_c=3, n_req=1)
    x = inputs.logits(wl)
    Q, scale = inputs.embedding_e4m3(wl)
    lse = row_stats(x)["lse"]
    full = soft_embed_e4m3(x, lse, 0, wl.V, Q, scale, 1.0)
    parts = sum(soft_embed_e4m3(x, lse, s, e, Q[s:e], scale[s:e], 1.0)
                for s, e in inputs.slice_bounds(wl.V, 4))
    assert np.allclose(full, parts, rtol=1e-12, atol=1e-15)
