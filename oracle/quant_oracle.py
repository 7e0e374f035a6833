"""CPU oracle of the self-conditioning soft embedding with an 8-bit embedding table.

TEST INFRASTRUCTURE ONLY: only the test suite, the smoke check and the benchmark's
CPU-baseline leg may import this module; the product path never calls it and shares no
code with it.

The pages say the model runs from quantised checkpoints (calvarado04.com, "Running it":
INT8 dynamic; agentlenshq.com, "量子化チェックポイント": FP8 weights with dynamic
activations, or NVFP4) but never that the embedding table is quantised, nor how.  The
reading taken here, the plainest one for a table that the step reads only through the
product E = gamma * P W:

* the table is held as FP8 E4M3 codes, one byte per entry, with one fp32 scale per
  vocabulary row: W[v, j] = scale_v * e4m3(Q[v, j]);
* the E4M3 format is the OCP 8-bit floating-point format ("E4M3FN"): 1 sign bit, 4
  exponent bits with bias 7, 3 mantissa bits; exponent field 0 holds the subnormals
  m * 2^-9; there is no infinity; S.1111.111 is NaN, so the largest finite magnitude is
  S.1111.110 = 448;
* a row is quantised against its largest magnitude: scale_v = amax_v / 448 in fp32, each
  entry divided by scale_v in fp32 and rounded to the nearest E4M3 value, ties to the even
  code, magnitudes past 448 saturating to 448; a row of zeros keeps scale 0 and codes 0;
* the product is the soft embedding of the dequantised table: the probabilities are taken
  exactly (float64), not cast to 8 bits.
"""
from __future__ import annotations

import numpy as np

from .sampler_oracle import VOCAB_CHUNK, bf16_bits_to_f64

E4M3_MAX = 448.0
NAN_CODES = (0x7F, 0xFF)


def _decode_one(code: int) -> float:
    """The value of one E4M3 code, from the format's definition."""
    sign = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return sign * m * 2.0 ** -9           # subnormal: 0.m * 2^(1 - 7)
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


E4M3_VALUES = np.array([_decode_one(c) for c in range(256)], np.float64)
# the non-negative finite codes 0x00 .. 0x7E in increasing order of value
_POS_VALUES = E4M3_VALUES[:0x7F]


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """float64 values of E4M3 codes (uint8)."""
    return E4M3_VALUES[np.asarray(codes, np.uint8)]


def e4m3_round(x: np.ndarray) -> np.ndarray:
    """E4M3 codes of x: the nearest finite E4M3 value, ties to the even code, magnitudes
    above 448 saturated to 448 (NaN maps to the NaN code 0x7F)."""
    x = np.asarray(x, np.float64)
    a = np.abs(x)
    # index of the first non-negative value >= |x|; the nearest is it or the one below
    hi = np.clip(np.searchsorted(_POS_VALUES, a, side="left"), 0, 0x7E)
    lo = np.clip(hi - 1, 0, 0x7E)
    d_hi = np.abs(_POS_VALUES[hi] - a)
    d_lo = np.abs(a - _POS_VALUES[lo])
    pick_lo = (d_lo < d_hi) | ((d_lo == d_hi) & (lo % 2 == 0))
    code = np.where(pick_lo, lo, hi)
    code = np.where(a >= E4M3_MAX, 0x7E, code)
    code = code | np.where(np.signbit(x), 0x80, 0)
    code = np.where(np.isnan(x), 0x7F, code)
    return code.astype(np.uint8)


def quantize_rows_e4m3(W_bits: np.ndarray) -> tuple:
    """Per-row E4M3 quantisation of a bf16 table [V, d] (uint16 bit patterns).

    scale_v = fp32(amax_v / 448), amax_v = max_j |W[v, j]|;
    Q[v, j] = e4m3_round(fp32(W[v, j] / scale_v)), both divisions correctly rounded fp32;
    a row with amax_v = 0 gets scale 0 and codes 0.  Returns (Q uint8 [V, d], scale fp32 [V]).
    """
    W = bf16_bits_to_f64(W_bits).astype(np.float32)          # bf16 -> fp32 is exact
    amax = np.max(np.abs(W), axis=1)
    scale = (amax / np.float32(E4M3_MAX)).astype(np.float32)
    Q = np.zeros(W.shape, np.uint8)
    nz = scale > 0
    if np.any(nz):
        x = (W[nz] / scale[nz, None]).astype(np.float32)     # fp32 / fp32, rounded to fp32
        Q[nz] = e4m3_round(x.astype(np.float64))
    return Q, scale


def dequantize_rows_e4m3(Q: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """float64 table W[v, j] = scale_v * e4m3(Q[v, j])."""
    return e4m3_decode(Q) * np.asarray(scale, np.float64)[:, None]


def soft_embed_e4m3(logits: np.ndarray, lse: np.ndarray, vocab_start: int, vocab_end: int,
                    Q_shard: np.ndarray, scale_shard: np.ndarray, gamma: float,
                    rows: np.ndarray | None = None) -> np.ndarray:
    """E = gamma * P[:, s:e] W_shard[0:e-s] with the 8-bit table W_shard[v] = scale_v e4m3(Q_v).

    P_{i,v} = exp(l_{i,v} - lse_i) over the full vocabulary, as for the bf16 table; row j
    of the shard is vocabulary entry s + j and padding rows are not part of the product.
    float64 throughout.
    """
    s, e = int(vocab_start), int(vocab_end)
    x = np.asarray(logits, dtype=np.float32)
    idx = np.arange(x.shape[0]) if rows is None else np.asarray(rows)
    d = Q_shard.shape[1]
    E = np.zeros((len(idx), d), np.float64)
    lse_sel = np.asarray(lse, np.float64)[idx]
    for v0 in range(s, e, VOCAB_CHUNK):
        v1 = min(e, v0 + VOCAB_CHUNK)
        P = np.exp(x[idx, v0:v1].astype(np.float64) - lse_sel[:, None])
        E += P @ dequantize_rows_e4m3(Q_shard[v0 - s:v1 - s], scale_shard[v0 - s:v1 - s])
    return float(gamma) * E
