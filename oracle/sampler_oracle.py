"""CPU oracle for the DiffusionGemma denoising-sampler step (fp64, plain and slow).

TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
benchmark's CPU-baseline leg may import this module.  The product path (the C-ABI
library and its Python binding) never calls it and shares no code with it.

Every quantity is computed in float64 from the fp32 logits and the bf16
embedding, straight from its definition, in the order the pages give:

* row statistics - the softmax over the full vocabulary, its entropy, the argmax
  candidate and its confidence (calvarado04.com, "Where the shapes stop
  agreeing", eq. e^sc: p_i is a distribution over all V tokens; agentlenshq.com,
  "サンプリングループとエントロピー境界デノイジング": candidates at every position and
  an entropy per position);
* entropy-bound acceptance - positions taken from most to least confident until
  the running entropy would pass the budget (agentlenshq.com, same section);
* the self-conditioning soft embedding E = gamma * P[:, s:e] W_shard[0:e-s]
  (calvarado04.com, eq. e^sc, "The fix": the partition identity and the
  fixed code, with gamma the learned normaliser applied after the sum);
* the sum of per-slice partials, E = gamma * sum_r S_r (calvarado04.com, "The fix").

Pinned by tests/test_oracle_pins.py against closed forms, brute force and the
pages' printed numbers.  Parity beyond the stated tolerance is unpinned for the
soft embedding: no page fixes the bf16 rounding of the probabilities or the
order of the additions, so only the tolerance bounds those.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

VOCAB_CHUNK = 16384     # vocabulary rows of W per matmul step


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Decode bfloat16 bit patterns (uint16) to float64: the top 16 bits of an IEEE single."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def row_stats(logits: np.ndarray) -> dict:
    """Per-row softmax statistics of fp32 logits [R, V] (float64 results).

    For row i with logits l_i:
      m_i    = max_v l_{i,v};  a_i = the smallest v with l_{i,v} = m_i (torch.argmax convention)
      Z_i    = sum_v exp(l_{i,v} - m_i)
      lse_i  = m_i + ln Z_i
      p_{i,v} = exp(l_{i,v} - lse_i)
      H_i    = -sum_{v: p_{i,v} > 0} p_{i,v} ln p_{i,v}           (nats, temperature 1)
      conf_i = p_{i,a_i} = 1 / Z_i
      kappa_i = -ln conf_i = ln Z_i, evaluated as log1p(rest_i) with
                rest_i = sum_{v != a_i} exp(l_{i,v} - m_i), so that rows near one-hot
                keep their order (1/Z rounds to 1 long before rest vanishes).
    A row whose logits are all -inf has no distribution: its statistics are NaN
    and its argmax is 0.
    """
    x = np.asarray(logits, dtype=np.float32)
    R, V = x.shape
    out = {k: np.empty(R, np.float64) for k in ("m", "lse", "H", "kappa", "conf")}
    out["argmax"] = np.empty(R, np.int64)

    def one_row(i: int) -> None:
        l = x[i].astype(np.float64)
        m = l.max()
        a = int(np.argmax(l))
        out["m"][i] = m
        out["argmax"][i] = a
        if m == -np.inf:
            for k in ("lse", "H", "kappa", "conf"):
                out[k][i] = np.nan
            out["argmax"][i] = 0
            return
        e = np.exp(l - m)
        Z = e.sum()
        lse = m + math.log(Z)
        p = np.exp(l - lse)
        pos = p > 0
        H = -np.sum(p[pos] * np.log(p[pos]))
        rest = np.delete(e, a).sum()
        out["lse"][i] = lse
        out["H"][i] = H
        out["kappa"][i] = math.log1p(rest)
        out["conf"][i] = 1.0 / Z

    # rows are independent; the pool only spreads them over the host's cores
    with ThreadPoolExecutor(max(1, min(32, os.cpu_count() or 1))) as ex:
        list(ex.map(one_row, range(R)))
    return out


def entropy_accept(H: np.ndarray, kappa: np.ndarray, n_req: int, L_c: int,
                   budgets: np.ndarray, min_accept: int = 0) -> dict:
    """Entropy-bound acceptance per request.

    For request q with positions 0..L_c-1 (rows q*L_c + j) and budget B_q:
      order  = positions from most to least confident: kappa ascending (= confidence
               descending), equal confidence broken by the lower position first; a
               position without a distribution (NaN statistics: all logits -inf) has no
               confidence and goes after every other;
      C_k    = H[order_1] + ... + H[order_k];
      n      = the largest k in 0..L_c with C_k <= B_q - positions are taken in order
               and taking stops at the first one that would carry the running
               entropy past the budget;
      n      = max(n, min(min_accept, L_c))   (min_accept = 0 is the literal rule);
      mask[order_j] = 1 for j < n.
    Returns order (local positions, int64 [R]), mask (uint8 [R]) and n_accepted
    (int64 [n_req]).
    """
    H = np.asarray(H, np.float64)
    kappa = np.asarray(kappa, np.float64)
    R = n_req * L_c
    order = np.empty(R, np.int64)
    mask = np.zeros(R, np.uint8)
    n_acc = np.empty(n_req, np.int64)
    for q in range(n_req):
        base = q * L_c
        pos = sorted(range(L_c), key=lambda j: (bool(np.isnan(kappa[base + j])), kappa[base + j], j))
        B = float(budgets[q])
        running, n = 0.0, 0
        for k, j in enumerate(pos):
            running += H[base + j]
            if running <= B:         # False once the sum is NaN: a NaN position stops it
                n = k + 1
            else:
                break
        n = max(n, min(int(min_accept), L_c))
        for k, j in enumerate(pos):
            order[base + k] = j
            if k < n:
                mask[base + j] = 1
        n_acc[q] = n
    return {"order": order, "mask": mask, "n_accepted": n_acc}


def soft_embed(logits: np.ndarray, lse: np.ndarray, vocab_start: int, vocab_end: int,
               W_shard_bits: np.ndarray, gamma: float, rows: np.ndarray | None = None) -> np.ndarray:
    """Self-conditioning soft embedding over the vocabulary slice [vocab_start, vocab_end).

      P_{i,v} = exp(l_{i,v} - lse_i)           (softmax over the FULL vocabulary; never
                                                renormalised inside the slice)
      E_{i,:} = gamma * sum_{v=s}^{e-1} P_{i,v} W_shard[v - s, :]

    W_shard holds the slice's rows first; any padding rows after row e-s are not
    part of the product.  ``rows`` optionally restricts the output to a subset of
    rows (the result then has len(rows) rows).  float64 throughout; the
    probabilities are not rounded to bf16.
    """
    s, e = int(vocab_start), int(vocab_end)
    x = np.asarray(logits, dtype=np.float32)
    idx = np.arange(x.shape[0]) if rows is None else np.asarray(rows)
    d = W_shard_bits.shape[1]
    E = np.zeros((len(idx), d), np.float64)
    lse_sel = np.asarray(lse, np.float64)[idx]
    for v0 in range(s, e, VOCAB_CHUNK):
        v1 = min(e, v0 + VOCAB_CHUNK)
        P = np.exp(x[idx, v0:v1].astype(np.float64) - lse_sel[:, None])
        Wc = bf16_bits_to_f64(W_shard_bits[v0 - s:v1 - s])
        E += P @ Wc
    return float(gamma) * E


def sum_partials(partials: list, gamma: float) -> np.ndarray:
    """E = gamma * (S_0 + S_1 + ... + S_{T-1}), summed in rank order."""
    acc = np.zeros_like(np.asarray(partials[0], np.float64))
    for S in partials:
        acc = acc + np.asarray(S, np.float64)
    return float(gamma) * acc
