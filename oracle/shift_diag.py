"""fp64 oracle of the shift-discrepancy diagnostics.

TEST INFRASTRUCTURE ONLY (like the rest of ``oracle/``): only the tests use it.

Source: "When Precision Meets Position: BFloat16 Breaks Down RoPE in
Long-Context Training", architecture page, §3.4 "Diagnostic Methodology:
Measuring the Breakdown":

* Eq. 4, the attention difference D(X, Δ1, Δ2): for one input and two shifts
  of every position, the absolute difference of the post-softmax attention
  weights, summed over the query rows of each key column j, weighted by
  n_j = 1 / (number of rows that may attend to j) and summed over columns and
  heads. Under causal masking the count is L - j + 1 for the 1-based column j,
  which is the page's n = [1/L, 1/(L-1), ..., 1].
* Eq. 5, the first-token logit difference D_logit: (1/T) times the sum over
  heads and query rows of |A_{i,1}(Δ1) - A_{i,1}(Δ2)|, A the pre-softmax logit
  and j = 1 the first token (index 0 here).
* Eq. 3 (same section): under exact arithmetic both are zero, because the
  shift cancels in R_{i+Δ}^T R_{j+Δ} = R_{j-i}.

Readings (also in the design notes): the logit is the softmax input, i.e. the
scaled dot product scale * q~_i . k~_j; "BFloat16 attention" means the
rotated q~, k~ are rounded to bfloat16 (round to nearest even) before the dot
products, which are then exact here (fp64); the column weight n_j counts the
rows of the mask actually in use (CAUSAL, INTRA_DOC or ANCHOR), and a row
that cannot see the first token contributes nothing to Eq. 5.
"""
from __future__ import annotations

import numpy as np

from .anchor_oracle import Problem, _as64, mask_rows, rotate


def round_to_bf16(x) -> np.ndarray:
    """Nearest bfloat16 value (8 significant bits, ties to even) of each fp64 entry."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                       # x = m * 2^e, 0.5 <= |m| < 1
    return np.ldexp(np.rint(m * 256.0) / 256.0, e)


def _rotated(prob: Problem, q, k, bf16_operands: bool):
    qr = rotate(q, prob.pos, prob.base, prob.layout, theta=prob.theta)
    kr = rotate(k, prob.pos, prob.base, prob.layout, theta=prob.theta)
    if bf16_operands:
        qr, kr = round_to_bf16(qr), round_to_bf16(kr)
    return qr, kr


def column_counts(prob: Problem) -> np.ndarray:
    """Number of query rows that may attend to each key (1 / n_j of Eq. 4)."""
    return mask_rows(np.arange(prob.T), prob.doc, prob.mask_mode).sum(axis=0)


def attention_under_shift(prob: Problem, qr, kr, h: int, allowed):
    """Logits A [T, T] (scale * q~_i . k~_j, every pair) and the masked softmax
    ATTN [T, T] of query head h for rotated operands qr [T, Hq, d], kr
    [T, Hkv, d]: the two matrices Eq. 4 and Eq. 5 compare across shifts.
    Masked entries of ATTN are exactly 0 and every row of ATTN sums to 1."""
    g = prob.kv_head(h)
    a = prob.scale * (qr[:, h, :] @ kr[:, g, :].T)
    s = np.where(allowed, a, -np.inf)
    p = np.exp(s - s.max(axis=1, keepdims=True))
    return a, p / p.sum(axis=1, keepdims=True)


def eq4_column_sums(attn1, attn2) -> np.ndarray:
    """Eq. 4's inner sum: for every key column j, sum over the query rows i of
    |ATTN_ij(Δ1) - ATTN_ij(Δ2)|."""
    return np.abs(np.asarray(attn1) - np.asarray(attn2)).sum(axis=0)


def eq4_weighted_total(C, count) -> float:
    """Eq. 4's outer sum for one head: sum_j n_j C_j with n_j = 1 / count_j
    (count_j = rows that may attend to key j); columns nobody sees add 0."""
    C, count = np.asarray(C, np.float64), np.asarray(count)
    seen = count > 0
    return float((C[seen] / count[seen]).sum())


def eq5_first_logit(a1, a2, allowed) -> np.ndarray:
    """Eq. 5's per-row term |A_{i,first}(Δ1) - A_{i,first}(Δ2)| for the first
    token (index 0), 0 for rows that may not attend to it."""
    return np.where(allowed[:, 0], np.abs(np.asarray(a1)[:, 0] - np.asarray(a2)[:, 0]), 0.0)


def shift_diagnostic(prob1: Problem, prob2: Problem, q, k, bf16_operands: bool = True):
    """Eq. 4 and Eq. 5 for one input under the two problems' position shifts.

    ``prob1`` and ``prob2`` must differ only in ``pos_shift``. Returns a dict:
      C [Hq, T]   sum over rows i of |ATTN_ij(Δ1) - ATTN_ij(Δ2)| per key column j
      E [Hq, T]   |A_{i,0}(Δ1) - A_{i,0}(Δ2)| per query row (0 where i cannot see key 0)
      count [T]   rows that may attend to key j
      D           sum_h sum_j C_hj / count_j                     (Eq. 4)
      D_logit     (1 / T) sum_h sum_i E_hi                        (Eq. 5)
    """
    q, k = _as64(q), _as64(k)
    T, Hq = prob1.T, prob1.Hq
    allowed = mask_rows(np.arange(T), prob1.doc, prob1.mask_mode)
    q1, k1 = _rotated(prob1, q, k, bf16_operands)
    q2, k2 = _rotated(prob2, q, k, bf16_operands)
    count = allowed.sum(axis=0)
    C = np.zeros((Hq, T))
    E = np.zeros((Hq, T))
    D = 0.0
    for h in range(Hq):
        a1, p1 = attention_under_shift(prob1, q1, k1, h, allowed)
        a2, p2 = attention_under_shift(prob2, q2, k2, h, allowed)
        C[h] = eq4_column_sums(p1, p2)
        E[h] = eq5_first_logit(a1, a2, allowed)
        D += eq4_weighted_total(C[h], count)
    D_logit = float(E.sum() / T)
    return {"C": C, "E": E, "count": count, "D": D, "D_logit": D_logit}
