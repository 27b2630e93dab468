"""Pins of the fp64 shift-discrepancy oracle ("When Precision Meets Position",
architecture page, §3.4 "Diagnostic Methodology: Measuring the Breakdown",
Eq. 4 and Eq. 5; Eq. 3 for the invariance they measure). CPU only."""
import math

import numpy as np
import pytest
import torch

import oracle as orc
from oracle.shift_diag import column_counts, round_to_bf16, shift_diagnostic


def _problems(cu, T, H, d, base, mode, d1, d2, layout=orc.ROPE_ADJACENT, Hkv=None):
    mk = lambda s: orc.Problem(cu, T, H, Hkv or H, d, base, mode, orc.POS_RESET, layout, pos_shift=s)
    return mk(d1), mk(d2)


def _qk(T, H, d, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(T, H, d, generator=g, dtype=torch.float64)
    k = torch.randn(T, H, d, generator=g, dtype=torch.float64)
    return q.numpy(), k.numpy()


def test_round_to_bf16_matches_torch_on_fp32_values():
    # fp32-representable inputs, so torch's fp32 -> bf16 conversion is a single rounding
    x = torch.randn(20000, dtype=torch.float32, generator=torch.Generator().manual_seed(0)) * 37
    ref = x.to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(round_to_bf16(x.double().numpy()), ref)


def test_round_to_bf16_ties_go_to_even():
    assert round_to_bf16(1 + 2 ** -8) == 1.0                       # tie, even mantissa below
    assert round_to_bf16(1 + 3 * 2 ** -8) == 1 + 2 ** -6           # tie, rounds up to even
    assert round_to_bf16(-(1 + 2 ** -8 + 2 ** -20)) == -(1 + 2 ** -7)


def test_causal_column_weights_are_the_pages_n():
    # n = [1/L, 1/(L-1), ..., 1]: column j (1-based) has L - j + 1 rows
    L = 37
    p, _ = _problems(None, L, 1, 4, 1e4, orc.MASK_CAUSAL, 0, 0)
    assert np.array_equal(column_counts(p), L - np.arange(L))


def test_anchor_column_is_seen_by_every_row():
    cu = [1, 10, 30, 64]
    p, _ = _problems(cu, 64, 1, 4, 1e4, orc.MASK_ANCHOR, 0, 0)
    cnt = column_counts(p)
    assert cnt[0] == 64 and cnt[9] == 1 and cnt[1] == 9    # doc [1, 10): key 1 seen by rows 1..9


@pytest.mark.parametrize("mode", [orc.MASK_CAUSAL, orc.MASK_ANCHOR])
def test_equal_shifts_give_zero(mode):
    cu = None if mode == orc.MASK_CAUSAL else [1, 50, 130, 200]
    q, k = _qk(200, 2, 16, 1)
    r = shift_diagnostic(*_problems(cu, 200, 2, 16, 1e4, mode, 7, 7), q, k)
    assert r["D"] == 0.0 and r["D_logit"] == 0.0 and not r["C"].any() and not r["E"].any()


@pytest.mark.parametrize("mode", [orc.MASK_CAUSAL, orc.MASK_ANCHOR, orc.MASK_INTRA_DOC])
def test_exact_arithmetic_is_shift_invariant(mode):
    # Eq. 3: without bfloat16 operands the shift cancels, D = D_logit = 0 up to fp64 rounding
    cu = None if mode == orc.MASK_CAUSAL else [1, 40, 41, 256]
    q, k = _qk(256, 2, 32, 2)
    r = shift_diagnostic(*_problems(cu, 256, 2, 32, 1e4, mode, 0, 1000), q, k, bf16_operands=False)
    assert r["D"] < 1e-9 and r["D_logit"] < 1e-9


def test_bfloat16_operands_break_the_invariance():
    q, k = _qk(256, 2, 32, 3)
    r = shift_diagnostic(*_problems(None, 256, 2, 32, 1e4, orc.MASK_CAUSAL, 0, 16), q, k)
    assert r["D"] > 1e-4 and r["D_logit"] > 1e-4


def test_no_rope_gives_exactly_zero():
    q, k = _qk(128, 1, 16, 4)
    r = shift_diagnostic(*_problems(None, 128, 1, 16, 1e4, orc.MASK_CAUSAL, 0, 500, orc.ROPE_NONE), q, k)
    assert r["D"] == 0.0 and r["D_logit"] == 0.0


def test_symmetric_and_bounded():
    q, k = _qk(160, 2, 16, 5)
    a = shift_diagnostic(*_problems(None, 160, 2, 16, 1e4, orc.MASK_CAUSAL, 3, 40), q, k)
    b = shift_diagnostic(*_problems(None, 160, 2, 16, 1e4, orc.MASK_CAUSAL, 40, 3), q, k)
    assert a["D"] == b["D"] and a["D_logit"] == b["D_logit"]
    # each row's two distributions are at L1 distance <= 2
    assert (a["C"].sum(axis=1) <= 2 * 160 + 1e-9).all()


def test_first_token_logits_closed_form():
    # d = 2 (one pair, theta_0 = 1), q_i = (1, 0), k_0 = (1, 0): the rotated
    # vectors are (cos, sin) of the positions, so A_i0 = scale (c_i c_0 + s_i s_0)
    # with every factor rounded to bfloat16
    T, d1, d2 = 50, 0, 16
    q = np.zeros((T, 1, 2)); q[:, 0, 0] = 1.0
    k = np.zeros((T, 1, 2)); k[:, 0, 0] = 1.0
    r = shift_diagnostic(*_problems(None, T, 1, 2, 1e4, orc.MASK_CAUSAL, d1, d2), q, k)
    bf = lambda x: float(round_to_bf16(x))
    scale = 1 / math.sqrt(2)

    def logit(i, s):
        return scale * (bf(math.cos(i + s)) * bf(math.cos(s)) + bf(math.sin(i + s)) * bf(math.sin(s)))
    want = [abs(logit(i, d1) - logit(i, d2)) for i in range(T)]
    assert np.allclose(r["E"][0], want, rtol=0, atol=1e-15)
    assert r["D_logit"] == pytest.approx(sum(want) / T, abs=1e-15)


# ---------------------------------------------------------------- Eq. 4 by hand
def test_eq4_hand_computed_three_by_three():
    # Eq. 4 for one head, causal L = 3, with two attention matrices written out
    # (rows i = queries, columns j = keys; each row sums to 1, zeros above the
    # diagonal):
    #   ATTN(Δ1) = [[1, 0, 0], [3/4, 1/4, 0], [1/2, 1/4, 1/4]]
    #   ATTN(Δ2) = [[1, 0, 0], [1/2, 1/2, 0], [1/4, 1/4, 1/2]]
    #   |diff|   = [[0, 0, 0], [1/4, 1/4, 0], [1/4, 0, 1/4]]
    # summed over the rows of each column: C = [1/2, 1/4, 1/4]; the causal
    # weights n = [1/L, 1/(L-1), 1] = [1/3, 1/2, 1], so
    #   D = (1/2)(1/3) + (1/4)(1/2) + (1/4)(1) = 13/24.
    # Summing over the wrong axis (row sums [0, 1/2, 1/2]) would give 3/4;
    # weighting by 1/(j+1) instead would give 17/24.
    from oracle.shift_diag import eq4_column_sums, eq4_weighted_total
    p1 = np.array([[1, 0, 0], [0.75, 0.25, 0], [0.5, 0.25, 0.25]])
    p2 = np.array([[1, 0, 0], [0.5, 0.5, 0], [0.25, 0.25, 0.5]])
    C = eq4_column_sums(p1, p2)
    assert np.array_equal(C, [0.5, 0.25, 0.25])
    p, _ = _problems(None, 3, 1, 2, 1e4, orc.MASK_CAUSAL, 0, 0)
    count = column_counts(p)
    assert np.array_equal(count, [3, 2, 1])
    assert eq4_weighted_total(C, count) == pytest.approx(13 / 24, abs=1e-15)


def test_eq4_one_hot_flip_worked_example():
    # End to end with d = 2 (one pair, theta_0 = 1 rad per position), causal
    # L = 3, every q_i = (1, 0) and every k_j = (cos 1/2, sin 1/2). In exact
    # arithmetic the logit of (i, j) is scale * cos(j - i + 1/2): row 1 ties
    # keys 0 and 1 (cos(-1/2) = cos(1/2)) and row 2 ties keys 1 and 2, key 0
    # far below (cos(-3/2) = 0.07). The shift cancels (Eq. 3); the bfloat16
    # rounding of the rotated operands breaks the ties. Rounded by hand (8
    # significant bits, to nearest):
    #   Δ = 0: q~_2 = (cos 2, sin 2) -> (-0.416015625, 0.91015625)
    #          k~_1 = (cos 1.5, sin 1.5) -> (0.07080078125, 0.99609375)
    #          k~_2 = (cos 2.5, sin 2.5) -> (-0.80078125, 0.59765625)
    #          row 2: key 1 0.877146721 > key 2 0.877098083 -> key 1
    #          row 1: key 0 0.875663757 > key 1 0.874729156 -> key 0
    #   Δ = 1: row 2: key 2 0.876731873 > key 1 0.876026154 -> key 2
    #          row 1: key 0 0.877146721 > key 1 0.877098083 -> key 0
    # With scale = 1e6 the smallest gap (4.9e-5) is 49 in the exponent, so
    # every softmax row is one-hot to within e^-49. Row 2 moves from key 1 to
    # key 2, rows 0 and 1 do not move: C = [0, 1, 1] and, with the weights
    # [1/3, 1/2, 1], D = 1/2 + 1 = 3/2.
    T = 3
    q = np.zeros((T, 1, 2)); q[:, 0, 0] = 1.0
    k = np.zeros((T, 1, 2)); k[:, 0, 0] = math.cos(0.5); k[:, 0, 1] = math.sin(0.5)
    mk = lambda s: orc.Problem(None, T, 1, 1, 2, 1e4, orc.MASK_CAUSAL, orc.POS_RESET, orc.ROPE_ADJACENT,
                               softmax_scale=1e6, pos_shift=s)
    r = shift_diagnostic(mk(0), mk(1), q, k)
    assert np.allclose(r["C"][0], [0.0, 1.0, 1.0], rtol=0, atol=1e-18)
    assert r["D"] == pytest.approx(1.5, abs=1e-18)


def test_attention_under_shift_equals_the_forward_oracle():
    # the per-shift attention is the forward oracle's softmax: ATTN @ v equals
    # forward()'s output for the same (already rotated, bf16) operands with
    # rotation off, and ATTN's rows sum to 1 with exact zeros where masked
    from oracle.shift_diag import attention_under_shift
    cu, T, H, Hkv, d = [1, 20, 21, 64], 64, 2, 1, 16
    q, k = _qk(T, H, d, 9)
    k = k[:, :Hkv]
    v = np.random.default_rng(9).standard_normal((T, Hkv, d))
    p = orc.Problem(cu, T, H, Hkv, d, 1e4, orc.MASK_ANCHOR, orc.POS_RESET, pos_shift=40)
    qr = round_to_bf16(orc.rotate(q, p.pos, 1e4))
    kr = round_to_bf16(orc.rotate(k, p.pos, 1e4))
    allowed = orc.mask_rows(np.arange(T), p.doc, orc.MASK_ANCHOR)
    none = orc.Problem(cu, T, H, Hkv, d, 1e4, orc.MASK_ANCHOR, orc.POS_RESET, orc.ROPE_NONE)
    O, _ = orc.forward(none, qr, kr, v)
    for h in range(H):
        _, attn = attention_under_shift(p, qr, kr, h, allowed)
        assert np.allclose(attn @ v[:, 0, :], O[:, h, :], rtol=0, atol=1e-12)
        assert np.allclose(attn.sum(axis=1), 1.0, rtol=0, atol=1e-14)
        assert not attn[~allowed].any()
