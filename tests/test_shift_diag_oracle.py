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
