"""GPU: the shift-discrepancy diagnostics (aa_shift_diag; "When Precision Meets
Position", architecture page, §3.4 "Diagnostic Methodology: Measuring the
Breakdown", Eq. 4 and Eq. 5) against the fp64 oracle with bf16 operands,
element by element.

The library rotates in fp32 and rounds to bf16; the oracle rotates exactly and
rounds to bf16. The two operands differ only where the exact value lies within
the fp32 rotation's error (ROT_U times the pair's magnitude, derived in
gpu_common) of a bf16 rounding midpoint; there the library may hold the
neighbouring bf16 value. Each per-element bound below follows from that and
from the library's fp32 arithmetic:
  * logit A_ij: the flagged operands' one-ulp moves, scale * sum_c (dq_c |k_c|
    + |q_c| dk_c + dq_c dk_c), plus the sequential fp32 dot product's
    rounding, u * sum_c (D - c) |q_c k_c| (a bound on u times the partial sums),
    plus one rounding of the scaled result;
  * Eq. 5 term |A_i0(Δ1) - A_i0(Δ2)|: the two logit bounds added;
  * ATTN_ij = exp(A_ij - LSE_i): with logit moves |δ_l| <= b_il the ratio
    ATTN'_ij / ATTN_ij lies within exp(+-(b_ij + ln sum_l ATTN_il e^{b_il})),
    and the fp32 online logsumexp and expf add at most
    u * (4 n_i + 64 + 4 max_l |A_il|) and u * (4 + 2 |A_ij - LSE_i|) to that
    exponent (n_i = keys row i sees);
  * Eq. 4 column sum C_j: the ATTN bounds of both shifts summed over the rows,
    plus the fp32 accumulation of the column (u * count_j * (C_j + bound)).
D and D_logit are checked against the same bounds summed with their weights.
The exact properties (equal shifts, no RoPE) are checked bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle as orc
from oracle.shift_diag import round_to_bf16, shift_diagnostic
from gpu_common import ROT_U, bf16_ulp, f64, inputs, pair_norm

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def aa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import packed_sequence_rope_gb300 as pkg
    return pkg


def _plans(aa, cu, T, Hq, Hkv, D, base, mode, d1, d2, layout=orc.ROPE_ADJACENT):
    mk = lambda s: aa.Plan(cu, T, Hq, Hkv, D, base, mode, orc.POS_RESET, layout, pos_shift=s)
    return mk(d1), mk(d2)


U = 2.0 ** -24


def _bf16_neighbours(r):
    """The bf16 values just above and just below each bf16 value r (r != 0)."""
    bits = np.asarray(r, np.float64).astype(np.float32).view(np.uint32)
    up = (bits + np.uint32(0x10000)).view(np.float32).astype(np.float64)
    down = (bits - np.uint32(0x10000)).view(np.float32).astype(np.float64)
    return up, down


def _operand_moves(exact, layout=orc.ROPE_ADJACENT):
    """bf16 rounding of the exact rotated operand, and how far the library's
    bf16 value can be from it: 0 unless the exact value lies within the fp32
    rotation's error of a rounding midpoint, else the spacing across it."""
    r = round_to_bf16(exact)
    up, down = _bf16_neighbours(r)
    tol = ROT_U * pair_norm(exact, layout)
    move = np.zeros_like(r)
    near_up = np.abs(exact - 0.5 * (r + up)) <= tol
    near_down = np.abs(exact - 0.5 * (r + down)) <= tol
    move[near_up] = np.abs(up - r)[near_up]
    move[near_down] = np.maximum(move, np.abs(down - r))[near_down]
    move[r == 0] = bf16_ulp(np.maximum(np.abs(exact), 1e-38))[r == 0]
    return r, move


def _logit_bound(q, dq, k, dk, scale, D):
    """|library logit - oracle logit| bound for every (row, key) of one head."""
    w = (D - np.arange(D, dtype=np.float64))[None, :]
    aq, ak = np.abs(q), np.abs(k)
    flips = dq @ ak.T + aq @ dk.T + dq @ dk.T
    dot = U * ((aq * w) @ ak.T)
    a = np.abs(scale * (q @ k.T))
    return scale * (flips + dot) + U * a


def _attn_bound(a, b, allowed):
    """Bound on |library ATTN - oracle ATTN| for one head and one shift, from
    the oracle's logits a, the logit bounds b and the mask."""
    s = np.where(allowed, a, -np.inf)
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    lse = m + np.log(e.sum(axis=1, keepdims=True))
    P = np.exp(s - lse)
    n = allowed.sum(axis=1, keepdims=True)
    amax = np.where(allowed, np.abs(a), 0.0).max(axis=1, keepdims=True)
    eps_lse = U * (4 * n + 64 + 4 * amax)
    eps_exp = U * (4 + 2 * np.abs(np.where(allowed, a - lse, 0.0)))
    log_s = np.log((P * np.exp(np.where(allowed, b, 0.0))).sum(axis=1, keepdims=True))
    x = np.where(allowed, b, 0.0) + log_s + eps_lse + eps_exp
    return np.where(allowed, P * np.expm1(x), 0.0)


def _elementwise_bounds(prob1, prob2, q, k):
    """Per-element bounds on |library - oracle| for C [Hq, T] and E [Hq, T]."""
    T, Hq, D = prob1.T, prob1.Hq, prob1.d
    allowed = orc.mask_rows(np.arange(T), prob1.doc, prob1.mask_mode)
    count = allowed.sum(axis=0)
    ops = []
    for p in (prob1, prob2):
        qe = orc.rotate(f64(q), p.pos, p.base, p.layout)
        ke = orc.rotate(f64(k), p.pos, p.base, p.layout)
        ops.append(_operand_moves(qe) + _operand_moves(ke))
    BC = np.zeros((Hq, T))
    BE = np.zeros((Hq, T))
    for h in range(Hq):
        g = prob1.kv_head(h)
        cols = np.zeros(T)
        for qr, dq, kr, dk in ops:
            b = _logit_bound(qr[:, h], dq[:, h], kr[:, g], dk[:, g], prob1.scale, D)
            a = prob1.scale * (qr[:, h] @ kr[:, g].T)
            cols += _attn_bound(a, b, allowed).sum(axis=0)
            BE[h] += np.where(allowed[:, 0], b[:, 0], 0.0)
        BC[h] = cols
    return BC, BE, count


CASES = [
    # name, cu, T, Hq, Hkv, D, base, mode, d1, d2
    ("causal", None, 300, 2, 2, 128, 1e4, orc.MASK_CAUSAL, 0, 16),
    ("causal_far", None, 257, 2, 1, 128, 1e4, orc.MASK_CAUSAL, 2000, 16),
    ("anchor_packed", [1, 40, 41, 200, 513], 513, 2, 2, 128, 5e5, orc.MASK_ANCHOR, 0, 16),
    ("intra_doc_d64", [1, 100, 333], 333, 4, 2, 64, 1e4, orc.MASK_INTRA_DOC, 5, 500),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_matches_oracle_elementwise(aa, case):
    name, cu, T, Hq, Hkv, D, base, mode, d1, d2 = case
    q, k, _, _ = inputs(T, Hq, Hkv, D, seed=11)
    p1, p2 = _plans(aa, cu, T, Hq, Hkv, D, base, mode, d1, d2)
    with p1, p2:
        col, first, res = p1.shift_diag(p2, q, k)
        torch.cuda.synchronize()
    col, first, res = f64(col), f64(first), res.cpu().numpy()
    mk = lambda s: orc.Problem(cu, T, Hq, Hkv, D, base, mode, orc.POS_RESET, orc.ROPE_ADJACENT, pos_shift=s)
    ref = shift_diagnostic(mk(d1), mk(d2), q.cpu(), k.cpu())
    BC, BE, count = _elementwise_bounds(mk(d1), mk(d2), q.cpu(), k.cpu())
    BC = BC + U * count * (ref["C"] + BC)
    BE = BE + U * (ref["E"] + BE)
    assert ref["D"] > 0 and ref["D_logit"] > 0
    ec, ee = np.abs(col - ref["C"]), np.abs(first - ref["E"])
    seen = ref["C"] > 0
    print(name, f"C: max err/bound {np.max(ec / np.maximum(BC, 1e-300)):.3f}, median bound/C "
          f"{np.median(BC[seen] / ref['C'][seen]):.3f}; E: max err/bound {np.max(ee / np.maximum(BE, 1e-300)):.3f}")
    assert (ec <= BC).all(), f"{name}: {int((ec > BC).sum())} column sums outside their bounds"
    assert (ee <= BE).all(), f"{name}: {int((ee > BE).sum())} first-token terms outside their bounds"
    # the totals, with the same bounds weighted as Eq. 4 and Eq. 5 weight the terms
    w = np.where(count > 0, 1.0 / np.maximum(count, 1), 0.0)
    assert abs(res[0] - ref["D"]) <= (BC * w).sum() + 1e-12
    assert abs(res[1] - ref["D_logit"]) <= BE.sum() / T + 1e-12
    # per-head sums add up to the totals
    assert res[2::2].sum() == pytest.approx(res[0], rel=1e-12)
    assert res[3::2].sum() / T == pytest.approx(res[1], rel=1e-12)
    # rows that cannot see token 0 report no first-token difference
    if mode == orc.MASK_INTRA_DOC:
        assert not first[:, 1:].any()


@pytest.mark.parametrize("mode", [orc.MASK_CAUSAL, orc.MASK_ANCHOR])
def test_equal_shifts_are_exactly_zero(aa, mode):
    cu = None if mode == orc.MASK_CAUSAL else [1, 64, 300]
    q, k, _, _ = inputs(300, 2, 2, 128, seed=12)
    p1, p2 = _plans(aa, cu, 300, 2, 2, 128, 1e4, mode, 9, 9)
    with p1, p2:
        col, first, res = p1.shift_diag(p2, q, k)
        torch.cuda.synchronize()
    assert not col.any() and not first.any() and not res.any()


def test_no_rope_is_exactly_zero(aa):
    q, k, _, _ = inputs(200, 2, 2, 128, seed=13)
    p1, p2 = _plans(aa, None, 200, 2, 2, 128, 1e4, orc.MASK_CAUSAL, 0, 1000, orc.ROPE_NONE)
    with p1, p2:
        col, first, res = p1.shift_diag(p2, q, k)
        torch.cuda.synchronize()
    assert not col.any() and not first.any() and not res.any()


def test_mismatched_plans_are_refused(aa):
    q, k, _, _ = inputs(128, 1, 1, 64, seed=14)
    with aa.Plan(None, 128, 1, 1, 64, 1e4, orc.MASK_CAUSAL) as p1, \
            aa.Plan(None, 128, 1, 1, 64, 5e5, orc.MASK_CAUSAL) as p2:
        with pytest.raises(aa.AAError, match="differ only in pos_shift"):
            p1.shift_diag(p2, q, k)
