"""GPU: the shift-discrepancy diagnostics (aa_shift_diag; "When Precision Meets
Position", architecture page, §3.4 "Diagnostic Methodology: Measuring the
Breakdown", Eq. 4 and Eq. 5) against the fp64 oracle with bf16 operands.

The library's rotated operands come from its fp32 RoPE kernel and the oracle's
from an exact rotation, each rounded to bf16; the two agree except where the
fp32 rotation lands on the other side of a bf16 rounding midpoint (a small
fraction of elements, each then one bf16 ulp apart). The diagnostics measure
exactly such rounding differences, so they are compared in aggregate. Observed
on a GB300: D within 1.5e-4 and D_logit within 1e-3 (relative), the per-column
vector within 2e-3 and the per-row first-token vector within 1.3e-2 (relative
L2); the bounds below are about 3-5x those. The exact properties (equal shifts,
no RoPE) are checked bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle as orc
from oracle.shift_diag import shift_diagnostic
from gpu_common import inputs

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


def _rel(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


CASES = [
    # name, cu, T, Hq, Hkv, D, base, mode, d1, d2
    ("causal", None, 300, 2, 2, 128, 1e4, orc.MASK_CAUSAL, 0, 16),
    ("causal_far", None, 257, 2, 1, 128, 1e4, orc.MASK_CAUSAL, 2000, 16),
    ("anchor_packed", [1, 40, 41, 200, 513], 513, 2, 2, 128, 5e5, orc.MASK_ANCHOR, 0, 16),
    ("intra_doc_d64", [1, 100, 333], 333, 4, 2, 64, 1e4, orc.MASK_INTRA_DOC, 5, 500),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_matches_oracle(aa, case):
    name, cu, T, Hq, Hkv, D, base, mode, d1, d2 = case
    q, k, _, _ = inputs(T, Hq, Hkv, D, seed=11)
    p1, p2 = _plans(aa, cu, T, Hq, Hkv, D, base, mode, d1, d2)
    with p1, p2:
        col, first, res = p1.shift_diag(p2, q, k)
        torch.cuda.synchronize()
    res = res.cpu().numpy()
    mk = lambda s: orc.Problem(cu, T, Hq, Hkv, D, base, mode, orc.POS_RESET, orc.ROPE_ADJACENT, pos_shift=s)
    ref = shift_diagnostic(mk(d1), mk(d2), q.cpu(), k.cpu())
    errs = {"D": abs(res[0] - ref["D"]) / ref["D"], "D_logit": abs(res[1] - ref["D_logit"]) / ref["D_logit"],
            "col": _rel(col.cpu(), ref["C"]), "first": _rel(first.cpu(), ref["E"])}
    print(name, {k_: f"{v:.2e}" for k_, v in errs.items()}, "D", res[0], ref["D"], "D_logit", res[1], ref["D_logit"])
    assert ref["D"] > 0 and ref["D_logit"] > 0
    assert errs["D"] <= 5e-4 and errs["D_logit"] <= 5e-3, errs
    assert errs["col"] <= 1e-2 and errs["first"] <= 5e-2, errs
    # per-head sums add up to the totals
    assert res[2::2].sum() == pytest.approx(res[0], rel=1e-12)
    assert res[3::2].sum() / T == pytest.approx(res[1], rel=1e-12)
    # rows that cannot see token 0 report no first-token difference
    if mode == orc.MASK_INTRA_DOC:
        assert not first.cpu()[:, 1:].any()


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
