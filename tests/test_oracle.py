"""Pins for the fp64 oracle: each check comes from something other than the oracle.

Hand-enumerated masks and positions (tests/golden), closed forms (pair count,
two-key softmax, anchor row), the RoPE relative property (Eq. 3) and its
complex-number form, an independent library attention (torch SDPA in fp64),
torch autograd and central finite differences for the backward pass.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle as orc
from aa_synth import pack, doc_lengths

MODES = {"ANCHOR": orc.MASK_ANCHOR, "INTRA_DOC": orc.MASK_INTRA_DOC, "CAUSAL": orc.MASK_CAUSAL}


def _read_masks(path):
    out, cur = {}, None
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        if line.startswith("mode"):
            cur = line.split()[1]
            out[cur] = []
        else:
            out[cur].append([int(x) for x in line.split()])
    return {k: np.array(v, dtype=bool) for k, v in out.items()}


def test_masks_match_hand_enumeration(golden_dir):
    masks = _read_masks(os.path.join(golden_dir, "mask_T8_docs3_4.txt"))
    for name, expected in masks.items():
        got = orc.attention_mask([1, 4, 8], 8, MODES[name])
        assert (got == expected).all(), name


def test_positions_match_hand_enumeration(golden_dir):
    rows = {}
    for line in open(os.path.join(golden_dir, "positions_T8_docs3_4.txt")):
        if line.strip() and not line.startswith("#"):
            f = line.split()
            rows[f[0]] = [int(x) for x in f[1:]]
    cu = [1, 4, 8]
    assert list(orc.position_ids(cu, 8, orc.MASK_ANCHOR, orc.POS_RESET)) == rows["RESET"]
    assert list(orc.position_ids(cu, 8, orc.MASK_ANCHOR, orc.POS_CONTINUOUS)) == rows["CONTINUOUS"]
    assert list(orc.position_ids(cu, 8, orc.MASK_ANCHOR, orc.POS_RESET, 5)) == rows["SHIFT5_RESET"]
    assert list(orc.position_ids(cu, 8, orc.MASK_CAUSAL, orc.POS_RESET)) == rows["CONTINUOUS"]


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_pair_count_closed_form(seed):
    # "Reduction in attention computations": K documents cost sum_k N_k(N_k+1)/2
    # intra-document causal pairs, plus one anchor edge per document token,
    # plus the anchor's own pair.
    rng = np.random.default_rng(seed)
    T = 1000 + 37 * seed
    cu = pack(doc_lengths("loguniform", T - 1, rng, lo=5, hi=300), T)
    n = np.diff(cu).astype(np.int64)
    intra = int((n * (n + 1) // 2).sum())
    assert orc.unmasked_pairs(cu, T, orc.MASK_ANCHOR) == 1 + intra + int(n.sum())
    assert orc.unmasked_pairs(cu, T, orc.MASK_INTRA_DOC) == 1 + intra
    assert orc.unmasked_pairs(cu, T, orc.MASK_CAUSAL) == T * (T + 1) // 2


def test_tile_counts_hand_cases():
    # single document: every causal tile is live in every mode
    assert orc.tile_counts([1, 256], 256, orc.MASK_ANCHOR) == (3, 3)
    # two documents split exactly at token 128: the (1,0) tile is live only
    # through the anchor column
    assert orc.tile_counts([1, 128, 256], 256, orc.MASK_ANCHOR) == (3, 3)
    assert orc.tile_counts([1, 128, 256], 256, orc.MASK_INTRA_DOC) == (2, 3)
    # ragged tail: T = 300 -> 3 tiles per side, 6 causal tiles
    assert orc.tile_counts([1, 300], 300, orc.MASK_CAUSAL) == (6, 6)


# --------------------------------------------------------------------------- RoPE

def _rotate_complex(x, pos, base, inverse=False):
    """Eq. 6 written as complex multiplication z_p * exp(i pos theta_p)."""
    x = np.asarray(x, np.float64)
    d = x.shape[-1]
    z = x[..., 0::2] + 1j * x[..., 1::2]
    theta = np.array([base ** (-(2.0 * p) / d) for p in range(d // 2)])
    ph = np.exp((-1j if inverse else 1j) * np.outer(pos, theta))[:, None, :]
    w = z * ph
    out = np.empty_like(x)
    out[..., 0::2], out[..., 1::2] = w.real, w.imag
    return out


def test_rope_literal_values():
    # d = 4, base = 10000: theta = [1, 10000^-0.5 = 0.01]
    assert np.allclose(orc.rope_theta(4, 1e4), [1.0, 0.01], rtol=0, atol=1e-15)
    x = np.array([[[1.0, 0.0, 0.0, 2.0]]])
    y = orc.rotate(x, [1], 1e4)
    assert np.allclose(y[0, 0], [math.cos(1), math.sin(1), -2 * math.sin(0.01), 2 * math.cos(0.01)],
                       atol=1e-15)


def test_rope_matches_complex_form_and_properties():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((50, 3, 64))
    pos = rng.integers(0, 200000, size=50)
    y = orc.rotate(x, pos, 5e6)
    assert np.allclose(y, _rotate_complex(x, pos, 5e6), atol=1e-11)
    assert np.allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), atol=1e-12)
    assert np.allclose(orc.rotate(y, pos, 5e6, inverse=True), x, atol=1e-11)
    assert np.array_equal(orc.rotate(x, np.zeros(50, int), 1e4), x)      # R_0 = I
    # relative property: (R_i q).(R_j k) = q.(R_{j-i} k)  (Eq. 3 / Eq. 7)
    i, j = rng.integers(0, 5000, 50), rng.integers(0, 5000, 50)
    q, k = x, rng.standard_normal((50, 3, 64))
    lhs = (orc.rotate(q, i, 1e4) * orc.rotate(k, j, 1e4)).sum(-1)
    rhs = (q * orc.rotate(k, j - i, 1e4)).sum(-1)
    assert np.allclose(lhs, rhs, atol=1e-9)


def test_rope_half_layout_is_permuted_adjacent():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((20, 2, 32))
    pos = np.arange(20) * 7
    perm = np.empty(32, int)
    perm[0::2], perm[1::2] = np.arange(16), np.arange(16, 32)
    # interleaving the two halves turns the half-split layout into Eq. 6
    yh = orc.rotate(x, pos, 1e4, orc.ROPE_HALF)
    ya = orc.rotate(x[..., perm], pos, 1e4, orc.ROPE_ADJACENT)
    assert np.allclose(yh[..., perm], ya, atol=1e-12)


# --------------------------------------------------------------------------- forward

def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def test_single_document_equals_causal_attention():
    # one document filling the packing: AnchorAttention = causal attention with
    # positions 0..T-1 (an independent library implementation, fp64)
    T, H, d = 97, 2, 16
    q, k, v = _rand((T, H, d), 1), _rand((T, H, d), 2), _rand((T, H, d), 3)
    prob = orc.Problem([1, T], T, H, H, d, 1e4)
    O, _ = orc.forward(prob, q, k, v)
    qr = torch.from_numpy(_rotate_complex(q, np.arange(T), 1e4)).permute(1, 0, 2)
    kr = torch.from_numpy(_rotate_complex(k, np.arange(T), 1e4)).permute(1, 0, 2)
    ref = torch.nn.functional.scaled_dot_product_attention(
        qr, kr, torch.from_numpy(v).permute(1, 0, 2), is_causal=True)
    assert np.allclose(O, ref.permute(1, 0, 2).numpy(), atol=1e-12)


def test_packed_equals_separate_documents():
    T, H, d = 120, 2, 8
    cu = [1, 30, 31, 77, 120]
    q, k, v = _rand((T, H, d), 5), _rand((T, H, d), 6), _rand((T, H, d), 7)
    O, L = orc.forward(orc.Problem(cu, T, H, H, d), q, k, v)
    for a, b in zip(cu[:-1], cu[1:]):
        idx = np.r_[0, a:b]
        sub = orc.Problem([1, b - a + 1], b - a + 1, H, H, d)
        Os, Ls = orc.forward(sub, q[idx], k[idx], v[idx])
        assert np.allclose(O[a:b], Os[1:], atol=1e-12)
        assert np.allclose(L[:, a:b], Ls[:, 1:], atol=1e-12)


def test_anchor_row_and_first_token_closed_forms():
    T, H, d = 40, 1, 8
    cu = [1, 10, 25, 40]
    q, k, v = _rand((T, H, d), 8), _rand((T, H, d), 9), _rand((T, H, d), 10)
    prob = orc.Problem(cu, T, H, H, d)
    O, L = orc.forward(prob, q, k, v)
    qr = _rotate_complex(q, prob.pos, 1e4)
    kr = _rotate_complex(k, prob.pos, 1e4)
    # anchor sees only itself
    assert np.allclose(O[0, 0], v[0, 0], atol=1e-14)
    assert math.isclose(L[0, 0], (qr[0, 0] @ kr[0, 0]) / math.sqrt(d), abs_tol=1e-12)
    # a document's first token sees {anchor, itself}: a two-key softmax
    for i in cu[:-1]:
        a = qr[i, 0] @ kr[0, 0] / math.sqrt(d)
        b = qr[i, 0] @ kr[i, 0] / math.sqrt(d)
        w = 1.0 / (1.0 + math.exp(b - a))
        assert np.allclose(O[i, 0], w * v[0, 0] + (1 - w) * v[i, 0], atol=1e-12)
        assert math.isclose(L[0, i], max(a, b) + math.log1p(math.exp(-abs(a - b))), abs_tol=1e-12)


@pytest.mark.parametrize("mode", [orc.MASK_ANCHOR, orc.MASK_INTRA_DOC, orc.MASK_CAUSAL])
@pytest.mark.parametrize("pos_mode", [orc.POS_RESET, orc.POS_CONTINUOUS])
def test_shift_invariance_fp64(mode, pos_mode):
    # Eq. 3: a constant shift Delta of every position leaves attention unchanged
    T, H, d = 64, 2, 32
    cu = [1, 20, 64]
    q, k, v = _rand((T, H, d), 11), _rand((T, H, d), 12), _rand((T, H, d), 13)
    O0, L0 = orc.forward(orc.Problem(cu, T, H, H, d, 5e5, mode, pos_mode), q, k, v)
    O1, L1 = orc.forward(orc.Problem(cu, T, H, H, d, 5e5, mode, pos_mode, pos_shift=1000), q, k, v)
    assert np.allclose(O0, O1, atol=1e-10) and np.allclose(L0, L1, atol=1e-10)


def test_reset_identical_documents_identical_outputs():
    # two identical documents: with reset IDs their rows match exactly in
    # structure (and to rounding); with continuous IDs the anchor logit
    # depends on the absolute position, so they differ
    d, n = 16, 12
    T = 1 + 2 * n
    base = _rand((n, 1, d), 14)
    q = np.concatenate([_rand((1, 1, d), 15), base, base])
    k = np.concatenate([_rand((1, 1, d), 16), base[::-1], base[::-1]])
    v = np.concatenate([_rand((1, 1, d), 17), base * 2, base * 2])
    cu = [1, 1 + n, T]
    Or, _ = orc.forward(orc.Problem(cu, T, 1, 1, d, 1e4, orc.MASK_ANCHOR, orc.POS_RESET), q, k, v)
    Oc, _ = orc.forward(orc.Problem(cu, T, 1, 1, d, 1e4, orc.MASK_ANCHOR, orc.POS_CONTINUOUS), q, k, v)
    assert np.allclose(Or[1:1 + n], Or[1 + n:], atol=1e-12)
    assert np.abs(Oc[1:1 + n] - Oc[1 + n:]).max() > 1e-3


def test_gqa_equals_repeated_kv_heads():
    T, Hq, Hkv, d = 50, 4, 2, 8
    cu = [1, 20, 50]
    q, k, v, do = _rand((T, Hq, d), 18), _rand((T, Hkv, d), 19), _rand((T, Hkv, d), 20), _rand((T, Hq, d), 21)
    g = orc.Problem(cu, T, Hq, Hkv, d)
    m = orc.Problem(cu, T, Hq, Hq, d)
    kk, vv = np.repeat(k, 2, axis=1), np.repeat(v, 2, axis=1)
    Og, Lg = orc.forward(g, q, k, v)
    Om, Lm = orc.forward(m, q, kk, vv)
    assert np.allclose(Og, Om, atol=1e-13) and np.allclose(Lg, Lm, atol=1e-13)
    dqg, dkg, dvg = orc.backward(g, q, k, v, do)
    dqm, dkm, dvm = orc.backward(m, q, kk, vv, do)
    assert np.allclose(dqg, dqm, atol=1e-12)
    assert np.allclose(dkg, dkm.reshape(T, Hkv, 2, d).sum(2), atol=1e-12)
    assert np.allclose(dvg, dvm.reshape(T, Hkv, 2, d).sum(2), atol=1e-12)


# --------------------------------------------------------------------------- backward

def _torch_attention(q, k, v, mask, pos, base, scale):
    """Independent formulation: complex-number RoPE + masked softmax, torch fp64."""
    d = q.shape[-1]
    theta = base ** (-torch.arange(0, d, 2, dtype=torch.float64) / d)
    ph = torch.polar(torch.ones(len(pos), d // 2, dtype=torch.float64),
                     torch.tensor(pos, dtype=torch.float64)[:, None] * theta[None, :])[:, None, :]

    def rot(x):
        z = torch.view_as_complex(x.reshape(*x.shape[:-1], d // 2, 2).contiguous())
        return torch.view_as_real(z * ph).reshape(x.shape)

    qr, kr = rot(q), rot(k)
    s = torch.einsum("ihc,jhc->hij", qr, kr) * scale
    s = s.masked_fill(~torch.from_numpy(mask)[None], float("-inf"))
    return torch.einsum("hij,jhc->ihc", torch.softmax(s, -1), v)


@pytest.mark.parametrize("mode,pos_mode", [(orc.MASK_ANCHOR, orc.POS_RESET),
                                           (orc.MASK_ANCHOR, orc.POS_CONTINUOUS),
                                           (orc.MASK_INTRA_DOC, orc.POS_RESET),
                                           (orc.MASK_CAUSAL, orc.POS_RESET)])
def test_backward_matches_autograd(mode, pos_mode):
    T, H, d = 45, 2, 16
    cu = [1, 9, 10, 30, 45]
    q, k, v, do = (_rand((T, H, d), s) for s in (22, 23, 24, 25))
    prob = orc.Problem(cu, T, H, H, d, 1e4, mode, pos_mode)
    dq, dk, dv = orc.backward(prob, q, k, v, do)
    tq, tk, tv = (torch.tensor(a, requires_grad=True) for a in (q, k, v))
    mask = orc.attention_mask(cu, T, mode)
    out = _torch_attention(tq, tk, tv, mask, prob.pos, 1e4, 1 / math.sqrt(d))
    out.backward(torch.from_numpy(do))
    assert np.allclose(dq, tq.grad.numpy(), atol=1e-11)
    assert np.allclose(dk, tk.grad.numpy(), atol=1e-11)
    assert np.allclose(dv, tv.grad.numpy(), atol=1e-11)
    O, _ = orc.forward(prob, q, k, v)
    assert np.allclose(O, out.detach().numpy(), atol=1e-12)


def test_backward_finite_differences():
    T, H, d = 12, 1, 4
    cu = [1, 5, 12]
    q, k, v, do = (_rand((T, H, d), s) for s in (26, 27, 28, 29))
    prob = orc.Problem(cu, T, H, H, d, 100.0)
    dq, dk, dv = orc.backward(prob, q, k, v, do)

    def f(q_, k_, v_):
        return float((orc.forward(prob, q_, k_, v_)[0] * do).sum())

    h = 1e-6
    for name, arr, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for idx in [(0, 0, 1), (3, 0, 2), (5, 0, 0), (11, 0, 3)]:
            p, m = arr.copy(), arr.copy()
            p[idx] += h
            m[idx] -= h
            args_p = {"q": (p, k, v), "k": (q, p, v), "v": (q, k, p)}[name]
            args_m = {"q": (m, k, v), "k": (q, m, v), "v": (q, k, m)}[name]
            num = (f(*args_p) - f(*args_m)) / (2 * h)
            assert abs(num - grad[idx]) <= 1e-6 * max(1.0, abs(num)), (name, idx)


def test_backward_rows_subset_is_document_separable():
    # restricting to one document's rows gives that document's full key
    # gradients (no other rows see those keys)
    T, H, d = 60, 1, 8
    cu = [1, 25, 60]
    q, k, v, do = (_rand((T, H, d), s) for s in (30, 31, 32, 33))
    prob = orc.Problem(cu, T, H, H, d)
    dq, dk, dv = orc.backward(prob, q, k, v, do)
    rows = np.arange(25, 60)
    dq2, dk2, dv2 = orc.backward(prob, q, k, v, do, rows=rows)
    assert np.allclose(dq[rows], dq2[rows], atol=1e-12)
    assert np.allclose(dk[25:], dk2[25:], atol=1e-12)
    assert np.allclose(dv[25:], dv2[25:], atol=1e-12)


# --------------------------------------------------------------------------- explicit frequency tables
def test_rotate_explicit_theta_equals_base_formula():
    rng = np.random.default_rng(21)
    x = rng.standard_normal((40, 2, 16))
    pos = rng.integers(0, 5000, 40)
    a = orc.rotate(x, pos, 5e5)
    b = orc.rotate(x, pos, 123.0, theta=orc.rope_theta(16, 5e5))   # base ignored with a table
    assert np.array_equal(a, b)


def test_rotate_zero_theta_is_identity():
    rng = np.random.default_rng(22)
    x = rng.standard_normal((30, 1, 8))
    assert np.array_equal(orc.rotate(x, np.arange(30) * 97, 1e4, theta=np.zeros(4)), x)


def test_rotate_custom_theta_complex_form():
    # each adjacent pair as a complex number times exp(i * pos * theta_p)
    rng = np.random.default_rng(23)
    theta = rng.uniform(1e-5, 2.0, 8)
    x = rng.standard_normal((25, 3, 16))
    pos = rng.integers(0, 100000, 25)
    z = (x[..., 0::2] + 1j * x[..., 1::2]) * np.exp(1j * pos[:, None, None] * theta[None, None, :])
    y = orc.rotate(x, pos, 1e4, theta=theta)
    assert np.allclose(y[..., 0::2], z.real, atol=1e-12) and np.allclose(y[..., 1::2], z.imag, atol=1e-12)


def test_custom_theta_keeps_shift_invariance():
    # Eq. 3 holds for any frequency table: shifting every position leaves the output unchanged
    rng = np.random.default_rng(24)
    theta = rng.uniform(1e-6, 1.0, 8)
    T, cu = 150, [1, 60, 150]
    q, k, v = (rng.standard_normal((T, 2, 16)) for _ in range(3))
    mk = lambda s: orc.Problem(cu, T, 2, 2, 16, 1e4, orc.MASK_ANCHOR, orc.POS_RESET, pos_shift=s, theta=theta)
    O0, L0 = orc.forward(mk(0), q, k, v)
    O1, L1 = orc.forward(mk(777), q, k, v)
    assert np.allclose(O0, O1, atol=1e-10) and np.allclose(L0, L1, atol=1e-10)


# --------------------------------------------------------------------------- documents given per token
def test_interleaved_mask_and_positions_by_hand():
    # tokens: anchor, d1, d2, d1, d2, d2, d1 (chunks of two documents interleaved)
    doc = [0, 1, 2, 1, 2, 2, 1]
    p = orc.Problem(None, 7, 1, 1, 4, 1e4, orc.MASK_ANCHOR, orc.POS_RESET, doc_of_token=doc)
    m = orc.mask_rows(np.arange(7), p.doc, orc.MASK_ANCHOR)
    want = [[0], [0, 1], [0, 2], [0, 1, 3], [0, 2, 4], [0, 2, 4, 5], [0, 1, 3, 6]]
    for i, js in enumerate(want):
        assert sorted(np.nonzero(m[i])[0].tolist()) == js, i
    assert p.pos.tolist() == [0, 1, 1, 2, 2, 3, 3]
    pc = orc.Problem(None, 7, 1, 1, 4, 1e4, orc.MASK_ANCHOR, orc.POS_CONTINUOUS, doc_of_token=doc, pos_shift=5)
    assert pc.pos.tolist() == [5, 6, 7, 8, 9, 10, 11]
    pi = orc.Problem(None, 7, 1, 1, 4, 1e4, orc.MASK_INTRA_DOC, orc.POS_RESET, doc_of_token=doc)
    mi = orc.mask_rows(np.arange(7), pi.doc, orc.MASK_INTRA_DOC)
    assert sorted(np.nonzero(mi[6])[0].tolist()) == [1, 3, 6] and np.nonzero(mi[0])[0].tolist() == [0]


def test_contiguous_doc_map_equals_cu_path():
    cu, T = [1, 30, 31, 90, 128], 128
    doc = np.zeros(T, int)
    for k in range(1, len(cu)):
        doc[cu[k - 1]:cu[k]] = k
    rng = np.random.default_rng(25)
    q, k, v = (rng.standard_normal((T, 2, 16)) for _ in range(3))
    for pos in (orc.POS_RESET, orc.POS_CONTINUOUS):
        a = orc.Problem(cu, T, 2, 2, 16, 1e4, orc.MASK_ANCHOR, pos)
        b = orc.Problem(None, T, 2, 2, 16, 1e4, orc.MASK_ANCHOR, pos, doc_of_token=doc)
        assert np.array_equal(a.doc, b.doc) and np.array_equal(a.pos, b.pos)
        Oa, La = orc.forward(a, q, k, v)
        Ob, Lb = orc.forward(b, q, k, v)
        assert np.array_equal(Oa, Ob) and np.array_equal(La, Lb)


def test_interleaved_equals_grouped_layout():
    # grouping a document's tokens (order kept) changes neither what a token
    # sees nor its RESET position: outputs move with the tokens
    from aa_synth import interleaved_chunks
    rng = np.random.default_rng(26)
    doc = interleaved_chunks([40, 25, 60], 4, rng)
    T = doc.size
    perm = np.concatenate([[0]] + [np.nonzero(doc == d)[0] for d in (1, 2, 3)])
    cu = np.concatenate([[1], 1 + np.cumsum([40, 25, 60])])
    q, k, v, do = (rng.standard_normal((T, 2, 16)) for _ in range(4))
    a = orc.Problem(None, T, 2, 1, 16, 1e4, orc.MASK_ANCHOR, orc.POS_RESET, doc_of_token=doc)
    b = orc.Problem(cu, T, 2, 1, 16, 1e4, orc.MASK_ANCHOR, orc.POS_RESET)
    Oa, La = orc.forward(a, q, k[:, :1], v[:, :1])
    Ob, Lb = orc.forward(b, q[perm], k[perm, :1], v[perm, :1])
    assert np.allclose(Oa[perm], Ob, atol=1e-12) and np.allclose(La[:, perm], Lb, atol=1e-12)
    ga = orc.backward(a, q, k[:, :1], v[:, :1], do)
    gb = orc.backward(b, q[perm], k[perm, :1], v[perm, :1], do[perm])
    for x, y in zip(ga, gb):
        assert np.allclose(x[perm], y, atol=1e-10)


def test_batched_rows_equal_one_concatenated_packing():
    # the anchor attends only to itself, so every row of a batch holds the same
    # anchor state: B packed rows = their documents concatenated after one
    # shared anchor (RESET positions), outputs per document unchanged and the
    # anchor's dk / dv summed over the rows
    rng = np.random.default_rng(27)
    rows = [[1, 40, 90], [1, 25, 30, 70]]          # cu_doclens of two rows
    Ts = [c[-1] for c in rows]
    a_q, a_k, a_v = (rng.standard_normal((1, 2, 16)) for _ in range(3))
    per = []
    for cu, T in zip(rows, Ts):
        q, k, v, do = (rng.standard_normal((T, 2, 16)) for _ in range(4))
        q[0], k[0], v[0] = a_q[0], a_k[0], a_v[0]
        per.append((cu, T, q, k, v, do))
    # concatenation: anchor, row 1's documents, row 2's documents
    cat = lambda i: np.concatenate([per[0][i][:1]] + [p[i][1:] for p in per])
    q, k, v, do = (cat(i) for i in (2, 3, 4, 5))
    do[0] = per[0][5][0] + per[1][5][0]            # the shared anchor row's upstream gradient
    T = 1 + sum(t - 1 for t in Ts)
    cu = np.concatenate([[1]] + [np.asarray(per[0][0][1:])] + [np.asarray(per[1][0][1:]) + Ts[0] - 1])
    big = orc.Problem(cu, T, 2, 2, 16, 1e4, orc.MASK_ANCHOR, orc.POS_RESET)
    O, L = orc.forward(big, q, k, v)
    dq, dk, dv = orc.backward(big, q, k, v, do)
    off = 1
    dk0 = np.zeros_like(dk[0]); dv0 = np.zeros_like(dv[0])
    for cu_r, T_r, qr, kr, vr, dor in per:
        small = orc.Problem(cu_r, T_r, 2, 2, 16, 1e4, orc.MASK_ANCHOR, orc.POS_RESET)
        Or, Lr = orc.forward(small, qr, kr, vr)
        gq, gk, gv = orc.backward(small, qr, kr, vr, dor)
        sl = slice(off, off + T_r - 1)
        assert np.allclose(O[sl], Or[1:], atol=1e-12) and np.allclose(L[:, sl], Lr[:, 1:], atol=1e-12)
        assert np.allclose(dq[sl], gq[1:], atol=1e-10) and np.allclose(dk[sl], gk[1:], atol=1e-10)
        assert np.allclose(dv[sl], gv[1:], atol=1e-10)
        assert np.allclose(O[0], Or[0], atol=1e-12)                 # every row's anchor output is v_0
        dk0 += gk[0]; dv0 += gv[0]
        off += T_r - 1
    assert np.allclose(dk[0], dk0, atol=1e-10) and np.allclose(dv[0], dv0, atol=1e-10)
