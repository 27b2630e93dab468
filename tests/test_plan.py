"""Host-side tests of the C-ABI library: exports, planner metadata bit-exact
against the oracle, statistics, and synchronous argument validation.
No GPU needed: plans are built with host_only = 1."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle as orc
from aa_synth import WORKLOADS, doc_lengths, pack, workload_cu_doclens

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def aa():
    import __graft_entry__
    __graft_entry__.build()
    import packed_sequence_rope_gb300 as pkg
    return pkg


def test_library_exports_every_declared_symbol(aa):
    header = open(os.path.join(ROOT, "include", "anchorattn.h")).read()
    declared = set(re.findall(r"^\s*(?:aa_status|size_t|const char\*)\s+(aa_\w+)\s*\(", header, re.M))
    assert declared == set(aa.EXPORTS)
    L = ctypes.CDLL(aa.binding.LIB_PATH)
    for name in declared:
        assert hasattr(L, name), name


def _plan(aa, cu, T, mode=orc.MASK_ANCHOR, pos=orc.POS_RESET, shift=0, Hq=2, Hkv=1, D=128):
    return aa.Plan(cu, T, Hq, Hkv, D, 1e4, mode, pos, pos_shift=shift, host_only=True)


@pytest.mark.parametrize("mode", [orc.MASK_ANCHOR, orc.MASK_INTRA_DOC, orc.MASK_CAUSAL])
@pytest.mark.parametrize("pos", [orc.POS_RESET, orc.POS_CONTINUOUS])
@pytest.mark.parametrize("seed", [0, 1])
def test_metadata_bit_exact_vs_oracle(aa, mode, pos, seed):
    rng = np.random.default_rng(seed)
    T = 700 + 291 * seed
    cu = pack(doc_lengths("loguniform", T - 1, rng, lo=3, hi=400), T)
    shift = 17 * seed
    with _plan(aa, cu, T, mode, pos, shift) as p:
        doc, posv = p.metadata()
        assert np.array_equal(doc, orc.document_ids(cu, T, mode))
        assert np.array_equal(posv, orc.position_ids(cu, T, mode, pos, shift))
        st = p.stats()
        assert st["unmasked_pairs"] == orc.unmasked_pairs(cu, T, mode)
        live, causal = orc.tile_counts(cu, T, mode)
        assert (st["live_tiles"], st["causal_tiles"]) == (live, causal)


def test_metadata_tiny_workload(aa):
    w = WORKLOADS["tiny_256"]
    cu = workload_cu_doclens(w)
    assert list(cu) == [1, 32, 96, 192, 256]
    with aa.Plan(cu, 256, 1, 1, 64, 1e4, host_only=True) as p:
        doc, pos = p.metadata()
        assert pos[0] == 0 and pos[1] == 1 and pos[31] == 31 and pos[32] == 1 and pos[255] == 64
        assert p.stats()["unmasked_pairs"] == orc.unmasked_pairs(cu, 256, orc.MASK_ANCHOR)


def test_work_counts(aa):
    # a single document: the forward visits every causal tile per head;
    # the backward the same count per kv head and group member
    T = 1000
    with aa.Plan([1, T], T, 4, 2, 128, 1e4, host_only=True) as p:
        nt = (T + 127) // 128
        w = p.work()
        assert w["fwd_tiles"] == 4 * nt * (nt + 1) // 2
        assert w["bwd_tiles"] == 4 * nt * (nt + 1) // 2


@pytest.mark.parametrize("kwargs,cu,msg", [
    (dict(total_tokens=1), [1], "total_tokens"),
    (dict(num_q_heads=3, num_kv_heads=2), [1, 64], "Hq % Hkv"),
    (dict(head_dim=96), [1, 64], "head_dim"),
    (dict(), [0, 64], "cu_doclens\\[0\\]"),
    (dict(), [1, 63], "must equal T"),
    (dict(), [1, 30, 30, 64], "increase strictly"),
    (dict(rope_base=1.0), [1, 64], "rope_base"),
    (dict(pos_shift=-1), [1, 64], "pos_shift"),
    (dict(mask_mode=7), [1, 64], "mask_mode"),
])
def test_invalid_arguments_rejected(aa, kwargs, cu, msg):
    args = dict(total_tokens=64, num_q_heads=2, num_kv_heads=1, head_dim=128, rope_base=1e4,
                mask_mode=orc.MASK_ANCHOR, pos_shift=0)
    args.update(kwargs)
    with pytest.raises(aa.AAError, match=msg) as ei:
        aa.Plan(cu, args["total_tokens"], args["num_q_heads"], args["num_kv_heads"], args["head_dim"],
                args["rope_base"], args["mask_mode"], pos_shift=args["pos_shift"], host_only=True)
    assert ei.value.status in (1, 2)


def test_compute_on_host_only_plan_is_refused(aa):
    with _plan(aa, [1, 64], 64) as p:
        L = aa.lib()
        assert L.aa_fwd(p._h, None, None, None, None, None, None, 0, None) == 1
        assert "host_only" in L.aa_last_error().decode()
        assert L.aa_bwd_from_fwd(p._h, *([None] * 8), None, 0, None) == 1
        assert "host_only" in L.aa_last_error().decode()
        assert L.aa_check_device_error(p._h, None) == 1


@pytest.mark.parametrize("layout", [orc.ROPE_ADJACENT, orc.ROPE_NONE])
@pytest.mark.parametrize("segmented", [False, True])
def test_workspace_sizes(aa, layout, segmented):
    # Forward: rotated K then rotated Q (bf16), nothing without RoPE, then a
    # 256-byte work counter; the
    # backward from the forward's rotated operands needs no copies of them.
    T, Hq, Hkv, D = 1000, 4, 2, 128
    al = lambda n: (n + 255) // 256 * 256
    doc = np.repeat(np.arange(1, 5, dtype=np.int32), [250, 250, 250, 249]) if segmented else None
    doc = None if doc is None else np.concatenate([[0], doc]).astype(np.int32)
    cu = None if segmented else [1, 300, 700, T]
    with aa.Plan(cu, T, Hq, Hkv, D, 1e4, rope_layout=layout, host_only=True, doc_of_token=doc) as p:
        L = aa.lib()
        fwd, bwd, from_fwd = (int(L.aa_fwd_workspace_bytes(p._h)), int(L.aa_bwd_workspace_bytes(p._h)),
                              int(L.aa_bwd_from_fwd_workspace_bytes(p._h)))
    rot = al(T * Hkv * D * 2) + al(T * Hq * D * 2) if layout != orc.ROPE_NONE else 0
    tq, tk = al(T * Hq * D * 2), al(T * Hkv * D * 2)
    # segment plans: the forward keeps a grouped V (and, without RoPE, grouped
    # Q and K, which no rotation pass reads through the permutation)
    seg_fwd = (tk + (0 if layout != orc.ROPE_NONE else tq + tk)) if segmented else 0
    assert fwd == rot + 256 + seg_fwd
    # the two backward entry points differ by the rotated copies and, for
    # segment plans, by the grouped V (from the forward in aa_bwd_from_fwd)
    # and, without RoPE, grouped q and k; both hold the grouped dO
    seg_qk = (tk + (0 if layout != orc.ROPE_NONE else tq + tk)) if segmented else 0
    assert bwd - from_fwd == rot + seg_qk


def test_status_strings(aa):
    L = aa.lib()
    assert [L.aa_status_string(i).decode() for i in range(6)] == [
        "AA_OK", "AA_ERR_INVALID_ARG", "AA_ERR_UNSUPPORTED", "AA_ERR_CUDA", "AA_ERR_NO_MEMORY", "AA_ERR_TIMEOUT"]


def test_causal_mode_ignores_cu_doclens(aa):
    with aa.Plan(None, 300, 1, 1, 64, 1e4, orc.MASK_CAUSAL, host_only=True) as p:
        doc, pos = p.metadata()
        assert not doc.any() and np.array_equal(pos, np.arange(300))
        assert p.stats()["unmasked_pairs"] == 300 * 301 // 2


@pytest.mark.parametrize("name", ["llama7b_8k", "llama7b_64k"])
def test_workload_stats_vs_oracle(aa, name):
    w = WORKLOADS[name]
    cu = workload_cu_doclens(w)
    T = w.total_tokens
    with aa.Plan(cu, T, w.num_q_heads, w.num_kv_heads, w.head_dim, w.rope_base, host_only=True) as p:
        st = p.stats()
        assert st["unmasked_pairs"] == orc.unmasked_pairs(cu, T, orc.MASK_ANCHOR)
        if T <= 8192:
            assert st["live_tiles"] == orc.tile_counts(cu, T, orc.MASK_ANCHOR)[0]


def test_plan_with_theta_validation_and_metadata(aa):
    cu = [1, 40, 100]
    theta = orc.rope_theta(64, 5e5)
    with aa.Plan(cu, 100, 2, 1, 64, 1e4, host_only=True) as p0, \
            aa.Plan(cu, 100, 2, 1, 64, 1e4, host_only=True, theta=theta) as p1:
        assert all(np.array_equal(a, b) for a, b in zip(p0.metadata(), p1.metadata()))
    # the table replaces rope_base, which is then not checked
    with aa.Plan(cu, 100, 2, 1, 64, 0.5, host_only=True, theta=theta):
        pass
    for bad, msg in ((np.nan, "theta\\[3\\]"), (-1.0, "theta\\[3\\]"), (np.inf, "theta\\[3\\]")):
        t = theta.copy()
        t[3] = bad
        with pytest.raises(aa.AAError, match=msg):
            aa.Plan(cu, 100, 2, 1, 64, 1e4, host_only=True, theta=t)
    with pytest.raises(ValueError, match="head_dim / 2"):
        aa.Plan(cu, 100, 2, 1, 64, 1e4, host_only=True, theta=theta[:10])
    L = aa.lib()
    h = ctypes.c_void_p()
    cfg = aa.binding.AAConfig(100, 2, 1, 64, 1e4, 0.0, 0, orc.MASK_CAUSAL, 0, 0, 1)
    assert L.aa_plan_with_theta(ctypes.byref(cfg), None, 0, None, None, ctypes.byref(h)) == 1


@pytest.mark.parametrize("pos", [orc.POS_RESET, orc.POS_CONTINUOUS])
def test_segment_plan_metadata_vs_oracle(aa, pos):
    from aa_synth import interleaved_chunks
    doc = interleaved_chunks([300, 5, 170, 1, 90], 3, np.random.default_rng(7))
    T = doc.size
    with aa.Plan(None, T, 2, 1, 64, 1e4, orc.MASK_ANCHOR, pos, pos_shift=11, host_only=True,
                 doc_of_token=doc) as p:
        d, ps = p.metadata()
        prob = orc.Problem(None, T, 2, 1, 64, 1e4, orc.MASK_ANCHOR, pos, pos_shift=11, doc_of_token=doc)
        assert np.array_equal(d, doc) and np.array_equal(ps, prob.pos)
        assert p.stats()["unmasked_pairs"] == int(orc.mask_rows(np.arange(T), prob.doc, orc.MASK_ANCHOR).sum())


def test_segment_plan_rejects_bad_maps(aa):
    doc = np.array([0, 1, 2, 1, 2], np.int32)
    with pytest.raises(aa.AAError, match="ANCHOR or INTRA_DOC"):
        aa.Plan(None, 5, 1, 1, 64, 1e4, orc.MASK_CAUSAL, host_only=True, doc_of_token=doc)
    with pytest.raises(aa.AAError, match="doc_of_token\\[0\\]"):
        aa.Plan(None, 5, 1, 1, 64, 1e4, host_only=True, doc_of_token=np.array([1, 1, 2, 1, 2]))
    with pytest.raises(aa.AAError, match="doc_of_token\\[3\\]"):
        aa.Plan(None, 5, 1, 1, 64, 1e4, host_only=True, doc_of_token=np.array([0, 1, 2, 0, 2]))


@pytest.mark.parametrize("seed", range(12))
def test_random_packings_vs_oracle(aa, seed):
    # documents of awkward lengths (1, tile-edge, random), T from 2 tokens up:
    # metadata, pair and tile counts against the oracle, and the forward and
    # backward work lists covering the same (query tile, key tile) pairs
    rng = np.random.default_rng(100 + seed)
    T = int(rng.integers(2, 3000))
    lens, rem = [], T - 1
    while rem > 0:
        n = min(int(rng.choice([1, 2, 127, 128, 129, 255, 256, 257, int(rng.integers(1, 600))])), rem)
        lens.append(n)
        rem -= n
    cu = np.concatenate([[1], 1 + np.cumsum(lens)]).astype(np.int32)
    for mode in (orc.MASK_ANCHOR, orc.MASK_INTRA_DOC, orc.MASK_CAUSAL):
        c = None if mode == orc.MASK_CAUSAL else cu
        with aa.Plan(c, T, 4, 2, 64, 1e4, mode, host_only=True) as p:
            doc, pos = p.metadata()
            assert np.array_equal(doc, orc.document_ids(c, T, mode))
            assert np.array_equal(pos, orc.position_ids(c, T, mode, orc.POS_RESET, 0))
            st, w = p.stats(), p.work()
        assert st["unmasked_pairs"] == orc.unmasked_pairs(c, T, mode)
        assert (st["live_tiles"], st["causal_tiles"]) == orc.tile_counts(c, T, mode)
        assert w["fwd_tiles"] == w["bwd_tiles"]


@pytest.mark.parametrize("pos", [orc.POS_RESET, orc.POS_CONTINUOUS])
def test_metadata_at_one_million_tokens(aa, pos):
    # the largest packing the GPU tests run (2^20 tokens, 32 heads of 128):
    # metadata bit-exact, and the visible pairs against the closed form
    # sum_k N_k (N_k + 1) / 2 + (T - 1) + 1 (each document's causal triangle,
    # every token's anchor pair, the anchor itself), which the oracle's
    # explicit-mask count is pinned to at small sizes
    T = 1 << 20
    cu = pack(doc_lengths("lognormal", T - 1, np.random.default_rng(3), median=3000, sigma=1.0, lo=64, hi=T - 1), T)
    with aa.Plan(cu, T, 32, 32, 128, 5e6, orc.MASK_ANCHOR, pos, host_only=True) as p:
        doc, posv = p.metadata()
        assert np.array_equal(doc, orc.document_ids(cu, T, orc.MASK_ANCHOR))
        assert np.array_equal(posv, orc.position_ids(cu, T, orc.MASK_ANCHOR, pos))
        n = np.diff(cu).astype(np.int64)
        assert p.stats()["unmasked_pairs"] == int((n * (n + 1) // 2).sum()) + (T - 1) + 1
