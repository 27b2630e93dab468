"""GPU: the hot path on a 1M-token packing, the largest size these tests run.

T = 2^20 tokens with 32 query and 32 kv heads of dimension 128: every
[T, H, D] tensor holds 2^32 elements (8 GiB in bf16), so each row past token
2^19 lies beyond 2^31 elements and every kernel's row offsets must be 64-bit;
the fp32 dQ accumulator spans 16 GiB, and CONTINUOUS positions reach
2^20 - 1, the far end of the RoPE tables. The benchmark's path (aa_fwd +
aa_bwd_from_fwd) runs on the whole packing; the fp64 oracle checks whole
documents at the start, past row 2^19 and at the end. Documents are
independent apart from the anchor ("When Precision Meets Position",
architecture page, §3.4 "AnchorAttention: The Shared Anchor Design", "Mask
construction"), and under RESET a document's positions are 1..N whatever its
place in the packing, so the oracle on [anchor + document] gives that
document's O, LSE, dq, dk and dv.

About 100 GB of device memory; the oracle side takes a few seconds.
"""
import numpy as np
import pytest
import torch

import oracle as orc
from aa_synth import Workload, make_qkv, workload_cu_doclens
from gpu_common import REL_L2, check_forward, problem, rel_l2

pytestmark = pytest.mark.gpu

MAX_1M = Workload("max_1m", 1 << 20, 32, 32, 128, 5e6, "lognormal",
                  {"median": 3000, "sigma": 1.0, "lo": 64, "hi": (1 << 20) - 1}, seed=3)
HEADS = [0, 31]


@pytest.fixture(scope="module")
def aa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import packed_sequence_rope_gb300 as pkg
    return pkg


@pytest.fixture(scope="module")
def packing(aa):
    w = MAX_1M
    cu = workload_cu_doclens(w)
    q, k, v, do = make_qkv(w, device="cuda")
    yield w, cu, q, k, v, do
    del q, k, v, do
    torch.cuda.empty_cache()


def _doc_picks(cu):
    # the first document, the one holding row 2^19 + 1 (the first rows whose
    # offsets pass 2^31 elements) and the last one
    mid = int(np.searchsorted(cu, (1 << 19) + 1, side="right")) - 1
    return sorted({0, mid, len(cu) - 2})


def _anchor_plus_doc(t, a, b, heads):
    idx = torch.cat([torch.zeros(1, dtype=torch.long, device=t.device), torch.arange(a, b, device=t.device)])
    return t[idx][:, heads].cpu()


def test_max_size_bench_path_documents(aa, packing):
    w, cu, q, k, v, do = packing
    T, D = w.total_tokens, w.head_dim
    assert T * w.num_q_heads * D == 1 << 32
    with aa.Plan(cu, T, w.num_q_heads, w.num_kv_heads, D, w.rope_base) as p:
        fws = p.alloc_fwd_workspace(q.device)
        o, lse = p.fwd(q, k, v, workspace=fws)
        dq, dk, dv = p.bwd_from_fwd(fws, v, o, lse, do)
        torch.cuda.synchronize()
        p.check_device_error()
        del fws
    heads = torch.tensor(HEADS, device=q.device)
    picks = _doc_picks(cu)
    assert int(cu[picks[-1]]) * w.num_q_heads * D > 1 << 31
    for d in picks:
        a, b = int(cu[d]), int(cu[d + 1])
        n = b - a
        qs, ks, vs, dos = (_anchor_plus_doc(x, a, b, heads) for x in (q, k, v, do))
        prob = problem([1, 1 + n], 1 + n, len(HEADS), len(HEADS), D, w.rope_base)
        O, L = orc.forward(prob, qs, ks, vs)
        check_forward(o[a:b][:, heads], lse[heads][:, a:b], O[1:], L[:, 1:], tag=f"doc {d} [{a}, {b})")
        gq, gk, gv = orc.backward(prob, qs, ks, vs, dos)
        for nm, got, ref in (("dq", dq[a:b][:, heads], gq[1:]), ("dk", dk[a:b][:, heads], gk[1:]),
                             ("dv", dv[a:b][:, heads], gv[1:])):
            e = rel_l2(got, ref)
            assert e <= REL_L2, f"doc {d} [{a}, {b}) {nm} rel-L2 {e:.3e}"


def test_max_size_continuous_positions_forward(aa, packing):
    # CONTINUOUS: positions run 0 .. 2^20 - 1 over the packing
    w, cu, q, k, v, _ = packing
    T, D = w.total_tokens, w.head_dim
    with aa.Plan(cu, T, w.num_q_heads, w.num_kv_heads, D, w.rope_base, orc.MASK_ANCHOR, orc.POS_CONTINUOUS) as p:
        o, lse = p.fwd(q, k, v)
        torch.cuda.synchronize()
        p.check_device_error()
    rng = np.random.default_rng(5)
    rows = np.unique(np.concatenate([[0, 1, T - 1], rng.integers(T - (1 << 15), T, 24), rng.integers(1, T, 8)]))
    heads = torch.tensor(HEADS, device=q.device)
    qh, kh, vh = (x[:, heads].cpu() for x in (q, k, v))
    prob = problem(cu, T, len(HEADS), len(HEADS), D, w.rope_base, orc.MASK_ANCHOR, orc.POS_CONTINUOUS)
    O, L = orc.forward(prob, qh, kh, vh, rows=rows)
    r = torch.as_tensor(rows, device=q.device)
    check_forward(o[r][:, heads], lse[heads][:, r], O, L, tag="continuous 1M")
