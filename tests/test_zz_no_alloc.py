"""The backward entry point that allocates nothing (aa_bwd_static_workspace).

It exists for callers that cannot call cudaMalloc where they run the backward
pass (a plugin whose host framework owns all device memory, a loop where an
allocation would stall the device, a fixed memory budget): its scratch is a
64 MiB array the library reserves on each GPU. This test calls it twice in a
row through the C ABI and checks both results against aa_bwd with a
caller-provided workspace, at the tolerance of the other parity tests, for
plans from cu_doclens (D = 128 with GQA, D = 64 intra-document) and for a
segment plan (interleaved documents, whose grouped copies also live in the
array), and checks that a plan too large for the array is refused before any
launch.
The file is named to be collected last.
"""
import numpy as np
import pytest
import torch

import oracle as orc
from gpu_common import REL_L2, inputs, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def aa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import packed_sequence_rope_gb300 as pkg
    return pkg


def _interleaved(T, seed):
    # three documents cut into chunks and interleaved (token 0 is the anchor)
    rng = np.random.default_rng(seed)
    doc = np.concatenate([[0], rng.integers(1, 4, T - 1)]).astype(np.int32)
    return doc


CASES = [
    # name, cu_doclens, doc_of_token, T, Hq, Hkv, D, mask
    ("doclens_d128_gqa", [1, 5, 140, 141, 400, 1000, 1301], None, 1301, 4, 2, 128, orc.MASK_ANCHOR),
    ("doclens_d64_intra_doc", [1, 129, 500, 900], None, 900, 2, 1, 64, orc.MASK_INTRA_DOC),
    ("segments_d128", None, "interleaved", 700, 2, 2, 128, orc.MASK_ANCHOR),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_static_workspace_bwd_matches_workspace_bwd(aa, case):
    name, cu, doc, T, Hq, Hkv, D, mask = case
    doc = _interleaved(T, 5) if doc == "interleaved" else None
    q, k, v, do = inputs(T, Hq, Hkv, D, seed=11)
    with aa.Plan(cu, T, Hq, Hkv, D, 5e6, mask, doc_of_token=doc) as p:
        assert p.workspace_bytes() <= 64 << 20
        o, lse = p.fwd(q, k, v)
        ref = p.bwd(q, k, v, o, lse, do)
        for _ in range(2):  # two calls in a row share (and reuse) the static array
            got = p.bwd_static_workspace(q, k, v, o, lse, do)
            torch.cuda.synchronize()
            p.check_device_error()
            for nm, g, r in zip(("dq", "dk", "dv"), got, ref):
                e = rel_l2(g, r.float().cpu().numpy())
                assert e <= REL_L2, f"{name} {nm} rel-L2 {e:.3e} against aa_bwd"


def test_static_workspace_rejects_plans_beyond_its_size(aa):
    T, H, D = 65536, 32, 128  # needs ~1 GiB of scratch
    with aa.Plan([1, T], T, H, H, D, 5e6) as p:
        assert p.workspace_bytes() > 64 << 20
        x = torch.zeros(16, device="cuda", dtype=torch.bfloat16)  # never read: rejected first
        L = aa.lib()
        ptr = x.data_ptr()
        st = L.aa_bwd_static_workspace(p._h, ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, None)
        assert st == 1
        msg = L.aa_last_error().decode()
        assert "static workspace holds" in msg and "67108864" in msg
