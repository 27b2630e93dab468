"""GPU: the sharded step's kernel path. Every rank's local packings (its
documents and kv-head ranges, each with its own copy of the anchor) run
through the library's kernels; here the ranks of a 4-way split run one after
another in one process (nothing on the GPU waits across ranks: the exchanges
are host-level collectives, replaced by a plain sum), and the reassembled
outputs and anchor gradients must meet the fp64 oracle on the whole packing
at the parity tolerances ("When Precision Meets Position", architecture page,
§3.4 "AnchorAttention", "Mask construction")."""
import numpy as np
import pytest
import torch

import oracle as orc
from gpu_common import REL_L2, check_forward, f64, inputs, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def aa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import packed_sequence_rope_gb300 as pkg
    return pkg


def test_four_way_split_through_the_kernels(aa):
    from packed_sequence_rope_gb300 import shard
    cu = [1, 1501, 1641, 1900, 2300, 2301, 3000]   # the 1500-token document exceeds a rank's share
    T, Hq, Hkv, D, base, W = 3000, 4, 2, 128, 5e5, 4
    q, k, v, do = inputs(T, Hq, Hkv, D, seed=61)
    _, pieces, cost = shard.local_packings(cu, Hq, Hkv, W, 0)
    assert any(p[3] - p[2] < Hkv for p in pieces)
    compute = shard.kernel_compute(base, orc.MASK_ANCHOR)
    parts = [shard.run_local(q, k, v, do, cu, r, W, compute) for r in range(W)]
    torch.cuda.synchronize()
    o, lse, dq, dk, dv = (sum(p[0][i] for p in parts) for i in range(5))
    dk[0] = sum(p[1][0] for p in parts).to(dk.dtype)
    dv[0] = sum(p[1][1] for p in parts).to(dv.dtype)
    prob = orc.Problem(cu, T, Hq, Hkv, D, base)
    O, L = orc.forward(prob, q.cpu(), k.cpu(), v.cpu())
    check_forward(o, lse, O, L, tag="sharded")
    gq, gk, gv = orc.backward(prob, q.cpu(), k.cpu(), v.cpu(), do.cpu())
    for nm, got, ref in (("dq", dq, gq), ("dk", dk, gk), ("dv", dv, gv), ("dk_0", dk[0], gk[0]),
                         ("dv_0", dv[0], gv[0])):
        e = rel_l2(got, ref)
        assert e <= REL_L2, f"sharded {nm} rel-L2 {e:.3e}"
