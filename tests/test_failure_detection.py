"""Failure detection without a GPU fault.

GPU: a kernel waits on a barrier that nothing arrives on; the bounded wait runs
out, the error word is set, aa_check_device_error reports AA_ERR_TIMEOUT and
the context stays usable for the next call. Host: argument errors come back as
status codes before anything launches (see test_plan.py).
"""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def aa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import packed_sequence_rope_gb300 as pkg
    return pkg


def test_bounded_wait_reports_timeout_and_context_survives(aa):
    from gpu_common import inputs
    T, H, D = 600, 2, 128
    with aa.Plan([1, 300, 600], T, H, H, D, 1e4) as p:
        p.set_wait_limit(2_000_000)  # 2 ms
        p.selftest_bounded_wait()
        torch.cuda.synchronize()
        with pytest.raises(aa.AAError) as ei:
            p.check_device_error()
        assert ei.value.status == 5 and "900" in str(ei.value)
        p.check_device_error()  # the word was cleared
        p.set_wait_limit(2_000_000_000)
        q, k, v, do = inputs(T, H, H, D, seed=9)
        o, lse = p.fwd(q, k, v)
        torch.cuda.synchronize()
        p.check_device_error()
        assert torch.isfinite(o.float()).all()
