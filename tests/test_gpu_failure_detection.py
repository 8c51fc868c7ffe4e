"""Failure detection of the bounded waits, on the GPU and without a fault.

Every mbarrier wait in the kernels gives up after a time limit, records FA_ERR_TIMEOUT in a
device word and lets its CTA finish.  fa_back_selftest_timeout() runs that path on a barrier
that nothing completes (with a 1 ms limit); the error must reach the host once, be cleared by
reading it, and leave the context usable for a correct backward afterwards.
"""
import numpy as np
import pytest

import synth
from metrics import NMSE_TOL, check_components

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fb():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import flash_attention_backward_gb300 as m
    from flash_attention_backward_gb300 import build
    build.build()
    return m


def test_expired_wait_is_reported_and_the_context_stays_usable(fb):
    assert fb.fa_back_get_error() == 0
    assert fb.STATUS[fb.fa_back_selftest_timeout(1_000_000)] == "FA_OK"
    torch.cuda.synchronize()
    assert fb.STATUS[fb.fa_back_get_error()] == "FA_ERR_TIMEOUT"
    assert fb.fa_back_get_error() == 0  # reading clears it
    # the context is intact: a normal call still matches the oracle
    import oracle
    p = synth.from_config("0")
    t = synth.device.to_torch(p, "cuda")
    out = fb.backward(t["q"], t["k"], p.k_type, t["v"], p.v_type, t["dO"], H=p.H, Hkv=p.Hkv, D=p.D, Dv=p.Dv,
                      M=p.M, scale=p.scale, causal=p.causal)
    torch.cuda.synchronize()
    assert fb.fa_back_get_error() == 0
    check_components({k: v.cpu().numpy() for k, v in out.items()}, oracle.fa_back(p), NMSE_TOL)


def test_limit_out_of_range_is_rejected_before_launch(fb):
    assert fb.STATUS[fb.fa_back_selftest_timeout(0)] == "FA_ERR_SHAPE"
    assert fb.STATUS[fb.fa_back_selftest_timeout(3_000_000_000)] == "FA_ERR_SHAPE"
