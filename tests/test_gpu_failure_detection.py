"""Failure detection of the bounded waits, on the GPU and without a fault.

Every mbarrier wait in the kernels gives up after a time limit, records FA_ERR_TIMEOUT in a
device word and lets its CTA finish.  fa_back_selftest_timeout() runs that path on a barrier
that nothing completes (with a 1 ms limit); the error must reach the host once, be cleared by
reading it, and leave the context usable for a correct backward afterwards.

fa_back_test_wait_limit() makes the real passes give up: their waits run out after a short limit
instead of 2 s, so each CTA takes its abort path (stop issuing, wait for its own loads and
tensor-core products still in flight, free tensor memory) at whatever point its pipeline has
reached.  The call after must again match the oracle.
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


def _run(fb, p, workspace_bytes=None):
    t = synth.device.to_torch(p, "cuda")
    out = fb.backward(t["q"], t["k"], p.k_type, t["v"], p.v_type, t["dO"], H=p.H, Hkv=p.Hkv, D=p.D, Dv=p.Dv,
                      M=p.M, scale=p.scale, causal=p.causal, mask=t["mask"], mask_heads=p.mask_heads,
                      workspace_bytes=workspace_bytes)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


def _level(fb, p):
    return fb.fa_back_plan_info(p.N, p.M, p.H, p.Hkv, p.D, p.Dv,
                                fb.fa_back_workspace_size(p.N, p.M, p.H, p.Hkv, p.D, p.Dv))[1]


def test_passes_give_up_at_once_then_the_next_call_is_correct(fb):
    """Limit 0: every wait that is not complete at once gives up, in the LSE pass, the dK/dV pass
    and the dQ product (plan level 2); the timeout reaches the host once."""
    import oracle
    p = synth.from_config("0")
    assert _level(fb, p) == 2
    assert fb.fa_back_get_error() == 0
    assert fb.STATUS[fb.fa_back_test_wait_limit(0)] == "FA_OK"
    _run(fb, p)
    assert fb.STATUS[fb.fa_back_get_error()] == "FA_ERR_TIMEOUT"
    assert fb.fa_back_get_error() == 0
    got = _run(fb, p)  # the hook held for one call only
    assert fb.fa_back_get_error() == 0
    check_components(got, oracle.fa_back(p), NMSE_TOL)


@pytest.mark.parametrize("limit_ns", [2_000, 20_000])
def test_passes_give_up_mid_pipeline_then_the_next_call_is_correct(fb, limit_ns):
    """A limit of a few microseconds: some CTAs give up with loads and products in flight, others
    finish; whichever happened, the context stays usable and the next call is correct."""
    import oracle
    p = synth.from_config("1")
    assert _level(fb, p) == 2
    assert fb.fa_back_get_error() == 0
    assert fb.STATUS[fb.fa_back_test_wait_limit(limit_ns)] == "FA_OK"
    _run(fb, p)
    status = fb.STATUS[fb.fa_back_get_error()]
    print(limit_ns, status)
    assert status in ("FA_OK", "FA_ERR_TIMEOUT")
    got = _run(fb, p)
    assert fb.fa_back_get_error() == 0
    check_components(got, oracle.fa_back(p), NMSE_TOL)


def test_wait_limit_above_the_normal_one_is_rejected(fb):
    assert fb.STATUS[fb.fa_back_test_wait_limit(3_000_000_000)] == "FA_ERR_SHAPE"



def _run_forward(fb, p):
    t = synth.device.to_torch(p, "cuda")
    out = fb.forward(t["q"], t["k"], p.k_type, t["v"], p.v_type, H=p.H, Hkv=p.Hkv, D=p.D, Dv=p.Dv, M=p.M,
                     scale=p.scale, causal=p.causal, mask=t["mask"], mask_heads=p.mask_heads)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


@pytest.mark.parametrize("limit_ns", [0, 2_000, 20_000])
def test_forward_gives_up_then_the_next_call_is_correct(fb, limit_ns):
    """The one-pass forward's abort path: its producer, MMA issuer and softmax warps give up, the
    loads and products in flight are waited for before tensor memory is freed.  Limit 0 always
    times out (the issuer's first wait, for Q' in tensor memory, is never complete at once); a
    few microseconds may or may not.  The next call matches the oracle."""
    import oracle
    from metrics import nmse
    p = synth.from_config("1")
    assert fb.fa_back_get_error() == 0
    assert fb.STATUS[fb.fa_back_test_wait_limit(limit_ns)] == "FA_OK"
    _run_forward(fb, p)
    status = fb.STATUS[fb.fa_back_get_error()]
    print(limit_ns, status)
    assert status in (("FA_ERR_TIMEOUT",) if limit_ns == 0 else ("FA_OK", "FA_ERR_TIMEOUT"))
    got = _run_forward(fb, p)
    assert fb.fa_back_get_error() == 0
    ref = oracle.fa_forward(p)
    assert nmse(got["O"], ref["O"]) <= NMSE_TOL and nmse(got["lse"], ref["lse"]) <= NMSE_TOL
