"""fa_back_noalloc() against fa_back(): same results through the C ABI, two calls in a row.

fa_back_noalloc() serves callers that cannot allocate device memory (pool-owning graph
executors that give an operator no scratch pointer, services that allocate nothing after
set-up) from the library's static device scratch.  The two problems differ in shape, so a
second call that read stale scratch from the first would show up here.
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


def _outputs(p):
    return {"dQ": torch.empty((p.N, p.H, p.D), device="cuda"), "dK": torch.empty((p.M, p.Hkv, p.D), device="cuda"),
            "dV": torch.empty((p.M, p.Hkv, p.Dv), device="cuda"), "lse": torch.empty((p.N, p.H), device="cuda"),
            "delta": torch.empty((p.N, p.H), device="cuda")}


def _noalloc(fb, p, t):
    out = _outputs(p)
    mask = t["mask"].data_ptr() if t["mask"] is not None else None
    rc = fb.fa_back_noalloc(t["q"].data_ptr(), t["k"].data_ptr(), p.k_type, t["v"].data_ptr(), p.v_type, mask,
                            p.mask_heads, t["dO"].data_ptr(), p.scale, p.N, p.M, p.H, p.Hkv, p.D, p.Dv, p.causal,
                            out["dQ"].data_ptr(), out["dK"].data_ptr(), out["dV"].data_ptr(), out["lse"].data_ptr(),
                            out["delta"].data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert fb.STATUS[rc] == "FA_OK", fb.fa_back_status_string(rc)
    torch.cuda.synchronize()
    assert fb.fa_back_get_error() == 0
    return {k: v.cpu().numpy() for k, v in out.items()}


def _with_workspace(fb, p, t):
    out = fb.backward(t["q"], t["k"], p.k_type, t["v"], p.v_type, t["dO"], H=p.H, Hkv=p.Hkv, D=p.D, Dv=p.Dv, M=p.M,
                      scale=p.scale, causal=p.causal, mask=t["mask"], mask_heads=p.mask_heads)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


def test_noalloc_matches_fa_back_on_two_calls_in_a_row(fb):
    for cfg in ("3", "1"):
        p = synth.from_config(cfg)
        t = synth.device.to_torch(p, "cuda")
        ref = _with_workspace(fb, p, t)
        got = _noalloc(fb, p, t)
        check_components(got, ref, NMSE_TOL)


def test_noalloc_rejects_problems_beyond_its_scratch(fb):
    N, M, H, Hkv, D = 16384, 262144, 32, 8, 256
    assert fb.fa_back_workspace_size_min(N, M, H, Hkv, D, D) > fb._native.NOALLOC_SCRATCH_BYTES
    rc = fb.fa_back_noalloc(0x1000, 0x2000, 2, 0x3000, 2, None, 0, 0x4000, 0.0625, N, M, H, Hkv, D, D, 1,
                            0x5000, 0x6000, 0x7000, 0x8000, 0x9000, None)
    assert fb.STATUS[rc] == "FA_ERR_WORKSPACE"


@pytest.mark.slow
def test_noalloc_long_context_within_the_scratch(fb):
    """The long-context shape: the plan takes fewer key splits so its workspace fits the
    64 MiB scratch; results agree with fa_back() (whose plan splits more) within tolerance."""
    p = synth.from_config("4")
    assert fb.fa_back_workspace_size(p.N, p.M, p.H, p.Hkv, p.D, p.Dv) > (64 << 20)
    t = synth.device.to_torch(p, "cuda")
    ref = _with_workspace(fb, p, t)
    got = _noalloc(fb, p, t)
    check_components(got, ref, NMSE_TOL)


def test_noalloc_middle_plan_parity(fb):
    """A shape whose stored dS (2 N H M bytes) exceeds the 64 MiB scratch while the binary16 K/V
    copies fit: the plan recomputes dS in a dQ pass (k_rows_dq).  Sampled rows and keys against
    the oracle."""
    import oracle
    p = synth.make_problem("middle", N=256, M=17000, H=8, Hkv=2, D=128, Dv=128, k_type="q8_0", v_type="q8_0",
                           causal=True, seed=77)
    assert 2 * p.N * p.H * p.M > fb._native.NOALLOC_SCRATCH_BYTES
    t = synth.device.to_torch(p, "cuda")
    fb.fa_back_profile(True)
    got = _noalloc(fb, p, t)
    fb.fa_back_profile(False)
    launched = {k for k, v in fb.fa_back_profile_read().items() if v[1] > 0}
    assert "k_rows_dq" in launched and "k_dq_gemm" not in launched, launched
    rows = synth.sample_indices(78, synth.gen.S_SAMPLE, p.N, 48)
    keys = synth.sample_indices(78, synth.gen.S_SAMPLE + 1, p.M, 128)
    ref = oracle.fa_back(p, dq_rows=rows, dkv_keys=keys)
    sub = {"lse": got["lse"], "delta": got["delta"], "dQ": got["dQ"][rows], "dK": got["dK"][keys],
           "dV": got["dV"][keys]}
    print(check_components(sub, ref, NMSE_TOL))
