"""The statistics pass against numpy over the oracle's decoded inputs.

That pass finds max |x| and the largest squared row norm of Q, dO, K^ and V^. The operand scales
(powers of two), the dS multiplier's bound and the V shift's binade all follow from these
numbers, so they are checked directly rather than only through the gradients.

The library keeps its statistics record at the start of the workspace. The record holds eleven
binary32 scales and factors, then max |x| of Q, dO, K^ and V^, then their largest squared row
norms. This test reads the record back after one call. Max |x| must match exactly, because every
decoded value (code times d, or the stored value) is exact in binary32. Each squared row norm is
a binary32 sum of D positive terms, eight per lane and then a tree over the lanes, so it must
match within a relative 1e-5.
"""
import numpy as np
import pytest

import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

REC_AMAX, REC_NORM2 = 11, 15  # float offsets of the two arrays of four in the record


@pytest.fixture(scope="module")
def fb():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import flash_attention_backward_gb300 as m
    from flash_attention_backward_gb300 import build
    build.build()
    return m


def set_min_code(p):
    """Give the q8_0 K block with the largest |d| the code -128 in its first slot. That block then
    holds the largest |x| of K^, 128 |d|, which only a decoder that reads -128 as 128 in size
    reports."""
    raw = p.k.reshape(-1, 34)
    d = np.abs(raw[:, :2].copy().view(np.float16).astype(np.float64).ravel())
    b = int(np.argmax(d))
    raw[b, 2] = 0x80
    p.k = raw.reshape(p.k.shape)
    return p


def expected(p, with_dO=True):
    import oracle
    kd = oracle.dequant(p.k, p.k_type, p.D)
    vd = oracle.dequant(p.v, p.v_type, p.Dv)
    xs = [p.q.astype(np.float64), p.dO.astype(np.float64) if with_dO else None, kd, vd]
    amax = [0.0 if x is None else float(np.abs(x).max(initial=0.0)) for x in xs]
    norm2 = [0.0 if x is None else float((x * x).sum(-1).max(initial=0.0)) for x in xs]
    return np.array(amax), np.array(norm2)


def check_record(ws, amax_e, norm2_e):
    rec = ws[:256].cpu().numpy().view(np.float32)
    amax, norm2 = rec[REC_AMAX:REC_AMAX + 4], rec[REC_NORM2:REC_NORM2 + 4]
    assert np.array_equal(amax, amax_e.astype(np.float32)), (amax, amax_e)
    np.testing.assert_allclose(norm2, norm2_e, rtol=1e-5, atol=0.0)


CASES = {
    "q8_d256_min_code": dict(N=40, M=1000, H=8, Hkv=2, D=256, Dv=256, k_type="q8_0", v_type="q8_0"),
    "q4_d128_odd_m": dict(N=33, M=777, H=6, Hkv=3, D=128, Dv=128, k_type="q4_0", v_type="q4_0", causal=True),
    "f16_f32_d64": dict(N=17, M=301, H=4, Hkv=1, D=64, Dv=64, k_type="f16", v_type="f32"),
    "q8_q4_row_range": dict(N=64, M=515, H=4, Hkv=2, D=256, Dv=128, k_type="q8_0", v_type="q4_0",
                            row_decades=2.0),
    "f32_q8_d128_dv256": dict(N=9, M=2049, H=2, Hkv=2, D=128, Dv=256, k_type="f32", v_type="q8_0"),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_statistics_record(fb, name):
    p = synth.make_problem(name, seed=5200 + sorted(CASES).index(name), **CASES[name])
    if name == "q8_d256_min_code":
        p = set_min_code(p)
    t = synth.device.to_torch(p, "cuda")
    W = fb.Workspace("cuda")
    fb.backward(t["q"], t["k"], p.k_type, t["v"], p.v_type, t["dO"], H=p.H, Hkv=p.Hkv, D=p.D, Dv=p.Dv, M=p.M,
                scale=p.scale, causal=p.causal, mask=t["mask"], mask_heads=p.mask_heads, workspace=W)
    torch.cuda.synchronize()
    assert fb.fa_back_get_error() == 0
    check_record(W.buf, *expected(p))


def test_statistics_record_of_the_forward(fb):
    """The forward has no dO: its entries stay 0, the others are as in the backward."""
    p = synth.make_problem("fwd_stats", seed=5210, **CASES["q8_q4_row_range"])
    t = synth.device.to_torch(p, "cuda")
    W = fb.Workspace("cuda")
    fb.forward(t["q"], t["k"], p.k_type, t["v"], p.v_type, H=p.H, Hkv=p.Hkv, D=p.D, Dv=p.Dv, M=p.M,
               scale=p.scale, causal=p.causal, mask=t["mask"], mask_heads=p.mask_heads, workspace=W)
    torch.cuda.synchronize()
    assert fb.fa_back_get_error() == 0
    check_record(W.buf, *expected(p, with_dO=False))
