"""Score extensions (fa_back_ext): ALiBi slopes, a logit soft cap and per-head sink logits, CUDA
path against the oracle's double-precision definition of each, on every plan level.

Tolerance as for the plain operation: NMSE <= 1e-5 per component (dQ, dK, dV, lse, delta);
lse = -inf positions agree exactly; rows without a key give delta = 0 and a zero dQ row.  dsinks,
a sum over rows whose terms can cancel, passes at NMSE <= 1e-5 or within delta's per-row error
of the sum of its terms' magnitudes (metrics.check_dsinks).
"""
import numpy as np
import pytest

import synth
from metrics import NMSE_TOL, check_components, check_dsinks, nmse

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


def run_ext(fb, p, workspace_bytes=None, profile=False):
    t = synth.device.to_torch(p, "cuda")
    dev = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to("cuda")
    if profile:
        fb.fa_back_profile(True)
    out = fb.backward(t["q"], t["k"], p.k_type, t["v"], p.v_type, t["dO"], H=p.H, Hkv=p.Hkv, D=p.D, Dv=p.Dv,
                      M=p.M, scale=p.scale, causal=p.causal, mask=t["mask"], mask_heads=p.mask_heads,
                      workspace_bytes=workspace_bytes, alibi_slopes=dev(p.alibi), softcap=p.softcap,
                      sinks=dev(p.sinks))
    torch.cuda.synchronize()
    launched = None
    if profile:
        fb.fa_back_profile(False)
        launched = {k for k, v in fb.fa_back_profile_read().items() if v[1] > 0}
    assert fb.fa_back_get_error() == 0
    got = {k: v.cpu().numpy() for k, v in out.items()}
    return (got, launched) if profile else got


def level_workspace(fb, p, level):
    """A workspace size whose plan has the given level (None if no size gives it).  Levels 1 and 3
    sit between the smallest and the fastest plan's sizes; a scan of that range finds them."""
    lo = fb.fa_back_workspace_size_min(p.N, p.M, p.H, p.Hkv, p.D, p.Dv)
    hi = fb.fa_back_workspace_size(p.N, p.M, p.H, p.Hkv, p.D, p.Dv)
    if level == 0:
        return lo
    if level == 2:
        return hi
    for k in range(401):
        w = lo + (hi - lo) * k // 400
        if fb.fa_back_plan_info(p.N, p.M, p.H, p.Hkv, p.D, p.Dv, w)[1] == level:
            return w
    return None


def ext_parity(fb, p, level=2):
    import oracle
    ws = level_workspace(fb, p, level)
    if ws is None:
        pytest.skip(f"no workspace size gives plan level {level}")
    assert fb.fa_back_plan_info(p.N, p.M, p.H, p.Hkv, p.D, p.Dv, ws)[1] == level
    ref = oracle.fa_back(p)
    got, launched = run_ext(fb, p, workspace_bytes=ws, profile=True)
    res = check_components(got, ref)
    dead = ~np.isfinite(ref["lse"])
    assert np.all(got["dQ"][dead] == 0.0)
    if p.sinks is not None:
        assert "k_sink_grad" in launched, launched
        res["dsinks"] = check_dsinks(got["dsinks"], ref, p.sinks)
    return res


# One case per extension, then all three together with the mask, GQA, the causal tail, mixed cache
# types and ragged tiles.  The soft caps are small enough (c = 1.5 and 3 against logits of about
# 1 to 3) that tanh is far from linear, so a missing cap derivative would show at once.
EXT = {
    "softcap": dict(N=64, M=700, H=8, Hkv=2, D=128, Dv=128, k_type="q8_0", v_type="q8_0", causal=True,
                    q_sigma=2.0, softcap=1.5),
    "alibi": dict(N=96, M=1100, H=8, Hkv=2, D=64, Dv=64, k_type="q4_0", v_type="q8_0", causal=True, alibi=True),
    "alibi_noncausal": dict(N=40, M=300, H=4, Hkv=4, D=128, Dv=128, k_type="f16", v_type="f16", alibi=True),
    "sinks": dict(N=80, M=900, H=8, Hkv=2, D=128, Dv=128, k_type="q8_0", v_type="q4_0", causal=True, sinks=1.0,
                  mask="random", mask_p=0.05, full_rows=3, mask_heads=8),
    "all_d256": dict(N=37, M=777, H=6, Hkv=2, D=256, Dv=256, k_type="q8_0", v_type="q8_0", causal=True,
                     alibi=True, softcap=3.0, sinks=0.5, q_sigma=1.5),
    "all_mixed": dict(N=50, M=613, H=8, Hkv=2, D=256, Dv=128, k_type="q4_0", v_type="f16", alibi=True,
                      softcap=3.0, sinks=2.0, mask="finite", mask_p=0.05, full_rows=2, mask_heads=1),
}


@pytest.mark.parametrize("level", [2, 3, 1, 0])
@pytest.mark.parametrize("name", sorted(EXT))
def test_ext_cases(fb, name, level):
    p = synth.make_problem(name, seed=7000 + sorted(EXT).index(name), **EXT[name])
    print(name, level, ext_parity(fb, p, level))


@pytest.mark.slow
def test_ext_on_the_long_context_shape_sampled(fb):
    """All three extensions at N2048/M75520/H24/Hkv4/D256 (q8_0, causal tail), plan level 3: every
    lse/delta, 48 dQ rows and 128 dK/dV keys against the oracle, and dsinks."""
    import oracle
    p = synth.from_config("4")
    p = synth.make_problem("ext_long", N=p.N, M=p.M, H=p.H, Hkv=p.Hkv, D=p.D, Dv=p.Dv, k_type="q8_0",
                           v_type="q8_0", causal=True, seed=7100, alibi=True, softcap=20.0, sinks=1.0)
    w = level_workspace(fb, p, 3)
    got = run_ext(fb, p, workspace_bytes=w)
    rows = synth.sample_indices(7101, synth.gen.S_SAMPLE, p.N, 48)
    keys = synth.sample_indices(7101, synth.gen.S_SAMPLE + 1, p.M, 128)
    ref = oracle.fa_back(p, dq_rows=rows, dkv_keys=keys)
    sub = {"lse": got["lse"], "delta": got["delta"], "dQ": got["dQ"][rows], "dK": got["dK"][keys],
           "dV": got["dV"][keys]}
    print(check_components(sub, ref))
    # dsinks sums over every row: the sampled oracle has all lse and delta, so its dsinks is exact
    check_dsinks(got["dsinks"], ref, p.sinks)


def test_ext_off_is_fa_back(fb):
    """fa_back_ext with no extension runs fa_back's plan: bit-identical outputs."""
    p = synth.from_config("3")
    t = synth.device.to_torch(p, "cuda")
    kw = dict(H=p.H, Hkv=p.Hkv, D=p.D, Dv=p.Dv, M=p.M, scale=p.scale, causal=p.causal, mask=t["mask"],
              mask_heads=p.mask_heads)
    a = fb.backward(t["q"], t["k"], p.k_type, t["v"], p.v_type, t["dO"], **kw)
    out = {n: torch.empty_like(x) for n, x in a.items()}
    ws = torch.empty(fb.fa_back_workspace_size(p.N, p.M, p.H, p.Hkv, p.D, p.Dv), dtype=torch.uint8, device="cuda")
    rc = fb.fa_back_ext(t["q"].data_ptr(), t["k"].data_ptr(), p.k_type, t["v"].data_ptr(), p.v_type,
                        None if t["mask"] is None else t["mask"].data_ptr(), p.mask_heads, t["dO"].data_ptr(),
                        p.scale, p.N, p.M, p.H, p.Hkv, p.D, p.Dv, int(p.causal), None, 0.0, None, None,
                        *[out[n].data_ptr() for n in ("dQ", "dK", "dV", "lse", "delta")], ws.data_ptr(), ws.numel(),
                        torch.cuda.current_stream().cuda_stream)
    assert fb.STATUS[rc] == "FA_OK"
    torch.cuda.synchronize()
    for n in a:
        assert torch.equal(a[n], out[n]), n


def test_ext_runs_are_bit_identical(fb):
    p = synth.make_problem("all_d256", seed=7000 + sorted(EXT).index("all_d256"), **EXT["all_d256"])
    a = run_ext(fb, p)
    b = run_ext(fb, p)
    for k in a:
        assert np.array_equal(a[k], b[k], equal_nan=True), k


@pytest.mark.parametrize("N,M", [(0, 64), (16, 0)])
def test_ext_sinks_without_keys_or_rows(fb, N, M):
    """No keys: every row's softmax holds the sink alone (lse = sigma_h, delta = 0, dQ = 0) and the
    sink gradient is 0; no rows: the sink gradient is 0."""
    p = synth.make_problem("empty_sinks", N=N, M=M, H=4, Hkv=2, D=128, Dv=128, k_type="q8_0", v_type="q8_0", seed=9,
                           sinks=1.0)
    got = run_ext(fb, p)
    assert np.all(got["dK"] == 0) and np.all(got["dV"] == 0) and np.all(got["dQ"] == 0)
    assert np.all(got["delta"] == 0) and np.all(got["dsinks"] == 0)
    assert np.array_equal(got["lse"], np.broadcast_to(p.sinks.astype(np.float32), (N, p.H)))
