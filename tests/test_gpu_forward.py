"""fa_forward() against the oracle's forward (O and lse), through the C ABI.

Tolerance: NMSE <= 1e-5 per component, the bar of the backward's parity tests; lse = -inf
positions must match exactly and rows without keys must give O = 0 exactly.
"""
import numpy as np
import pytest

import synth
from metrics import NMSE_TOL, nmse

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


def forward_parity(fb, p):
    import oracle
    ref = oracle.fa_forward(p)
    t = synth.device.to_torch(p, "cuda")
    fb.fa_back_profile(True)
    out = fb.forward(t["q"], t["k"], p.k_type, t["v"], p.v_type, H=p.H, Hkv=p.Hkv, D=p.D, Dv=p.Dv, M=p.M,
                     scale=p.scale, causal=p.causal, mask=t["mask"], mask_heads=p.mask_heads)
    torch.cuda.synchronize()
    fb.fa_back_profile(False)
    launched = {k for k, v in fb.fa_back_profile_read().items() if v[1] > 0}
    assert "k_fwd" in launched and not launched & {"k_cols", "k_rows_lse", "k_dq_gemm"}, launched
    assert fb.fa_back_get_error() == 0
    got = {k: v.cpu().numpy() for k, v in out.items()}
    dead = ~np.isfinite(ref["lse"])
    assert np.array_equal(np.isneginf(got["lse"]), dead)
    assert np.all(got["O"][dead] == 0.0)
    res = {"lse": nmse(got["lse"], ref["lse"]), "O": nmse(got["O"], ref["O"])}
    assert all(v <= NMSE_TOL for v in res.values()), res
    return res


@pytest.mark.parametrize("cfg", ["0", "1", "1c", "2", "3"])
def test_forward_configs(fb, cfg):
    print(cfg, forward_parity(fb, synth.from_config(cfg)))


FWD_EDGE = {
    "n_gt_m_causal": dict(N=100, M=40, H=4, Hkv=1, D=64, Dv=64, k_type="q8_0", v_type="q8_0", causal=True),
    "d256_dv128": dict(N=50, M=700, H=8, Hkv=2, D=256, Dv=128, k_type="q8_0", v_type="q4_0"),
    "d128_dv256": dict(N=20, M=150, H=3, Hkv=1, D=128, Dv=256, k_type="f16", v_type="q8_0"),
    "d64_dv128_f32": dict(N=33, M=200, H=4, Hkv=4, D=64, Dv=128, k_type="f32", v_type="f32", causal=True),
    "finite_mask_hm1": dict(N=40, M=333, H=4, Hkv=2, D=128, Dv=128, k_type="q4_0", v_type="q4_0",
                            mask="finite", mask_p=0.05, full_rows=3, mask_heads=1),
    "d64_q4_mask_causal": dict(N=200, M=3001, H=8, Hkv=2, D=64, Dv=64, k_type="q4_0", v_type="q8_0", causal=True,
                               mask="random", mask_p=0.05, full_rows=2, mask_heads=8),
    "single_key": dict(N=5, M=1, H=2, Hkv=1, D=64, Dv=64, k_type="q8_0", v_type="q8_0"),
}


@pytest.mark.parametrize("name", sorted(FWD_EDGE))
def test_forward_edge_cases(fb, name):
    p = synth.make_problem(name, seed=5000 + sorted(FWD_EDGE).index(name), **FWD_EDGE[name])
    print(name, forward_parity(fb, p))


def test_forward_statistics_feed_the_backward(fb):
    """fa_forward's lse and rowsum(dO o O) given to fa_back_with_stats reproduce fa_back's gradients."""
    p = synth.from_config("3")
    t = synth.device.to_torch(p, "cuda")
    kw = dict(H=p.H, Hkv=p.Hkv, D=p.D, Dv=p.Dv, M=p.M, scale=p.scale, causal=p.causal, mask=t["mask"],
              mask_heads=p.mask_heads)
    f = fb.forward(t["q"], t["k"], p.k_type, t["v"], p.v_type, **kw)
    delta = (t["dO"] * f["O"]).sum(-1).contiguous()
    a = fb.backward(t["q"], t["k"], p.k_type, t["v"], p.v_type, t["dO"], **kw)
    b = fb.backward(t["q"], t["k"], p.k_type, t["v"], p.v_type, t["dO"], lse=f["lse"], delta=delta, **kw)
    torch.cuda.synchronize()
    assert fb.fa_back_get_error() == 0
    for n in ("dQ", "dK", "dV"):
        assert nmse(b[n].cpu().numpy(), a[n].cpu().numpy()) <= 1e-6, n


def test_forward_rescale_path(fb):
    """Rows whose logits spread widely (each Q row scaled by its own 10^u, |u| <= 1.5): many rows'
    maxima over later key tiles exceed their first tile's by more than the kernel's rescale
    threshold (8 in log2 units), so O rows are rescaled in tensor memory.  The host checks that
    such rows exist, then O and lse are compared with the oracle."""
    import oracle
    p = synth.make_problem("fwd_rescale", N=1024, M=1000, H=20, Hkv=1, D=64, Dv=64, k_type="q8_0", v_type="q8_0",
                           row_decades=1.5, seed=5100)
    kd = oracle.dequant(p.k, p.k_type, p.D).reshape(p.M, p.D)  # one KV head
    s = np.einsum("nhd,md->nhm", p.q.astype(np.float64), kd) * p.scale
    grow = s[:, :, 64:].max(-1) - s[:, :, :64].max(-1)
    assert np.count_nonzero(grow > 8.0 * np.log(2.0)) > 1000
    print(forward_parity(fb, p))
