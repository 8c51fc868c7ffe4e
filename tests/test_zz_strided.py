"""fa_back_strided(): inputs given as views and a bit-packed mask, through the C ABI.

The entry point copies each view into a contiguous region and runs fa_back() on it, so on the
same input values it must give bit-identical outputs to fa_back() on contiguous copies (same
plan, same kernels, same bytes).  One case is also compared with the oracle directly.
"""
import numpy as np
import pytest

import synth
from metrics import check_components

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


def contiguous(fb, p, mask=None, mask_heads=None):
    t = synth.device.to_torch(p, "cuda")
    m = t["mask"] if mask is None else mask
    out = fb.backward(t["q"], t["k"], p.k_type, t["v"], p.v_type, t["dO"], H=p.H, Hkv=p.Hkv, D=p.D, Dv=p.Dv, M=p.M,
                      scale=p.scale, causal=p.causal, mask=m, mask_heads=p.mask_heads if mask_heads is None else mask_heads)
    torch.cuda.synchronize()
    assert fb.fa_back_get_error() == 0
    return {k: v.cpu().numpy() for k, v in out.items()}


def strided(fb, p, q, k, v, dO, mask, mask_bits=False):
    out = fb.backward_strided(q, k, p.k_type, v, p.v_type, dO, H=p.H, Hkv=p.Hkv, D=p.D, Dv=p.Dv, M=p.M,
                              scale=p.scale, causal=p.causal, mask=mask, mask_heads=p.mask_heads if mask is not None else 0,
                              mask_bits=mask_bits)
    torch.cuda.synchronize()
    assert fb.fa_back_get_error() == 0
    return {k: v.cpu().numpy() for k, v in out.items()}


def same(a, b):
    for n in a:
        assert np.array_equal(a[n], b[n], equal_nan=True), n


def test_views_equal_contiguous_inputs(fb):
    p = synth.make_problem("views", N=37, M=301, H=6, Hkv=2, D=128, Dv=128, k_type="q8_0", v_type="q8_0", causal=True,
                           mask="finite", mask_p=0.05, full_rows=2, mask_heads=6, seed=7100)
    t = synth.device.to_torch(p, "cuda")
    N, M, H, Hkv, D, Dv = p.N, p.M, p.H, p.Hkv, p.D, p.Dv
    # Q stored head-major with every other component: strides (2D, 2ND, 2)
    qs = torch.zeros((H, N, 2 * D), dtype=torch.float32, device="cuda")
    qs[:, :, ::2] = t["q"].permute(1, 0, 2)
    qv = qs[:, :, ::2].permute(1, 0, 2)
    # dO inside a buffer with a spare head: strides ((H+1)Dv, Dv, 1)
    ds = torch.zeros((N, H + 1, Dv), dtype=torch.float32, device="cuda")
    ds[:, :H] = t["dO"]
    dv_ = ds[:, :H]
    # K rows inside padded cells (a spare head and 6 spare bytes a row): byte strides
    # ((Hkv+1)(rb+6), rb+6, 1)
    rb = t["k"].shape[2]
    ks = torch.zeros((M, Hkv + 1, rb + 6), dtype=torch.uint8, device="cuda")
    ks[:, :Hkv, :rb] = t["k"]
    kv = ks[:, :Hkv, :rb]
    # V stored head-major: byte strides (rb, M rb, 1)
    vs = t["v"].permute(1, 0, 2).contiguous()
    vv = vs.permute(1, 0, 2)
    # mask rows inside wider rows: strides (N (M+5), M+5, 1)
    ms = torch.zeros((p.mask_heads, N, M + 5), dtype=torch.int16, device="cuda")
    ms[:, :, :M] = t["mask"].view(p.mask_heads, N, M)
    mv = ms[:, :, :M]
    assert not any(x.is_contiguous() for x in (qv, dv_, kv, vv, mv))
    got = strided(fb, p, qv, kv, vv, dv_, mv)
    same(got, contiguous(fb, p))
    import oracle
    check_components(got, oracle.fa_back(p))


def test_broadcast_dO_equals_its_expanded_copy(fb):
    p = synth.make_problem("bcast", N=20, M=150, H=4, Hkv=1, D=64, Dv=64, k_type="f16", v_type="q4_0", seed=7200)
    p.dO[:] = p.dO[:, :1, :]  # one dO row shared by every head
    t = synth.device.to_torch(p, "cuda")
    dO_b = t["dO"][:, :1, :].expand(p.N, p.H, p.Dv)  # head stride 0
    assert dO_b.stride(1) == 0
    got = strided(fb, p, t["q"], t["k"], t["v"], dO_b, None)
    same(got, contiguous(fb, p))


def pack_bits(allowed: np.ndarray) -> np.ndarray:
    """[Hm][N][M] bool -> int32 words [Hm][N][ceil(M/32)], bit j % 32 of word j // 32 = key j allowed."""
    Hm, N, M = allowed.shape
    words = np.zeros((Hm, N, (M + 31) // 32), dtype=np.uint32)
    for j in range(M):
        words[:, :, j >> 5] |= allowed[:, :, j].astype(np.uint32) << np.uint32(j & 31)
    return words.view(np.int32)


@pytest.mark.parametrize("Hm", [1, 4])
def test_bit_packed_mask_equals_its_binary16_form(fb, Hm):
    p = synth.make_problem(f"bits{Hm}", N=40, M=333, H=4, Hkv=2, D=64, Dv=64, k_type="q4_0", v_type="q8_0",
                           causal=True, seed=7300 + Hm)
    rng = np.random.default_rng(7310 + Hm)
    allowed = rng.random((Hm, p.N, p.M)) > 0.1
    allowed[:, 3, :] = False  # a fully masked row
    f16 = np.where(allowed, np.float16(0.0), np.float16(-np.inf)).view(np.uint16)
    p.mask, p.mask_heads = np.ascontiguousarray(f16), Hm
    t = synth.device.to_torch(p, "cuda")
    words = torch.from_numpy(pack_bits(allowed)).cuda()
    got = strided(fb, p, t["q"], t["k"], t["v"], t["dO"], words, mask_bits=True)
    same(got, contiguous(fb, p))
    import oracle
    check_components(got, oracle.fa_back(p))
    assert np.all(got["lse"][3] == -np.inf) and np.all(got["dQ"][3] == 0.0)
