"""Pins for the CPU oracle: each check ties it to something other than itself.

Routes used: numpy's binary16 conversion, torch float64 autograd of the
forward softmax(scale*QK^T + mask)V, central finite differences of the loss
sum(dO * O), an exact sympy evaluation, closed forms for special cases, and
invariants that follow from the mathematics (sum_j dS_ij = 0).
"""
import math

import numpy as np
import pytest
import torch

import synth
from synth import TYPE_F16, TYPE_F32, TYPE_Q4_0, TYPE_Q8_0


# ------------------------------------------------------------------------------------------------
# independent decoders (numpy's binary16) used only to build the reference's K^ and V^

def np_decode(raw: np.ndarray, t: int, D: int) -> np.ndarray:
    lead = raw.shape[:-1]
    if t == TYPE_F32:
        return np.ascontiguousarray(raw).view(np.float32).astype(np.float64).reshape(*lead, D)
    if t == TYPE_F16:
        return np.ascontiguousarray(raw).view(np.float16).astype(np.float64).reshape(*lead, D)
    if t == TYPE_Q8_0:
        b = np.ascontiguousarray(raw).reshape(-1, 34)
        d = b[:, 0:2].copy().view(np.float16).astype(np.float64)
        q = b[:, 2:].copy().view(np.int8).astype(np.float64)
        return (q * d).reshape(*lead, D)
    b = np.ascontiguousarray(raw).reshape(-1, 18)
    d = b[:, 0:2].copy().view(np.float16).astype(np.float64)
    lo = (b[:, 2:] & 15).astype(np.float64) - 8
    hi = (b[:, 2:] >> 4).astype(np.float64) - 8
    return (np.concatenate([lo, hi], axis=1) * d).reshape(*lead, D)


def torch_reference(p, khat=None, vhat=None):
    """float64 autograd of L = sum(dO * softmax(scale*QK^T + mask) V), with the problem's optional
    soft-cap (c tanh(x / c) of the scaled product), ALiBi bias m_h (j - (M - N + i)) and sink
    logits (one more softmax column per row whose value is zero)."""
    N, M, H, Hkv = p.N, p.M, p.H, p.Hkv
    if khat is None:
        khat = np_decode(p.k, p.k_type, p.D)
    if vhat is None:
        vhat = np_decode(p.v, p.v_type, p.Dv)
    q = torch.tensor(p.q, dtype=torch.float64, requires_grad=True)
    k = torch.tensor(khat, dtype=torch.float64, requires_grad=True)
    v = torch.tensor(vhat, dtype=torch.float64, requires_grad=True)
    dO = torch.tensor(p.dO, dtype=torch.float64)
    G = H // Hkv
    kk = k.repeat_interleave(G, dim=1)
    vv = v.repeat_interleave(G, dim=1)
    s = torch.einsum("nhd,mhd->hnm", q, kk) * p.scale
    if getattr(p, "softcap", 0.0):
        s = p.softcap * torch.tanh(s / p.softcap)
    if p.mask is not None:
        s = s + torch.tensor(p.mask.view(np.float16).astype(np.float64))
    i = torch.arange(N, dtype=torch.float64)[:, None]
    j = torch.arange(M, dtype=torch.float64)[None, :]
    if getattr(p, "alibi", None) is not None:
        s = s + torch.tensor(p.alibi, dtype=torch.float64)[:, None, None] * (j - (M - N + i))
    if p.causal:
        s = s.masked_fill(j > M - N + i, float("-inf"))
    sk = None
    if getattr(p, "sinks", None) is not None:
        sk = torch.tensor(p.sinks, dtype=torch.float64, requires_grad=True)
        s = torch.cat([s, sk[:, None, None].expand(H, N, 1)], dim=-1)
    lse = torch.logsumexp(s, dim=-1).T.contiguous()
    pr = torch.softmax(s, dim=-1)[..., :M]
    o = torch.einsum("hnm,mhd->nhd", pr, vv)
    (o * dO).sum().backward()
    delta = (o * dO).sum(-1)
    out = {"lse": lse.detach().numpy(), "delta": delta.detach().numpy(), "dQ": q.grad.numpy(),
           "dK": k.grad.numpy(), "dV": v.grad.numpy(), "O": o.detach().numpy()}
    if sk is not None:
        out["dsinks"] = sk.grad.numpy()
    return out


def rel_err(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = max(np.max(np.abs(b)), 1e-300)
    return float(np.max(np.abs(a - b)) / den)


# ------------------------------------------------------------------------------------------------
# decoders

def test_binary16_every_bit_pattern(oracle_lib):
    bits = np.arange(65536, dtype=np.uint16)
    got = oracle_lib.dequant(bits.view(np.uint8).reshape(1, -1), TYPE_F16, 65536)[0]
    ref = bits.view(np.float16).astype(np.float64)
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.array_equal(got[np.isinf(ref)], ref[np.isinf(ref)])
    assert np.all(np.isnan(got[np.isnan(ref)]))


def _f16_bits(x: float) -> bytes:
    return np.array([x], dtype=np.float16).tobytes()


def test_q8_0_hand_built_blocks(oracle_lib):
    codes = np.array(list(range(-127, 128, 8)) + [127], dtype=np.int8)[:32]
    assert codes.size == 32
    blocks = [(0.5, codes), (-1.5, codes[::-1].copy()), (2.0 ** -24, codes)]  # last: subnormal scale
    raw = b"".join(_f16_bits(d) + c.tobytes() for d, c in blocks)
    got = oracle_lib.dequant(np.frombuffer(raw, dtype=np.uint8).reshape(1, -1), TYPE_Q8_0, 96)[0]
    want = np.concatenate([c.astype(np.float64) * d for d, c in blocks])
    assert np.array_equal(got, want)


def test_q8_0_every_code(oracle_lib):
    """All 256 int8 codes, -128 included (a valid code that the quantizers here never write), in
    eight blocks with their own scales: each decodes to code times its block's d."""
    codes = np.arange(-128, 128, dtype=np.int16).astype(np.int8).reshape(8, 32)
    scales = [1.0, -0.5, 0.125, 3.0, -2.0 ** -14, 7.5, 2.0 ** -20, -1.0]
    raw = b"".join(_f16_bits(d) + c.tobytes() for d, c in zip(scales, codes))
    got = oracle_lib.dequant(np.frombuffer(raw, dtype=np.uint8).reshape(1, -1), TYPE_Q8_0, 256)[0]
    want = np.concatenate([c.astype(np.float64) * np.float64(np.float16(d)) for d, c in zip(scales, codes)])
    assert np.array_equal(got, want)
    assert got[0] == -128.0


def test_q4_0_nibble_order_ramp(oracle_lib):
    # byte b: low nibble b (element b), high nibble 15-b (element b+16)
    body = bytes(((15 - b) << 4) | b for b in range(16))
    raw = _f16_bits(0.25) + body + _f16_bits(-3.0) + body
    got = oracle_lib.dequant(np.frombuffer(raw, dtype=np.uint8).reshape(1, -1), TYPE_Q4_0, 64)[0]
    first = [(b - 8) * 0.25 for b in range(16)] + [(15 - b - 8) * 0.25 for b in range(16)]
    second = [(b - 8) * -3.0 for b in range(16)] + [(15 - b - 8) * -3.0 for b in range(16)]
    assert np.array_equal(got, np.array(first + second))


@pytest.mark.parametrize("t", [TYPE_Q8_0, TYPE_Q4_0, TYPE_F16, TYPE_F32])
def test_decoder_matches_numpy_on_quantized_normals(oracle_lib, t):
    x = synth.gen.normal_f32(7, 1, (64, 256))
    raw = synth.quantize_rows(x, t)
    assert np.array_equal(oracle_lib.dequant(raw, t, 256), np_decode(raw, t, 256))
    # quantizer sanity: the decoded rows stay within one step of the input
    err = np.abs(oracle_lib.dequant(raw, t, 256) - x).reshape(-1, 32).max(axis=1)
    amax = np.abs(x).reshape(-1, 32).max(axis=1)
    bound = {TYPE_Q8_0: 0.51 * amax / 127 + 2e-3 * amax, TYPE_Q4_0: 1.01 * amax / 8 + 2e-3 * amax,  # the far side clips to code 15
             TYPE_F16: 1e-3 * amax, TYPE_F32: 0 * amax}[t]
    assert np.all(err <= bound + 1e-30)


# ------------------------------------------------------------------------------------------------
# against torch float64 autograd

AUTOGRAD_CASES = [
    dict(N=5, M=7, H=2, Hkv=2, D=8, Dv=8, k_type="f32", v_type="f32"),
    dict(N=6, M=9, H=4, Hkv=2, D=16, Dv=8, k_type="f16", v_type="f16", causal=True),
    dict(N=7, M=40, H=6, Hkv=2, D=32, Dv=32, k_type="q8_0", v_type="q8_0", mask="finite", mask_p=0.2,
         mask_heads=1),
    dict(N=9, M=33, H=4, Hkv=1, D=64, Dv=32, k_type="q4_0", v_type="q8_0", mask="random", mask_p=0.3,
         mask_heads=4, causal=True),
    dict(N=3, M=50, H=3, Hkv=3, D=32, Dv=64, k_type="q8_0", v_type="f32", mask="finite", mask_p=0.0,
         mask_heads=3, scale=0.37),
]


@pytest.mark.parametrize("case", range(len(AUTOGRAD_CASES)))
def test_oracle_matches_torch_autograd(oracle_lib, case):
    p = synth.make_problem(f"ag{case}", seed=300 + case, **AUTOGRAD_CASES[case])
    ref = torch_reference(p)
    # rows whose keys are all masked are checked elsewhere; here every row keeps a key
    assert np.all(np.isfinite(ref["lse"]))
    got = oracle_lib.fa_back(p)
    for name in ("lse", "delta", "dQ", "dK", "dV"):
        assert rel_err(got[name], ref[name]) < 1e-12, name


# the extensions (ALiBi, soft-capping, sink logits), alone and together, against the same
# autograd route
EXT_CASES = [
    dict(N=5, M=9, H=2, Hkv=2, D=8, Dv=8, k_type="f32", v_type="f32", alibi=True),
    dict(N=6, M=11, H=4, Hkv=2, D=16, Dv=8, k_type="f16", v_type="f16", causal=True, softcap=1.5),
    dict(N=4, M=13, H=2, Hkv=1, D=32, Dv=32, k_type="q8_0", v_type="q8_0", sinks=1.0),
    dict(N=9, M=33, H=4, Hkv=2, D=64, Dv=32, k_type="q4_0", v_type="q8_0", mask="finite", mask_p=0.2,
         mask_heads=4, causal=True, alibi=True, softcap=2.0, sinks=0.5),
]


@pytest.mark.parametrize("case", range(len(EXT_CASES)))
def test_extensions_match_torch_autograd(oracle_lib, case):
    p = synth.make_problem(f"ext{case}", seed=320 + case, **EXT_CASES[case])
    ref = torch_reference(p)
    got = oracle_lib.fa_back(p)
    names = ["lse", "delta", "dQ", "dK", "dV"] + (["dsinks"] if p.sinks is not None else [])
    for name in names:
        assert rel_err(got[name], ref[name]) < 1e-11, name


def test_extensions_switched_off_equal_the_plain_oracle(oracle_lib):
    """Zero ALiBi slopes and a sink logit of -1e300 change nothing; a soft-cap of 1e7 changes the
    logits by less than x^3 / (3 c^2)."""
    base = dict(N=7, M=20, H=4, Hkv=2, D=32, Dv=32, k_type="q8_0", v_type="q8_0", causal=True, seed=330)
    p = synth.make_problem("plain", **base)
    ref = oracle_lib.fa_back(p)
    q = synth.make_problem("off", alibi=True, sinks=1.0, **base)
    q.alibi = np.zeros(p.H, dtype=np.float32)
    q.sinks = np.full(p.H, -1e300)
    got = oracle_lib.fa_back(q)
    for name in ("lse", "delta", "dQ", "dK", "dV"):
        assert np.array_equal(got[name], ref[name]), name
    assert np.all(got["dsinks"] == 0.0)
    r = synth.make_problem("cap", softcap=1e7, **base)
    got = oracle_lib.fa_back(r)
    for name in ("lse", "delta", "dQ", "dK", "dV"):
        assert rel_err(got[name], ref[name]) < 1e-12, name


def test_sink_with_a_fully_masked_row(oracle_lib):
    """A row without an allowed key: with a sink its lse is the sink logit, its delta, dQ row and
    share of the sink's gradient are zero."""
    p = synth.make_problem("sinkmask", N=6, M=15, H=2, Hkv=1, D=16, Dv=16, k_type="f32", v_type="f32",
                           mask="random", mask_p=0.1, full_rows=2, mask_heads=2, sinks=1.0, seed=331)
    got = oracle_lib.fa_back(p)
    rows = p.meta["full_rows"]
    for h in range(p.H):
        assert np.array_equal(got["lse"][rows, h], np.full(len(rows), float(p.sinks[h])))
    assert np.all(got["delta"][rows] == 0.0) and np.all(got["dQ"][rows] == 0.0)
    ref = torch_reference(p)
    assert rel_err(got["dsinks"], ref["dsinks"]) < 1e-11


def test_delta_is_rowsum_dO_times_O(oracle_lib):
    p = synth.make_problem("delta", N=16, M=64, H=4, Hkv=2, D=32, Dv=32, k_type="q8_0", v_type="q8_0",
                           causal=True, seed=41)
    vhat = np_decode(p.v, p.v_type, p.Dv)
    khat = np_decode(p.k, p.k_type, p.D)
    # O formed explicitly with plain numpy
    O = np.zeros((p.N, p.H, p.Dv))
    for i in range(p.N):
        for h in range(p.H):
            hk = h // p.G
            s = p.scale * (khat[:, hk, :] @ p.q[i, h].astype(np.float64))
            s[np.arange(p.M) > p.M - p.N + i] = -np.inf
            w = np.exp(s - s.max())
            w /= w.sum()
            O[i, h] = w @ vhat[:, hk, :]
    got = oracle_lib.fa_back(p, want_dkv=False)
    assert rel_err(got["delta"], (p.dO.astype(np.float64) * O).sum(-1)) < 1e-12


# ------------------------------------------------------------------------------------------------
# finite differences of the loss

def _np_loss(q, khat, vhat, dO, p):
    N, M, H, G = p.N, p.M, p.H, p.G
    maskv = None if p.mask is None else p.mask.view(np.float16).astype(np.float64)
    tot = 0.0
    for i in range(N):
        for h in range(H):
            hk = h // G
            s = p.scale * (khat[:, hk, :] @ q[i, h])
            if maskv is not None:
                s = s + maskv[h % p.mask_heads, i]
            if p.causal:
                s[np.arange(M) > M - N + i] = -np.inf
            w = np.exp(s - s.max())
            w /= w.sum()
            tot += float(dO[i, h] @ (w @ vhat[:, hk, :]))
    return tot


def test_oracle_matches_finite_differences(oracle_lib):
    p = synth.make_problem("fd", N=3, M=5, H=2, Hkv=1, D=4, Dv=3, k_type="f32", v_type="f32", causal=True,
                           mask="finite", mask_p=0.2, mask_heads=2, seed=11)
    q = p.q.astype(np.float64)
    khat = np_decode(p.k, p.k_type, p.D)
    vhat = np_decode(p.v, p.v_type, p.Dv)
    dO = p.dO.astype(np.float64)
    got = oracle_lib.fa_back(p)
    step = 1e-6

    def fd(arr, which):
        g = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            a = arr.copy()
            a[idx] += step
            args = {"q": q, "k": khat, "v": vhat}
            args[which] = a
            up = _np_loss(args["q"], args["k"], args["v"], dO, p)
            a[idx] -= 2 * step
            dn = _np_loss(args["q"], args["k"], args["v"], dO, p)
            g[idx] = (up - dn) / (2 * step)
        return g

    assert rel_err(got["dQ"], fd(q, "q")) < 1e-6
    assert rel_err(got["dK"], fd(khat, "k")) < 1e-6
    assert rel_err(got["dV"], fd(vhat, "v")) < 1e-6


# ------------------------------------------------------------------------------------------------
# exact evaluation with sympy

def test_oracle_matches_exact_sympy_evaluation(oracle_lib):
    sp = pytest.importorskip("sympy")
    N, M, D, Dv = 2, 3, 2, 2
    qv = [[0.5, -1.25], [2.0, 0.75]]
    kv = [[1.0, 0.5], [-0.25, 1.5], [0.75, -1.0]]
    vv = [[0.5, 2.0], [-1.0, 0.25], [1.5, -0.5]]
    dov = [[1.0, -0.5], [0.25, 1.25]]
    maskv = [[0.0, -0.5, 0.0], [-1.0, 0.0, float("-inf")]]  # [N][M] for the single head
    scale = 0.5
    f32 = np.float32
    p = synth.gen.Problem(name="sympy", N=N, M=M, H=1, Hkv=1, D=D, Dv=Dv, k_type=TYPE_F32, v_type=TYPE_F32,
                          causal=False, scale=scale, q=np.array(qv, dtype=f32).reshape(N, 1, D),
                          k=np.array(kv, dtype=f32).reshape(M, 1, D).view(np.uint8).reshape(M, 1, 4 * D),
                          v=np.array(vv, dtype=f32).reshape(M, 1, Dv).view(np.uint8).reshape(M, 1, 4 * Dv),
                          dO=np.array(dov, dtype=f32).reshape(N, 1, Dv),
                          mask=np.array(maskv, dtype=np.float16).view(np.uint16).reshape(1, N, M), mask_heads=1)
    R = sp.Rational
    Q = sp.Matrix([[R(str(x)) for x in r] for r in qv])
    K = sp.Matrix([[R(str(x)) for x in r] for r in kv])
    V = sp.Matrix([[R(str(x)) for x in r] for r in vv])
    dO = sp.Matrix([[R(str(x)) for x in r] for r in dov])
    sc = R(1, 2)
    lse, delta = [], []
    dQ = sp.zeros(N, D)
    dK = sp.zeros(M, D)
    dV = sp.zeros(M, Dv)
    for i in range(N):
        keys = [j for j in range(M) if maskv[i][j] != float("-inf")]
        s = {j: sc * (Q.row(i) * K.row(j).T)[0] + R(str(maskv[i][j])) for j in keys}
        Z = sum(sp.exp(s[j]) for j in keys)
        pr = {j: sp.exp(s[j]) / Z for j in keys}
        dp = {j: (dO.row(i) * V.row(j).T)[0] for j in keys}
        de = sum(pr[j] * dp[j] for j in keys)
        lse.append(sp.log(Z))
        delta.append(de)
        for j in keys:
            ds = pr[j] * (dp[j] - de)
            dQ[i, :] += sc * ds * K.row(j)
            dK[j, :] += sc * ds * Q.row(i)
            dV[j, :] += pr[j] * dO.row(i)
    ev = lambda e: float(sp.N(e, 30))  # noqa: E731
    got = oracle_lib.fa_back(p)
    assert np.allclose(got["lse"][:, 0], [ev(x) for x in lse], rtol=1e-14, atol=0)
    assert np.allclose(got["delta"][:, 0], [ev(x) for x in delta], rtol=1e-13, atol=1e-15)
    assert np.allclose(got["dQ"][:, 0, :], np.array([[ev(x) for x in dQ.row(i)] for i in range(N)]),
                       rtol=1e-13, atol=1e-15)
    assert np.allclose(got["dK"][:, 0, :], np.array([[ev(x) for x in dK.row(j)] for j in range(M)]),
                       rtol=1e-13, atol=1e-15)
    assert np.allclose(got["dV"][:, 0, :], np.array([[ev(x) for x in dV.row(j)] for j in range(M)]),
                       rtol=1e-13, atol=1e-15)


# ------------------------------------------------------------------------------------------------
# closed forms for special cases

def test_zero_queries_give_uniform_softmax(oracle_lib):
    p = synth.make_problem("q0", N=4, M=10, H=4, Hkv=2, D=32, Dv=32, k_type="q8_0", v_type="f16", seed=5)
    p.q[:] = 0.0
    got = oracle_lib.fa_back(p)
    khat = np_decode(p.k, p.k_type, p.D)
    vhat = np_decode(p.v, p.v_type, p.Dv)
    assert np.allclose(got["lse"], math.log(p.M), rtol=1e-15)
    for i in range(p.N):
        for h in range(p.H):
            hk = h // p.G
            dp = vhat[:, hk, :] @ p.dO[i, h].astype(np.float64)
            assert abs(got["delta"][i, h] - dp.mean()) <= 1e-13 * np.abs(dp).max()
            want = p.scale * ((dp - dp.mean()) / p.M) @ khat[:, hk, :]
            assert rel_err(got["dQ"][i, h], want) < 1e-12
    assert np.all(got["dK"] == 0.0)


def test_single_key_gives_zero_score_gradients(oracle_lib):
    p = synth.make_problem("m1", N=3, M=1, H=4, Hkv=2, D=32, Dv=32, k_type="q8_0", v_type="q8_0", seed=6)
    got = oracle_lib.fa_back(p)
    khat = np_decode(p.k, p.k_type, p.D)
    vhat = np_decode(p.v, p.v_type, p.Dv)
    for i in range(p.N):
        for h in range(p.H):
            hk = h // p.G
            s = p.scale * float(p.q[i, h].astype(np.float64) @ khat[0, hk])
            assert abs(got["lse"][i, h] - s) <= 1e-14 * max(1.0, abs(s))
            assert abs(got["delta"][i, h] - float(p.dO[i, h].astype(np.float64) @ vhat[0, hk])) < 1e-12
    assert np.max(np.abs(got["dQ"])) < 1e-14 and np.max(np.abs(got["dK"])) < 1e-14
    for hk in range(p.Hkv):
        want = p.dO[:, hk * p.G:(hk + 1) * p.G].astype(np.float64).sum(axis=(0, 1))
        assert rel_err(got["dV"][0, hk], want) < 1e-14


def test_fully_masked_rows_and_causal_rows_without_keys(oracle_lib):
    p = synth.make_problem("fm", N=12, M=8, H=4, Hkv=2, D=32, Dv=32, k_type="q4_0", v_type="q8_0",
                           causal=True, mask="random", mask_p=0.1, full_rows=2, mask_heads=4, seed=8)
    got = oracle_lib.fa_back(p)
    empty = set(p.meta["full_rows"].tolist()) | set(range(p.N - p.M))  # causal rows i < N-M see no key
    for i in range(p.N):
        if i in empty:
            assert np.all(got["lse"][i] == -np.inf)
            assert np.all(got["delta"][i] == 0.0)
            assert np.all(got["dQ"][i] == 0.0)
        else:
            assert np.all(np.isfinite(got["lse"][i]))


@pytest.mark.parametrize("cfg", ["1", "3"])
def test_gradient_sum_invariants(oracle_lib, cfg):
    p = synth.from_config(cfg)
    got = oracle_lib.fa_back(p)
    live = np.isfinite(got["lse"])  # [N][H]
    for hk in range(p.Hkv):
        heads = slice(hk * p.G, (hk + 1) * p.G)
        # sum_j dS_ij = 0 for every row, hence sum_j dK_j = 0
        sk = got["dK"][:, hk].sum(axis=0)
        assert np.max(np.abs(sk)) <= 1e-11 * np.abs(got["dK"][:, hk]).sum(axis=0).max()
        # sum_j p_ij = 1 for every live row, hence sum_j dV_j = sum of those rows of dO
        want = (p.dO[:, heads].astype(np.float64) * live[:, heads, None]).sum(axis=(0, 1))
        assert rel_err(got["dV"][:, hk].sum(axis=0), want) < 1e-11


def test_masked_keys_contribute_nothing(oracle_lib):
    p = synth.make_problem("mk", N=6, M=20, H=4, Hkv=2, D=32, Dv=32, k_type="q8_0", v_type="q8_0",
                           mask="random", mask_p=0.1, mask_heads=4, seed=9)
    dead = [3, 11]
    m = p.mask.copy()
    m[:, :, dead] = synth.gen.F16_NEG_INF
    p.mask = m
    a = oracle_lib.fa_back(p)
    g = synth.make_problem("mk2", N=6, M=20, H=4, Hkv=2, D=32, Dv=32, k_type="q8_0", v_type="q8_0", seed=99)
    p.k = p.k.copy()
    p.v = p.v.copy()
    p.k[dead] = g.k[dead]
    p.v[dead] = g.v[dead]
    b = oracle_lib.fa_back(p)
    for name in ("lse", "delta", "dQ"):
        assert np.array_equal(a[name], b[name]), name
    keep = [j for j in range(p.M) if j not in dead]
    assert np.array_equal(a["dK"][keep], b["dK"][keep]) and np.array_equal(a["dV"][keep], b["dV"][keep])
    assert np.all(b["dK"][dead] == 0.0) and np.all(b["dV"][dead] == 0.0)


def test_sampled_rows_and_keys_equal_full_run(oracle_lib):
    p = synth.from_config("3")
    full = oracle_lib.fa_back(p)
    rows = np.array([0, 5, 76, 127])
    keys = np.array([1, 200, 4095])
    sub = oracle_lib.fa_back(p, dq_rows=rows, dkv_keys=keys)
    assert np.array_equal(sub["lse"], full["lse"]) and np.array_equal(sub["delta"], full["delta"])
    assert np.array_equal(sub["dQ"], full["dQ"][rows])
    assert np.array_equal(sub["dK"], full["dK"][keys]) and np.array_equal(sub["dV"], full["dV"][keys])


def test_empty_problems(oracle_lib):
    p = synth.make_problem("e0", N=0, M=16, H=2, Hkv=1, D=32, Dv=32, k_type="q8_0", v_type="q8_0", seed=1)
    got = oracle_lib.fa_back(p)
    assert np.all(got["dK"] == 0) and np.all(got["dV"] == 0)
    p = synth.make_problem("e1", N=4, M=0, H=2, Hkv=1, D=32, Dv=32, k_type="q8_0", v_type="q8_0", seed=1)
    got = oracle_lib.fa_back(p)
    assert np.all(got["lse"] == -np.inf) and np.all(got["delta"] == 0) and np.all(got["dQ"] == 0)


# ------------------------------------------------------------------------------------------------
# forward output O (oracle_fa_forward)

@pytest.mark.parametrize("case", range(len(AUTOGRAD_CASES)))
def test_forward_matches_torch(oracle_lib, case):
    p = synth.make_problem(f"fw{case}", seed=300 + case, **AUTOGRAD_CASES[case])
    ref = torch_reference(p)
    got = oracle_lib.fa_forward(p)
    assert rel_err(got["lse"], ref["lse"]) < 1e-12
    assert rel_err(got["O"], ref["O"]) < 1e-12


def test_forward_O_gives_the_backward_delta(oracle_lib):
    """rowsum(dO o O) from the forward's O equals the backward's delta (formed as sum p * dP)."""
    p = synth.make_problem("fwd_delta", N=24, M=300, H=8, Hkv=2, D=64, Dv=128, k_type="q4_0", v_type="q8_0",
                           causal=True, mask="random", mask_p=0.1, full_rows=2, seed=71)
    fw = oracle_lib.fa_forward(p)
    bw = oracle_lib.fa_back(p, want_dq=False, want_dkv=False)
    assert np.array_equal(fw["lse"], bw["lse"])
    d = (p.dO.astype(np.float64) * fw["O"]).sum(-1)
    assert rel_err(d, bw["delta"]) < 1e-12
    dead = ~np.isfinite(fw["lse"])
    assert dead.any() and np.all(fw["O"][dead] == 0.0)


def test_forward_single_key_and_zero_queries(oracle_lib):
    p = synth.make_problem("fw_m1", N=3, M=1, H=4, Hkv=2, D=32, Dv=64, k_type="q8_0", v_type="q4_0", seed=72)
    vhat = np_decode(p.v, p.v_type, p.Dv)
    got = oracle_lib.fa_forward(p)
    for h in range(p.H):
        assert np.array_equal(got["O"][:, h], np.broadcast_to(vhat[0, h // p.G], (p.N, p.Dv)))
    p = synth.make_problem("fw_q0", N=4, M=10, H=4, Hkv=2, D=32, Dv=32, k_type="f16", v_type="q8_0", seed=73)
    p.q[:] = 0.0
    vhat = np_decode(p.v, p.v_type, p.Dv)
    got = oracle_lib.fa_forward(p)
    for h in range(p.H):
        want = vhat[:, h // p.G].mean(axis=0)
        assert rel_err(got["O"][:, h], np.broadcast_to(want, (p.N, p.Dv))) < 1e-14
