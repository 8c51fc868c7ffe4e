"""Seeded random problems against the oracle, on every plan level, and for the forward.

Each case draws its shape (ragged N and M, GQA ratio, D and Dv), cache types, mask kind, causal
tail and score extensions from a seeded generator, then runs the CUDA path with the workspace
of one plan level and compares every component with the oracle (NMSE <= 1e-5; lse = -inf
positions exact; rows without keys give delta = 0 and dQ = 0; dsinks as check_dsinks states).
The draws cover combinations that the hand-picked cases do not.  FAB_FUZZ_CASES,
FAB_FUZZ_PRECISION and FAB_FUZZ_FORWARD set how many draws of each kind run (32, 16 and 16 by
default), for a wider sweep.
"""
import os

import numpy as np
import pytest

import synth
from metrics import check_components, check_dsinks

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TYPES = ["f32", "f16", "q8_0", "q4_0"]
HEADS = [(1, 1), (2, 1), (4, 2), (6, 2), (8, 2), (4, 4), (12, 4)]
N_CASES = int(os.environ.get("FAB_FUZZ_CASES", "32"))
N_PRECISION = int(os.environ.get("FAB_FUZZ_PRECISION", "16"))
N_FORWARD = int(os.environ.get("FAB_FUZZ_FORWARD", "16"))
DIMS = [64, 128, 256]


def draw(case: int) -> dict:
    """The problem of fuzz case `case` (a pure function of the case number)."""
    rng = np.random.default_rng(91000 + case)
    H, Hkv = HEADS[rng.integers(len(HEADS))]
    D = int(rng.choice(DIMS))
    Dv = int(rng.choice(DIMS)) if rng.random() < 0.3 else D
    N = int(rng.integers(1, 160))
    M = int(rng.integers(1, 1500))
    kw = dict(N=N, M=M, H=H, Hkv=Hkv, D=D, Dv=Dv, k_type=TYPES[rng.integers(4)], v_type=TYPES[rng.integers(4)],
              causal=bool(rng.random() < 0.5), seed=92000 + case)
    mk = rng.random()
    if mk < 0.25:
        kw.update(mask="random", mask_p=float(rng.uniform(0.0, 0.3)), full_rows=int(rng.integers(0, 3)),
                  mask_heads=int(rng.choice([1, H])))
    elif mk < 0.4:
        kw.update(mask="finite", mask_p=float(rng.uniform(0.0, 0.2)), full_rows=int(rng.integers(0, 2)),
                  mask_heads=int(rng.choice([1, H])))
    if rng.random() < 0.3:  # score extensions, each on its own
        kw.update(alibi=bool(rng.random() < 0.5), softcap=float(rng.choice([0.0, 2.0, 10.0])),
                  sinks=float(rng.uniform(0.5, 2.0)) if rng.random() < 0.5 else None)
    return kw


@pytest.fixture(scope="module")
def fb():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import flash_attention_backward_gb300 as m
    from flash_attention_backward_gb300 import build
    build.build()
    return m


def level_workspace(fb, p, level):
    lo = fb.fa_back_workspace_size_min(p.N, p.M, p.H, p.Hkv, p.D, p.Dv)
    hi = fb.fa_back_workspace_size(p.N, p.M, p.H, p.Hkv, p.D, p.Dv)
    if level == 0:
        return lo
    if level == 2:
        return hi
    for k in range(201):
        w = lo + (hi - lo) * k // 200
        if fb.fa_back_plan_info(p.N, p.M, p.H, p.Hkv, p.D, p.Dv, w)[1] == level:
            return w
    return None


@pytest.mark.parametrize("case", range(N_CASES))
def test_fuzz_against_the_oracle(fb, case):
    import oracle
    kw = draw(case)
    p = synth.make_problem(f"fuzz{case}", **kw)
    level = case % 4  # 0, 1, 2, 3 in turn
    ws = level_workspace(fb, p, level)
    if ws is None:
        ws, level = fb.fa_back_workspace_size(p.N, p.M, p.H, p.Hkv, p.D, p.Dv), 2
    t = synth.device.to_torch(p, "cuda")
    dev = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to("cuda")
    out = fb.backward(t["q"], t["k"], p.k_type, t["v"], p.v_type, t["dO"], H=p.H, Hkv=p.Hkv, D=p.D, Dv=p.Dv,
                      M=p.M, scale=p.scale, causal=p.causal, mask=t["mask"], mask_heads=p.mask_heads,
                      workspace_bytes=ws, alibi_slopes=dev(p.alibi), softcap=p.softcap, sinks=dev(p.sinks))
    torch.cuda.synchronize()
    assert fb.fa_back_get_error() == 0
    got = {k: v.cpu().numpy() for k, v in out.items()}
    ref = oracle.fa_back(p)
    res = check_components(got, ref)
    dead = ~np.isfinite(ref["lse"])
    assert np.all(got["dQ"][dead] == 0.0)
    if p.sinks is not None:
        res["dsinks"] = check_dsinks(got["dsinks"], ref, p.sinks)
    print(case, level, {k: v for k, v in kw.items() if k != "seed"}, res)


def draw_precision(case: int) -> dict:
    """Precision stress inside the envelope the design states (logits up to about 2): a V that is
    nearly constant along the keys (offset much larger than its spread), tiny dO, per-row ranges of
    Q and dO rows, larger Q."""
    kw = draw(1000 + case)
    rng = np.random.default_rng(93000 + case)
    kind = case % 4
    if kind == 0:
        kw.update(v_offset=float(rng.choice([3.0, 10.0])), v_sigma=float(rng.choice([0.01, 0.05])))
    elif kind == 1:
        kw.update(do_sigma=1e-6)
    elif kind == 2:
        kw.update(row_decades=float(rng.uniform(1.0, 2.5)), scale=1e-3 / kw["D"] ** 0.5)
    else:
        kw.update(q_sigma=2.0)
    for k in ("alibi", "softcap", "sinks"):  # the plain operation
        kw.pop(k, None)
    return kw


@pytest.mark.parametrize("case", range(N_PRECISION))
def test_fuzz_precision_against_the_oracle(fb, case):
    import oracle
    kw = draw_precision(case)
    p = synth.make_problem(f"fuzzp{case}", **kw)
    level = (case // 4) % 4
    ws = level_workspace(fb, p, level)
    if ws is None:
        ws, level = fb.fa_back_workspace_size(p.N, p.M, p.H, p.Hkv, p.D, p.Dv), 2
    t = synth.device.to_torch(p, "cuda")
    out = fb.backward(t["q"], t["k"], p.k_type, t["v"], p.v_type, t["dO"], H=p.H, Hkv=p.Hkv, D=p.D, Dv=p.Dv,
                      M=p.M, scale=p.scale, causal=p.causal, mask=t["mask"], mask_heads=p.mask_heads,
                      workspace_bytes=ws)
    torch.cuda.synchronize()
    assert fb.fa_back_get_error() == 0
    got = {k: v.cpu().numpy() for k, v in out.items()}
    res = check_components(got, oracle.fa_back(p))
    print(case, level, {k: v for k, v in kw.items() if k != "seed"}, res)


def draw_forward(case: int) -> dict:
    """A forward problem: a draw of the kind above without the score extensions; every third case
    with larger logits (Q sigma 3) and every third with per-row ranges of Q (so rows' running
    maxima move past the kernel's rescale threshold)."""
    kw = draw(3000 + case)
    for k in ("alibi", "softcap", "sinks"):
        kw.pop(k, None)
    rng = np.random.default_rng(94000 + case)
    if case % 3 == 1:
        kw.update(q_sigma=3.0)
    elif case % 3 == 2:
        kw.update(row_decades=float(rng.uniform(0.5, 1.5)))
    return kw


@pytest.mark.parametrize("case", range(N_FORWARD))
def test_fuzz_forward_against_the_oracle(fb, case):
    import oracle
    from metrics import NMSE_TOL, nmse
    kw = draw_forward(case)
    p = synth.make_problem(f"fuzzf{case}", **kw)
    t = synth.device.to_torch(p, "cuda")
    out = fb.forward(t["q"], t["k"], p.k_type, t["v"], p.v_type, H=p.H, Hkv=p.Hkv, D=p.D, Dv=p.Dv, M=p.M,
                     scale=p.scale, causal=p.causal, mask=t["mask"], mask_heads=p.mask_heads)
    torch.cuda.synchronize()
    assert fb.fa_back_get_error() == 0
    got = {k: v.cpu().numpy() for k, v in out.items()}
    ref = oracle.fa_forward(p)
    dead = ~np.isfinite(ref["lse"])
    assert np.array_equal(np.isneginf(got["lse"]), dead)
    assert np.all(got["O"][dead] == 0.0)
    res = {"lse": nmse(got["lse"], ref["lse"]), "O": nmse(got["O"], ref["O"])}
    print(case, {k: v for k, v in kw.items() if k != "seed"}, res)
    assert all(v <= NMSE_TOL for v in res.values()), res
