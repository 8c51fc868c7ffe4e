"""CUDA path vs the CPU oracle, element by element, through the C ABI.

Tolerance: NMSE <= 1e-5 per component (dQ, dK, dV, lse, delta tested separately), the bar the
pages' CPU-oracle comparison uses; lse = -inf positions must agree exactly and fully masked rows
must give delta = 0 and dQ = 0 exactly.
"""
import numpy as np
import pytest

import synth
from metrics import NMSE_TOL, check_components, nmse

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


def run_gpu(fb, p, ws=None, workspace_bytes=None, nocopy=False):
    t = synth.device.to_torch(p, "cuda")
    out = fb.backward(t["q"], t["k"], p.k_type, t["v"], p.v_type, t["dO"], H=p.H, Hkv=p.Hkv, D=p.D, Dv=p.Dv,
                      M=p.M, scale=p.scale, causal=p.causal, mask=t["mask"], mask_heads=p.mask_heads,
                      workspace=ws, workspace_bytes=workspace_bytes, nocopy=nocopy)
    torch.cuda.synchronize()
    assert fb.fa_back_get_error() == 0
    return {k: v.cpu().numpy() for k, v in out.items()}


def parity(fb, p, tol=NMSE_TOL, workspace_bytes=None, nocopy=False):
    import oracle
    ref = oracle.fa_back(p)
    got = run_gpu(fb, p, workspace_bytes=workspace_bytes, nocopy=nocopy)
    res = check_components(got, ref, tol)
    dead = ~np.isfinite(ref["lse"])
    assert np.all(got["dQ"][dead] == 0.0)
    return res


@pytest.mark.parametrize("cfg", ["0", "1", "1c", "1t", "2", "3"])
def test_configs(fb, cfg):
    p = synth.from_config(cfg)
    res = parity(fb, p)
    print(cfg, res)


EDGE = {
    # ragged rows and keys, several tiles, f16 cache, causal tail
    "ragged_f16_causal": dict(N=37, M=301, H=6, Hkv=2, D=128, Dv=128, k_type="f16", v_type="f16", causal=True),
    # more queries than keys under the causal tail: rows i < N-M see no key
    "n_gt_m_causal": dict(N=100, M=40, H=4, Hkv=1, D=64, Dv=64, k_type="q8_0", v_type="q8_0", causal=True),
    # Dv != D, mixed cache types
    "d256_dv128": dict(N=50, M=700, H=8, Hkv=2, D=256, Dv=128, k_type="q8_0", v_type="q4_0"),
    "d64_dv128_f32": dict(N=33, M=200, H=4, Hkv=4, D=64, Dv=128, k_type="f32", v_type="f32", causal=True),
    "d128_dv256": dict(N=20, M=150, H=3, Hkv=1, D=128, Dv=256, k_type="f16", v_type="q8_0"),
    # additive finite mask shared by all heads (Hm = 1) with -inf entries and dead rows
    "finite_mask_hm1": dict(N=40, M=333, H=4, Hkv=2, D=128, Dv=128, k_type="q4_0", v_type="q4_0",
                            mask="finite", mask_p=0.05, full_rows=3, mask_heads=1),
    # one key, one query
    "single_key": dict(N=5, M=1, H=2, Hkv=1, D=64, Dv=64, k_type="q8_0", v_type="q8_0"),
    "single_query": dict(N=1, M=257, H=8, Hkv=2, D=256, Dv=256, k_type="q8_0", v_type="q8_0", causal=True),
    # D = 64 everywhere (128-key tiles in every pass), q4_0 K, per-head mask with the causal tail,
    # several key splits and a ragged last tile
    "d64_q4_mask_causal": dict(N=200, M=3001, H=8, Hkv=2, D=64, Dv=64, k_type="q4_0", v_type="q8_0", causal=True,
                               mask="random", mask_p=0.05, full_rows=2, mask_heads=8),
    # D = 128 f16 K with q4_0 V, GQA 4, rows not a multiple of the 128-row tile
    "d128_f16k_q4v": dict(N=77, M=1500, H=16, Hkv=4, D=128, Dv=128, k_type="f16", v_type="q4_0"),
    # large-magnitude inputs (scales are chosen from the data)
    "big_values": dict(N=16, M=128, H=2, Hkv=1, D=64, Dv=64, k_type="f32", v_type="f32", q_sigma=300.0,
                       k_sigma=0.01, do_sigma=1e4, v_sigma=50.0),
    # small-magnitude binary16 K and q8_0 V: their power-of-two operand scales exceed 2^16, which
    # binary16 cannot hold (the decoders apply them in f32)
    "small_f16k_q8v": dict(N=40, M=300, H=4, Hkv=2, D=128, Dv=128, k_type="f16", v_type="q8_0", k_sigma=0.004,
                           v_sigma=0.003, causal=True),
}


@pytest.mark.parametrize("name", sorted(EDGE))
def test_edge_cases(fb, name):
    p = synth.make_problem(name, seed=2000 + sorted(EDGE).index(name), **EDGE[name])
    print(name, parity(fb, p))


# Shapes that stress the precision of delta: it is a softmax-weighted mean of dP_ij, so when the
# softmax of a row is spread over many keys it is small next to its terms.  Near-uniform rows come
# from Q scaled close to zero.  The row-range case multiplies every (i, h) row of Q and of dO by
# its own factor in [1e-3, 1e3] (the scale is reduced so that the largest rows' logits stay near
# one); rows with a small dO then depend on the per-row multiplier of dS in the dQ product.  The
# logit case doubles Q (logits about 2 in size), inside the envelope of single-pass binary16 S.
PRECISION = {
    "d64_q4v_17k": dict(N=256, M=17000, H=8, Hkv=2, D=64, Dv=64, k_type="q8_0", v_type="q4_0", causal=True),
    "uniform_d64_65k": dict(N=64, M=65536, H=8, Hkv=2, D=64, Dv=64, k_type="q8_0", v_type="q8_0", q_sigma=1e-3),
    "uniform_d256_65k": dict(N=32, M=65536, H=4, Hkv=1, D=256, Dv=256, k_type="q8_0", v_type="q8_0",
                             q_sigma=1e-3, causal=True),
    "row_range_d128": dict(N=128, M=4096, H=8, Hkv=2, D=128, Dv=128, k_type="q8_0", v_type="q4_0", causal=True,
                           row_decades=3.0, scale=1e-3 / 128 ** 0.5),
    "logits_x2_d128": dict(N=128, M=4096, H=8, Hkv=2, D=128, Dv=128, k_type="q8_0", v_type="q8_0", causal=True,
                           q_sigma=2.0),
}


def row_nmse(got, ref):
    """NMSE of every (i, h) row of a [N][H][D] output, each against its own reference row."""
    g = np.asarray(got, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    num = np.sum((g - r) ** 2, axis=-1)
    den = np.sum(r ** 2, axis=-1)
    return np.where(den > 0, num / np.where(den > 0, den, 1.0), np.where(num > 0, np.inf, 0.0))


@pytest.mark.parametrize("name", sorted(PRECISION))
def test_precision_cases(fb, name):
    import oracle
    p = synth.make_problem(name, seed=3000 + sorted(PRECISION).index(name), **PRECISION[name])
    ref = oracle.fa_back(p)
    got = run_gpu(fb, p)
    print(name, check_components(got, ref))
    # every query row on its own: no row of dQ may be hidden behind the large ones
    rn = row_nmse(got["dQ"], ref["dQ"])
    live = np.isfinite(ref["lse"])
    print(name, "worst dQ row NMSE", float(np.max(rn[live], initial=0.0)))
    assert np.all(rn[live] <= NMSE_TOL), float(np.max(rn[live]))


# The plan for the smallest workspace: row passes that decode the raw cache in shared memory.
@pytest.mark.parametrize("name", ["d256_dv128", "d64_q4_mask_causal", "ragged_f16_causal", "small_f16k_q8v",
                                  "finite_mask_hm1"])
def test_edge_cases_minimum_workspace(fb, name):
    p = synth.make_problem(name, seed=2000 + sorted(EDGE).index(name), **EDGE[name])
    wmin = fb.fa_back_workspace_size_min(p.N, p.M, p.H, p.Hkv, p.D, p.Dv)
    print(name, parity(fb, p, workspace_bytes=wmin))


@pytest.mark.parametrize("cfg", ["1", "3"])
def test_configs_minimum_workspace(fb, cfg):
    p = synth.from_config(cfg)
    wmin = fb.fa_back_workspace_size_min(p.N, p.M, p.H, p.Hkv, p.D, p.Dv)
    print(cfg, parity(fb, p, workspace_bytes=wmin))


# The plan that stores dS but keeps no decoded copy of the cache (level 3): every pass decodes raw
# cache tiles in shared memory, and dQ is one product over the stored dS (k_dq_raw, two row tiles
# per CTA).  Ragged tiles, both raw staging forms (rows of 16-byte multiples by TMA, others by
# 4-byte copies), key splits, the causal tail, Dv != D and masks.
NOCOPY_EDGE = ["ragged_f16_causal", "n_gt_m_causal", "d256_dv128", "d64_dv128_f32", "d128_dv256", "finite_mask_hm1",
               "single_key", "single_query", "d64_q4_mask_causal", "d128_f16k_q4v", "small_f16k_q8v"]


def nocopy_parity(fb, p):
    wn = fb.fa_back_workspace_size_nocopy(p.N, p.M, p.H, p.Hkv, p.D, p.Dv)
    assert 0 < wn < fb.fa_back_workspace_size(p.N, p.M, p.H, p.Hkv, p.D, p.Dv)
    fb.fa_back_profile(True)
    res = parity(fb, p, workspace_bytes=wn, nocopy=True)
    fb.fa_back_profile(False)
    launched = {k for k, v in fb.fa_back_profile_read().items() if v[1] > 0}
    assert "k_dq_raw" in launched and "k_predecode" not in launched, launched
    assert "k_rows_dq" not in launched and "k_dq_gemm" not in launched, launched
    return res


@pytest.mark.parametrize("cfg", ["0", "1", "1c", "1t", "2", "3"])
def test_configs_nocopy(fb, cfg):
    print(cfg, nocopy_parity(fb, synth.from_config(cfg)))


@pytest.mark.parametrize("name", NOCOPY_EDGE)
def test_edge_cases_nocopy(fb, name):
    p = synth.make_problem(name, seed=2000 + sorted(EDGE).index(name), **EDGE[name])
    print(name, nocopy_parity(fb, p))


@pytest.mark.parametrize("name", ["row_range_d128", "d64_q4v_17k"])
def test_precision_cases_nocopy(fb, name):
    import oracle
    p = synth.make_problem(name, seed=3000 + sorted(PRECISION).index(name), **PRECISION[name])
    ref = oracle.fa_back(p)
    got = run_gpu(fb, p, nocopy=True)
    print(name, check_components(got, ref))
    rn = row_nmse(got["dQ"], ref["dQ"])
    live = np.isfinite(ref["lse"])
    assert np.all(rn[live] <= NMSE_TOL), float(np.max(rn[live]))


def test_nocopy_reruns_are_bit_identical(fb):
    p = synth.from_config("3")
    a = run_gpu(fb, p, nocopy=True)
    b = run_gpu(fb, p, nocopy=True)
    for k in a:
        assert np.array_equal(a[k], b[k], equal_nan=True), k


def test_nocopy_below_its_workspace_runs_level_0(fb):
    p = synth.from_config("1")
    wmin = fb.fa_back_workspace_size_min(p.N, p.M, p.H, p.Hkv, p.D, p.Dv)
    fb.fa_back_profile(True)
    print(parity(fb, p, workspace_bytes=wmin, nocopy=True))
    fb.fa_back_profile(False)
    launched = {k for k, v in fb.fa_back_profile_read().items() if v[1] > 0}
    assert "k_rows_dq" in launched and "k_dq_raw" not in launched and "k_predecode" not in launched, launched


@pytest.mark.parametrize("N,M", [(0, 64), (16, 0)])
def test_empty_inputs(fb, N, M):
    p = synth.make_problem("empty", N=N, M=M, H=4, Hkv=2, D=128, Dv=128, k_type="q8_0", v_type="q8_0", seed=5)
    got = run_gpu(fb, p)
    assert np.all(got["dK"] == 0) and np.all(got["dV"] == 0)
    assert np.all(np.isneginf(got["lse"])) and np.all(got["delta"] == 0) and np.all(got["dQ"] == 0)


def test_bit_identical_reruns(fb):
    p = synth.from_config("3")
    a = run_gpu(fb, p)
    b = run_gpu(fb, p)
    for k in a:
        assert np.array_equal(a[k], b[k], equal_nan=True), k


def test_workspace_too_small_is_rejected(fb):
    p = synth.from_config("1")
    t = synth.device.to_torch(p, "cuda")
    need = fb.fa_back_workspace_size_min(p.N, p.M, p.H, p.Hkv, p.D, p.Dv)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    outs = [torch.empty(1 << 20, device="cuda") for _ in range(5)]
    rc = fb.fa_back(t["q"].data_ptr(), t["k"].data_ptr(), p.k_type, t["v"].data_ptr(), p.v_type, None, 0,
                    t["dO"].data_ptr(), p.scale, p.N, p.M, p.H, p.Hkv, p.D, p.Dv, 1,
                    *[o.data_ptr() for o in outs], ws.data_ptr(), need - 1, None)
    assert fb.STATUS[rc] == "FA_ERR_WORKSPACE"


@pytest.mark.slow
def test_long_context_sampled(fb):
    """N2048/M75520/H24/Hkv4/D256 q8_0, causal tail: every lse/delta, 64 dQ rows and 256 dK/dV
    key positions against the oracle, plus invariants over the whole output."""
    import oracle
    p = synth.from_config("4")
    got = run_gpu(fb, p)
    rows = synth.sample_indices(1004, synth.gen.S_SAMPLE, p.N, 64)
    keys = synth.sample_indices(1004, synth.gen.S_SAMPLE + 1, p.M, 256)
    ref = oracle.fa_back(p, dq_rows=rows, dkv_keys=keys)
    sub = {"lse": got["lse"], "delta": got["delta"], "dQ": got["dQ"][rows], "dK": got["dK"][keys],
           "dV": got["dV"][keys]}
    print(check_components(sub, ref))
    # sum_j dS_ij = 0  =>  sum_j dK_j = 0;  sum_j p_ij = 1  =>  sum_j dV_j = sum_i dO_i
    for hk in range(p.Hkv):
        sk = got["dK"][:, hk].astype(np.float64).sum(axis=0)
        scale_k = np.abs(got["dK"][:, hk].astype(np.float64)).sum(axis=0).max()
        assert np.max(np.abs(sk)) <= 1e-3 * scale_k
        want = p.dO[:, hk * p.G:(hk + 1) * p.G].astype(np.float64).sum(axis=(0, 1))
        assert nmse(got["dV"][:, hk].astype(np.float64).sum(axis=0), want) <= NMSE_TOL


# fa_back_with_stats: the row statistics (lse, delta) given, as from a forward pass.  They are
# the oracle's, so dQ, dK and dV are checked against the oracle at the same bar; the LSE pass
# must not run.
def with_stats(fb, p, workspace_bytes=None):
    import oracle
    ref = oracle.fa_back(p)
    t = synth.device.to_torch(p, "cuda")
    lse = torch.tensor(np.asarray(ref["lse"], dtype=np.float32), device="cuda").contiguous()
    delta = torch.tensor(np.asarray(ref["delta"], dtype=np.float32), device="cuda").contiguous()
    fb.fa_back_profile(True)
    out = fb.backward(t["q"], t["k"], p.k_type, t["v"], p.v_type, t["dO"], H=p.H, Hkv=p.Hkv, D=p.D, Dv=p.Dv,
                      M=p.M, scale=p.scale, causal=p.causal, mask=t["mask"], mask_heads=p.mask_heads,
                      workspace_bytes=workspace_bytes, lse=lse, delta=delta)
    torch.cuda.synchronize()
    fb.fa_back_profile(False)
    launched = {k for k, v in fb.fa_back_profile_read().items() if v[1] > 0}
    assert "k_stats_in" in launched and "k_rows_lse" not in launched, launched
    assert fb.fa_back_get_error() == 0
    assert set(out) == {"dQ", "dK", "dV"}
    got = {k: v.cpu().numpy() for k, v in out.items()}
    res = {n: nmse(got[n], ref[n]) for n in ("dQ", "dK", "dV")}
    assert all(v <= NMSE_TOL for v in res.values()), res
    dead = ~np.isfinite(ref["lse"])
    assert np.all(got["dQ"][dead] == 0.0)
    return res


@pytest.mark.parametrize("cfg", ["1", "1c", "3"])
def test_with_stats_configs(fb, cfg):
    print(cfg, with_stats(fb, synth.from_config(cfg)))


@pytest.mark.parametrize("name", ["n_gt_m_causal", "finite_mask_hm1", "d256_dv128", "ragged_f16_causal"])
def test_with_stats_edge_cases(fb, name):
    p = synth.make_problem(name, seed=2000 + sorted(EDGE).index(name), **EDGE[name])
    print(name, with_stats(fb, p))


def test_with_stats_minimum_workspace(fb):
    p = synth.from_config("3")
    print(with_stats(fb, p, fb.fa_back_workspace_size_min(p.N, p.M, p.H, p.Hkv, p.D, p.Dv)))


def test_with_stats_matches_fa_back_given_its_own_statistics(fb):
    """Feeding fa_back's own lse/delta outputs back gives fa_back's gradients (up to the rounding
    of lse and delta to f32)."""
    p = synth.from_config("3")
    t = synth.device.to_torch(p, "cuda")
    kw = dict(H=p.H, Hkv=p.Hkv, D=p.D, Dv=p.Dv, M=p.M, scale=p.scale, causal=p.causal, mask=t["mask"],
              mask_heads=p.mask_heads)
    a = fb.backward(t["q"], t["k"], p.k_type, t["v"], p.v_type, t["dO"], **kw)
    b = fb.backward(t["q"], t["k"], p.k_type, t["v"], p.v_type, t["dO"], lse=a["lse"], delta=a["delta"], **kw)
    torch.cuda.synchronize()
    for n in ("dQ", "dK", "dV"):
        assert nmse(b[n].cpu().numpy(), a[n].cpu().numpy()) <= 1e-9, n


def _stack(problems, key):
    arrs = [getattr(q, key) for q in problems]
    return None if arrs[0] is None else np.ascontiguousarray(np.stack(arrs))


def run_batched(fb, problems, mask_per_batch):
    p0 = problems[0]
    B = len(problems)
    dev = lambda a, dt=None: None if a is None else torch.from_numpy(a).to("cuda")
    q, k, v, dO = (dev(_stack(problems, n)) for n in ("q", "k", "v", "dO"))
    mask = dev(_stack(problems, "mask")) if mask_per_batch else dev(p0.mask)
    out = {"dQ": torch.empty((B, p0.N, p0.H, p0.D), device="cuda"),
           "dK": torch.empty((B, p0.M, p0.Hkv, p0.D), device="cuda"),
           "dV": torch.empty((B, p0.M, p0.Hkv, p0.Dv), device="cuda"),
           "lse": torch.empty((B, p0.N, p0.H), device="cuda"), "delta": torch.empty((B, p0.N, p0.H), device="cuda")}
    need = fb.fa_back_workspace_size(p0.N, p0.M, p0.H, p0.Hkv, p0.D, p0.Dv)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    rc = fb.fa_back_batched(B, q.data_ptr(), k.data_ptr(), p0.k_type, v.data_ptr(), p0.v_type,
                            None if mask is None else mask.data_ptr(), p0.mask_heads, int(mask_per_batch),
                            dO.data_ptr(), p0.scale, p0.N, p0.M, p0.H, p0.Hkv, p0.D, p0.Dv, int(p0.causal),
                            *[out[n].data_ptr() for n in ("dQ", "dK", "dV", "lse", "delta")], ws.data_ptr(), need,
                            torch.cuda.current_stream().cuda_stream)
    assert fb.STATUS[rc] == "FA_OK"
    torch.cuda.synchronize()
    assert fb.fa_back_get_error() == 0
    return {n: t.cpu().numpy() for n, t in out.items()}


def test_batched_slices_match_the_oracle(fb):
    import oracle
    shape = dict(N=64, M=512, H=8, Hkv=2, D=128, Dv=128, k_type="q8_0", v_type="q8_0", causal=True)
    problems = [synth.make_problem(f"b{b}", seed=6100 + b, **shape) for b in range(3)]
    got = run_batched(fb, problems, False)
    for b, p in enumerate(problems):
        ref = oracle.fa_back(p)
        print(b, check_components({n: got[n][b] for n in got}, ref))


def test_batched_per_batch_mask_equals_separate_calls(fb):
    shape = dict(N=40, M=333, H=4, Hkv=2, D=128, Dv=128, k_type="q4_0", v_type="q8_0", mask="random", mask_p=0.1,
                 full_rows=2, mask_heads=4)
    problems = [synth.make_problem(f"bm{b}", seed=6200 + b, **shape) for b in range(2)]
    got = run_batched(fb, problems, True)
    for b, p in enumerate(problems):
        one = run_gpu(fb, p)
        for n in one:
            assert np.array_equal(got[n][b], one[n], equal_nan=True), (b, n)


@pytest.mark.parametrize("name", ["gqa_causal_mask_worked_example.txt", "gqa_two_kv_heads_worked_example.txt"])
def test_golden_worked_example(fb, name):
    """The CUDA path against the hand-worked examples under tests/golden/ (GQA with one and with
    two KV heads, the causal tail, an additive and a -inf mask entry, a row without keys, a
    single-key row), embedded in D = Dv = 64 with zero components after the worked ones."""
    import golden_io
    fix = golden_io.load(name)
    p = golden_io.worked_problem(fix, 64)
    want = golden_io.worked_expected(fix, 64)
    got = run_gpu(fb, p)
    print(check_components(got, want))
    assert np.all(got["dQ"][~np.isfinite(want["lse"])] == 0.0)


def test_captured_in_a_cuda_graph_and_replayed(fb):
    """fa_back enqueues only kernels on the caller's stream (its host work, argument checks and
    tensor maps, runs at the call), so a CUDA graph captured around one call replays it: the
    replay's outputs equal a direct call's bit for bit, also after the inputs change in place."""
    p = synth.from_config("3")
    t = synth.device.to_torch(p, "cuda")
    kw = dict(H=p.H, Hkv=p.Hkv, D=p.D, Dv=p.Dv, M=p.M, scale=p.scale, causal=p.causal, mask=t["mask"],
              mask_heads=p.mask_heads)
    ws = fb.Workspace("cuda")
    ws.get(fb.fa_back_workspace_size(p.N, p.M, p.H, p.Hkv, p.D, p.Dv))
    direct = fb.backward(t["q"], t["k"], p.k_type, t["v"], p.v_type, t["dO"], workspace=ws, **kw)
    out = {k: torch.empty_like(v) for k, v in direct.items()}
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            fb.backward(t["q"], t["k"], p.k_type, t["v"], p.v_type, t["dO"], workspace=ws, out=out, **kw)
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    assert fb.fa_back_get_error() == 0
    for k in direct:
        assert torch.equal(out[k], direct[k]), k
    # new values in the captured input buffers: the replay follows them
    t["dO"].mul_(0.5)
    again = fb.backward(t["q"], t["k"], p.k_type, t["v"], p.v_type, t["dO"], workspace=fb.Workspace("cuda"), **kw)
    g.replay()
    torch.cuda.synchronize()
    for k in again:
        assert torch.equal(out[k], again[k]), k
