"""The oracle against the hand-worked fixtures under tests/golden/.

Each fixture states its inputs, the passage its rules come from, and values worked out by hand
from those rules.  A dropped term, a wrong sign, a transposed GQA map or a wrong nibble order in
the oracle moves at least one value by far more than the tolerances here.
"""
import numpy as np
import pytest

import golden_io
import synth

WORKED_EXAMPLES = ["gqa_causal_mask_worked_example.txt", "gqa_two_kv_heads_worked_example.txt"]


@pytest.mark.parametrize("D_pad", [0, 64])
@pytest.mark.parametrize("name", WORKED_EXAMPLES)
def test_worked_example_backward(oracle_lib, name, D_pad):
    fix = golden_io.load(name)
    p = golden_io.worked_problem(fix, D_pad)
    want = golden_io.worked_expected(fix, D_pad)
    got = oracle_lib.fa_back(p)
    # the only rounded input is q[1][0] = 2 log 3 as f32 (relative error 2^-24): its effect on every
    # output is below 1e-7, while a wrong term, sign or scale moves some output by more than 0.1
    assert np.array_equal(np.isneginf(got["lse"]), np.isneginf(want["lse"]))
    live = np.isfinite(want["lse"])
    assert np.allclose(got["lse"][live], want["lse"][live], rtol=0, atol=1e-7)
    for n in ("delta", "dQ", "dK", "dV"):
        assert np.allclose(got[n], want[n], rtol=0, atol=1e-7), (n, got[n], want[n])
    # a fully masked row gives exact zeros
    dead = ~live
    assert np.all(got["dQ"][dead] == 0.0) and np.all(got["delta"][dead] == 0.0)


@pytest.mark.parametrize("name", WORKED_EXAMPLES)
def test_worked_example_forward(oracle_lib, name):
    fix = golden_io.load(name)
    p = golden_io.worked_problem(fix)
    want = golden_io.worked_expected(fix)
    got = oracle_lib.fa_forward(p)
    assert np.array_equal(np.isneginf(got["lse"]), np.isneginf(want["lse"]))
    live = np.isfinite(want["lse"])
    assert np.allclose(got["lse"][live], want["lse"][live], rtol=0, atol=1e-7)
    assert np.allclose(got["O"], want["O"], rtol=0, atol=1e-7)
    assert np.all(got["O"][~live] == 0.0)


@pytest.mark.parametrize("name", WORKED_EXAMPLES)
def test_worked_example_is_self_consistent(name):
    """The fixture's own sums: delta = dO.O per live row, sum_j dK_j = 0 and sum_j dV_j = the
    live rows' dO summed over each KV head's group (the working in the fixture, checked as
    arithmetic)."""
    fix = golden_io.load(name)
    p = golden_io.worked_problem(fix)
    want = golden_io.worked_expected(fix)
    live = np.isfinite(want["lse"])
    dO = p.dO.astype(np.float64)
    assert np.allclose(np.sum(dO * want["O"], axis=-1)[live], want["delta"][live], atol=1e-12)
    assert np.allclose(want["dK"].sum(axis=0), 0.0, atol=1e-12)
    for hk in range(p.Hkv):
        heads = slice(hk * p.G, (hk + 1) * p.G)
        live_dO = dO[:, heads][live[:, heads]]
        assert np.allclose(want["dV"].sum(axis=0)[hk], live_dO.sum(axis=0), atol=1e-12)


@pytest.mark.parametrize("block,t", [("q8_0 ramp", synth.TYPE_Q8_0),
                                     ("q8_0 negative subnormal scale", synth.TYPE_Q8_0),
                                     ("q4_0 nibble order", synth.TYPE_Q4_0)])
def test_cache_blocks_decode_to_the_worked_values(oracle_lib, block, t):
    sec = golden_io.load("cache_blocks.txt")[block]
    raw = np.array([int(x, 16) for x in sec["bytes"].split()], dtype=np.uint8)
    want = np.array(golden_io.vector(sec["values"]))
    assert raw.size == synth.row_bytes(t, 32) and want.size == 32
    got = oracle_lib.dequant(raw[None, :], t, 32)[0]
    assert np.array_equal(got, want), (got, want)
