"""The oracle against the hand-worked fixtures under tests/golden/.

Each fixture states its inputs, the passage its rules come from, and values worked out by hand
from those rules.  A dropped term, a wrong sign, a transposed GQA map or a wrong nibble order in
the oracle moves at least one value by far more than the tolerances here.
"""
import numpy as np
import pytest

import golden_io
import synth

WORKED = "gqa_causal_mask_worked_example.txt"


@pytest.mark.parametrize("D_pad", [0, 64])
def test_worked_example_backward(oracle_lib, D_pad):
    fix = golden_io.load(WORKED)
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
    # the fully masked row and the single-key row give exact zeros
    assert np.all(got["dQ"][0] == 0.0) and got["delta"][0, 1] == 0.0


def test_worked_example_forward(oracle_lib):
    fix = golden_io.load(WORKED)
    p = golden_io.worked_problem(fix)
    want = golden_io.worked_expected(fix)
    got = oracle_lib.fa_forward(p)
    assert np.array_equal(np.isneginf(got["lse"]), np.isneginf(want["lse"]))
    live = np.isfinite(want["lse"])
    assert np.allclose(got["lse"][live], want["lse"][live], rtol=0, atol=1e-7)
    assert np.allclose(got["O"], want["O"], rtol=0, atol=1e-7)
    assert np.all(got["O"][0, 1] == 0.0)


def test_worked_example_is_self_consistent():
    """The fixture's own sums: delta = dO.O per live row, sum_j dK_j = 0, sum_j dV_j = the live
    rows' dO summed (the working in the fixture, checked as arithmetic)."""
    fix = golden_io.load(WORKED)
    p = golden_io.worked_problem(fix)
    want = golden_io.worked_expected(fix)
    live = np.isfinite(want["lse"])
    dO = p.dO.astype(np.float64)
    assert np.allclose(np.sum(dO * want["O"], axis=-1)[live], want["delta"][live], atol=1e-12)
    assert np.allclose(want["dK"].sum(axis=0), 0.0, atol=1e-12)
    assert np.allclose(want["dV"].sum(axis=0)[0], dO[live].sum(axis=0), atol=1e-12)


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
