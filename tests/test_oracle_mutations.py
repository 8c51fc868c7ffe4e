"""The oracle's pins are strong enough to catch plausible mistakes.

Each case copies the oracle's C source, plants one mistake (a dropped term,
a wrong sign, a wrong index, a swapped operand), compiles the copy on the
CPU and checks that the torch float64 autograd pin rejects it, and that the
hand-worked fixtures under tests/golden/ reject it too.
"""
import os

import numpy as np
import pytest

import synth
from oracle import oracle as orc
from test_oracle_pins import rel_err, torch_reference

SRC = os.path.join(os.path.dirname(orc.__file__), "fa_oracle.c")

MUTATIONS = {
    "gqa_index_in_dq": ("const double* k = J->Kh + ((int64_t)j * Hkv + (h / G)) * D;",
                        "const double* k = J->Kh + ((int64_t)j * Hkv + (h % Hkv)) * D;"),
    "mask_term_dropped": ("  s += mv;", "  s += 0.0 * mv;"),
    "ds_sign": ("const double ds = p * (dp[j] - delta) * fac[j];", "const double ds = p * (dp[j] + delta) * fac[j];"),
    "causal_off_by_one": ("if (J->causal && (int64_t)j > (int64_t)J->M - J->N + i) return 0;",
                          "if (J->causal && (int64_t)j >= (int64_t)J->M - J->N + i) return 0;"),
    "dk_scale_dropped": ("dk[c] += J->scale * ds * q[c];", "dk[c] += ds * q[c];"),
    "dv_uses_ds": ("dv[c] += p * d[c];", "dv[c] += ds * d[c];"),
    "q4_nibbles_swapped": ("int lo = blk[2 + t] & 15, hi = blk[2 + t] >> 4;",
                           "int hi = blk[2 + t] & 15, lo = blk[2 + t] >> 4;"),
    "lse_max_dropped": ("const double lse = mx + log(sum);", "const double lse = log(sum);"),
    "dp_uses_k_in_phase2": ("for (int t = 0; t < RB; ++t) acc2[t] += oc * vc[t];",
                            "for (int t = 0; t < RB; ++t) acc2[t] += oc * (kt + (vc - vt))[t];"),
    "q8_scale_ignored": ("out[32 * b + t] = (double)(int8_t)blk[2 + t] * d;",
                         "out[32 * b + t] = (double)(int8_t)blk[2 + t] * 0.01;"),
}

# mistakes in the extensions, caught by the extension pin (ALiBi, soft-cap and sinks together)
EXT_MUTATIONS = {
    "softcap_derivative_dropped": ("*fac = 1.0 - t * t;", "*fac = 1.0;"),
    "alibi_sign": ("s += J->alibi[h] * ((double)j - ((double)J->M - J->N + i));",
                   "s -= J->alibi[h] * ((double)j - ((double)J->M - J->N + i));"),
    "alibi_position_from_row_start": ("s += J->alibi[h] * ((double)j - ((double)J->M - J->N + i));",
                                      "s += J->alibi[h] * ((double)j - (double)i);"),
    "sink_not_in_denominator": ("if (J->sinks) sum += exp(sink - mx);", "if (J->sinks) sum += 0.0;"),
    "sink_gradient_sign": ("acc -= exp(sinks[h] - lse[o]) * delta[o];", "acc += exp(sinks[h] - lse[o]) * delta[o];"),
    "softcap_inside_scale": ("const double t = tanh(raw / J->softcap);", "const double t = tanh(raw);"),
}


@pytest.fixture(scope="module")
def problem():
    return synth.make_problem("mut", N=9, M=33, H=4, Hkv=2, D=64, Dv=64, k_type="q4_0", v_type="q8_0",
                              mask="finite", mask_p=0.2, mask_heads=4, causal=True, seed=77)


def test_unmutated_copy_passes(problem, tmp_path):
    lib = orc.load(orc.compile_source(SRC, str(tmp_path / "lib_ok.so")))
    got = orc.fa_back(problem, lib=lib)
    ref = torch_reference(problem)
    assert max(rel_err(got[k], ref[k]) for k in ("lse", "delta", "dQ", "dK", "dV")) < 1e-12


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(problem, tmp_path, name):
    old, new = MUTATIONS[name]
    text = open(SRC).read()
    assert text.count(old) == 1, name
    src = tmp_path / f"mut_{name}.c"
    src.write_text(text.replace(old, new))
    lib = orc.load(orc.compile_source(str(src), str(tmp_path / f"lib_{name}.so")))
    got = orc.fa_back(problem, lib=lib)
    ref = torch_reference(problem)
    errs = {k: rel_err(np.nan_to_num(got[k], nan=1e30, posinf=1e30, neginf=-1e30),
                       np.nan_to_num(ref[k], nan=1e30, posinf=1e30, neginf=-1e30))
            for k in ("lse", "delta", "dQ", "dK", "dV")}
    assert max(errs.values()) > 1e-6, (name, errs)


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_fails_the_golden_fixtures(tmp_path, name):
    """The hand-worked fixtures under tests/golden/ alone reject every planted mistake."""
    import golden_io
    old, new = MUTATIONS[name]
    src = tmp_path / f"mut_{name}.c"
    src.write_text(open(SRC).read().replace(old, new))
    lib = orc.load(orc.compile_source(str(src), str(tmp_path / f"lib_{name}.so")))
    worst = 0.0
    for example in ("gqa_causal_mask_worked_example.txt", "gqa_two_kv_heads_worked_example.txt"):
        fix = golden_io.load(example)
        got = orc.fa_back(golden_io.worked_problem(fix), lib=lib)
        want = golden_io.worked_expected(fix)
        worst = max([worst] + [float(np.max(np.abs(np.nan_to_num(got[k], nan=1e30, posinf=1e30, neginf=-1e30)
                                                   - np.nan_to_num(want[k], nan=1e30, posinf=1e30, neginf=-1e30))))
                               for k in ("lse", "delta", "dQ", "dK", "dV")])
    blocks = golden_io.load("cache_blocks.txt")
    for block, t in (("q8_0 ramp", synth.TYPE_Q8_0), ("q4_0 nibble order", synth.TYPE_Q4_0)):
        raw = np.array([int(x, 16) for x in blocks[block]["bytes"].split()], dtype=np.uint8)
        out = np.empty((1, 32), dtype=np.float64)  # decoded by the mutated library
        assert lib.oracle_dequant(raw.ctypes.data, t, 1, 32, out.ctypes.data) == 0
        worst = max(worst, float(np.max(np.abs(out[0] - np.array(golden_io.vector(blocks[block]["values"]))))))
    assert worst > 0.1, (name, worst)


@pytest.fixture(scope="module")
def ext_problem():
    return synth.make_problem("mutx", N=9, M=33, H=4, Hkv=2, D=64, Dv=32, k_type="q4_0", v_type="q8_0",
                              mask="finite", mask_p=0.2, mask_heads=4, causal=True, alibi=True, softcap=2.0,
                              sinks=0.5, seed=78)


@pytest.mark.parametrize("name", sorted(EXT_MUTATIONS))
def test_planted_extension_mistake_is_caught(ext_problem, tmp_path, name):
    old, new = EXT_MUTATIONS[name]
    text = open(SRC).read()
    assert text.count(old) == 1, name
    src = tmp_path / f"mutx_{name}.c"
    src.write_text(text.replace(old, new))
    lib = orc.load(orc.compile_source(str(src), str(tmp_path / f"libx_{name}.so")))
    got = orc.fa_back(ext_problem, lib=lib)
    ref = torch_reference(ext_problem)
    worst = max(rel_err(got[k], ref[k]) for k in ("lse", "delta", "dQ", "dK", "dV", "dsinks"))
    assert worst > 1e-6, (name, worst)
