"""The comparison helpers themselves (no GPU): the sink-gradient check's error model."""
import numpy as np
import pytest

from metrics import check_dsinks


def _ref():
    # two rows, one head: terms p_sink * delta of opposite signs that nearly cancel
    lse = np.array([[0.0], [0.0]])
    delta = np.array([[1.0], [-0.999]])
    sinks = np.array([0.0])  # p_sink = 1 for both rows
    return {"lse": lse, "delta": delta, "dsinks": np.array([-(1.0 - 0.999)])}, sinks


def test_exact_value_passes():
    ref, sinks = _ref()
    assert check_dsinks(ref["dsinks"].copy(), ref, sinks) == 0.0


def test_error_within_the_terms_bound_passes():
    ref, sinks = _ref()
    # 1e-4 of the terms' magnitude (1.999): NMSE about 4e-2, yet within delta's per-row error
    got = ref["dsinks"] + 1e-4 * 1.999
    check_dsinks(got, ref, sinks)


def test_error_beyond_the_terms_bound_fails():
    ref, sinks = _ref()
    got = ref["dsinks"] + 1e-3 * 1.999
    with pytest.raises(AssertionError):
        check_dsinks(got, ref, sinks)
