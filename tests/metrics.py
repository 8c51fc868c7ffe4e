"""Comparison helpers shared by the parity tests (no method arithmetic)."""
import numpy as np

NMSE_TOL = 1e-5  # per component, the tolerance the pages' CPU-oracle comparison uses


def nmse(got, ref) -> float:
    """sum (x - r)^2 / sum r^2 over the entries where the reference is finite."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    fin = np.isfinite(ref)
    if not np.all(np.isfinite(got[fin])):
        return float("inf")
    den = float(np.sum(ref[fin] ** 2))
    num = float(np.sum((got[fin] - ref[fin]) ** 2))
    if den == 0.0:
        return 0.0 if np.max(np.abs(got[fin]), initial=0.0) <= 1e-30 else float("inf")
    return num / den


def check_components(got: dict, ref: dict, tol: float = NMSE_TOL, names=("lse", "delta", "dQ", "dK", "dV")):
    """Assert NMSE <= tol per component, exact -inf agreement of lse, exact zeros of dead rows."""
    out = {}
    for n in names:
        out[n] = nmse(got[n], ref[n])
    lse_g, lse_r = np.asarray(got["lse"]), np.asarray(ref["lse"])
    dead = ~np.isfinite(lse_r)
    assert np.array_equal(np.isneginf(lse_g), np.isneginf(lse_r)), "lse -inf positions differ"
    if "delta" in got:
        assert np.all(np.asarray(got["delta"])[dead] == 0.0), "delta of fully masked rows is not 0"
    bad = {n: v for n, v in out.items() if not (v <= tol)}
    assert not bad, f"NMSE above {tol}: {bad} (all: {out})"
    return out


DSINKS_TERM_TOL = 3e-4  # delta's relative error per row at NMSE 1e-7: sqrt(1e-7)


def check_dsinks(got, ref: dict, sinks, tol: float = NMSE_TOL, term_tol: float = DSINKS_TERM_TOL) -> float:
    """dsinks_h = -sum_i p_sink(i, h) delta_ih is a sum whose terms can cancel (rows with deltas
    of both signs).  Accept NMSE <= tol, or, head by head, an error within term_tol of the sum of
    the terms' magnitudes: the bound that a per-row relative error of term_tol in delta gives.
    Returns the NMSE; raises AssertionError with the details otherwise."""
    got = np.asarray(got, dtype=np.float64)
    r = np.asarray(ref["dsinks"], dtype=np.float64)
    e = nmse(got, r)
    if e <= tol:
        return e
    lse = np.asarray(ref["lse"], dtype=np.float64)
    terms = np.exp(np.asarray(sinks, dtype=np.float64)[None, :] - lse) * np.asarray(ref["delta"], dtype=np.float64)
    mag = np.sum(np.where(np.isfinite(terms), np.abs(terms), 0.0), axis=0)
    err = np.abs(got - r)
    assert np.all(err <= term_tol * mag), f"dsinks NMSE {e}; errors {err} against {term_tol} x {mag}"
    return e

