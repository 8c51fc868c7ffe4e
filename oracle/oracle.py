"""ctypes wrapper and gcc build of the C oracle (test infrastructure only)."""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fa_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def lib_path() -> str:
    return _LIB


def compile_source(src: str, out: str) -> str:
    """gcc -O3 shared library from one C file (no machine-specific flags)."""
    tmp = out + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-std=c11", "-O3", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
           "-Wall", "-Wextra", "-Wno-unused-parameter", src, "-o", tmp, "-lm"]
    subprocess.check_call(cmd)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile fa_oracle.c into liboracle.so."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        compile_source(_SRC, _LIB)
    return _LIB


def load(path: str):
    """Open a compiled oracle library and declare its entry points."""
    L = ctypes.CDLL(path)
    _declare(L)
    return L


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = load(_LIB)
    return _lib


def _declare(L):
    L.oracle_half_to_double.restype = ctypes.c_double
    L.oracle_half_to_double.argtypes = [ctypes.c_uint16]
    L.oracle_row_bytes.restype = ctypes.c_long
    L.oracle_row_bytes.argtypes = [ctypes.c_int, ctypes.c_int]
    L.oracle_dequant.restype = ctypes.c_int
    L.oracle_dequant.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p]
    L.oracle_default_threads.restype = ctypes.c_int
    L.oracle_fa_back.restype = ctypes.c_int
    L.oracle_fa_back.argtypes = (
        [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int,
         ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_double]
        + [ctypes.c_int] * 7
        + [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int]
        + [ctypes.c_void_p] * 5 + [ctypes.c_int])
    L.oracle_fa_back_ext.restype = ctypes.c_int
    L.oracle_fa_back_ext.argtypes = (
        [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int,
         ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_double]
        + [ctypes.c_int] * 7
        + [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int]
        + [ctypes.c_void_p] * 5 + [ctypes.c_void_p, ctypes.c_double, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int])
    L.oracle_fa_forward.restype = ctypes.c_int
    L.oracle_fa_forward.argtypes = (
        [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int,
         ctypes.c_double] + [ctypes.c_int] * 7 + [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int])


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def default_threads() -> int:
    return int(_load().oracle_default_threads())


def half_to_double(bits: int) -> float:
    return float(_load().oracle_half_to_double(int(bits) & 0xFFFF))


def dequant(raw: np.ndarray, type_: int, D: int) -> np.ndarray:
    """Decode raw rows (uint8 [..., row_bytes]) into float64 [..., D]."""
    L = _load()
    rb = L.oracle_row_bytes(type_, D)
    raw = np.ascontiguousarray(raw, dtype=np.uint8)
    assert raw.shape[-1] == rb, (raw.shape, rb)
    lead = raw.shape[:-1]
    nrows = int(np.prod(lead)) if lead else 1
    out = np.empty((nrows, D), dtype=np.float64)
    rc = L.oracle_dequant(_ptr(raw), type_, nrows, D, _ptr(out))
    if rc:
        raise ValueError("oracle_dequant failed")
    return out.reshape(*lead, D)


def fa_back(p, dq_rows: Optional[Sequence[int]] = None, dkv_keys: Optional[Sequence[int]] = None,
            nthreads: int = 0, want_dq: bool = True, want_dkv: bool = True, lib=None) -> dict:
    """Run the oracle on a synth.Problem.

    Returns float64 arrays: lse, delta [N][H]; dQ [n_dq][H][D];
    dK [n_keys][Hkv][D]; dV [n_keys][Hkv][Dv]; with the problem's optional
    extensions (ALiBi slopes, soft-cap, sink logits) also dsinks [H] when it
    has sink logits.
    """
    L = lib if lib is not None else _load()
    N, M, H, Hkv, D, Dv = p.N, p.M, p.H, p.Hkv, p.D, p.Dv
    q = np.ascontiguousarray(p.q, dtype=np.float32)
    dO = np.ascontiguousarray(p.dO, dtype=np.float32)
    k = np.ascontiguousarray(p.k, dtype=np.uint8)
    v = np.ascontiguousarray(p.v, dtype=np.uint8)
    mask = None if p.mask is None else np.ascontiguousarray(p.mask, dtype=np.uint16)
    rows = None if dq_rows is None else np.ascontiguousarray(np.asarray(dq_rows, dtype=np.int64))
    keys = None if dkv_keys is None else np.ascontiguousarray(np.asarray(dkv_keys, dtype=np.int64))
    nq = N if rows is None else rows.size
    nk = M if keys is None else keys.size
    lse = np.empty((N, H), dtype=np.float64)
    delta = np.empty((N, H), dtype=np.float64)
    dQ = np.empty((nq, H, D), dtype=np.float64) if want_dq else None
    dK = np.empty((nk, Hkv, D), dtype=np.float64) if want_dkv else None
    dV = np.empty((nk, Hkv, Dv), dtype=np.float64) if want_dkv else None
    alibi = getattr(p, "alibi", None)
    softcap = float(getattr(p, "softcap", 0.0) or 0.0)
    sinks = getattr(p, "sinks", None)
    common = [_ptr(q), _ptr(k), p.k_type, _ptr(v), p.v_type, _ptr(mask), p.mask_heads if mask is not None else 0,
              _ptr(dO), float(p.scale), N, M, H, Hkv, D, Dv, int(p.causal),
              _ptr(rows), 0 if rows is None else rows.size, _ptr(keys), 0 if keys is None else keys.size,
              _ptr(lse), _ptr(delta), _ptr(dQ), _ptr(dK), _ptr(dV)]
    out = {"lse": lse, "delta": delta, "dQ": dQ, "dK": dK, "dV": dV}
    if alibi is None and softcap == 0.0 and sinks is None:
        rc = L.oracle_fa_back(*common, int(nthreads))
    else:
        al = None if alibi is None else np.ascontiguousarray(alibi, dtype=np.float64)
        sk = None if sinks is None else np.ascontiguousarray(sinks, dtype=np.float64)
        ds = None if sinks is None else np.empty(H, dtype=np.float64)
        rc = L.oracle_fa_back_ext(*common, _ptr(al), softcap, _ptr(sk), _ptr(ds), int(nthreads))
        if ds is not None:
            out["dsinks"] = ds
    if rc:
        raise RuntimeError("oracle_fa_back failed with code %d" % rc)
    return out


def fa_forward(p, nthreads: int = 0, lib=None) -> dict:
    """Forward of a synth.Problem (dO unused): float64 lse [N][H] and O [N][H][Dv]."""
    L = lib if lib is not None else _load()
    N, M, H, Hkv, D, Dv = p.N, p.M, p.H, p.Hkv, p.D, p.Dv
    q = np.ascontiguousarray(p.q, dtype=np.float32)
    k = np.ascontiguousarray(p.k, dtype=np.uint8)
    v = np.ascontiguousarray(p.v, dtype=np.uint8)
    mask = None if p.mask is None else np.ascontiguousarray(p.mask, dtype=np.uint16)
    lse = np.empty((N, H), dtype=np.float64)
    O = np.empty((N, H, Dv), dtype=np.float64)
    rc = L.oracle_fa_forward(_ptr(q), _ptr(k), p.k_type, _ptr(v), p.v_type, _ptr(mask),
                             p.mask_heads if mask is not None else 0, float(p.scale), N, M, H, Hkv, D, Dv,
                             int(p.causal), _ptr(lse), _ptr(O), int(nthreads))
    if rc:
        raise RuntimeError("oracle_fa_forward failed with code %d" % rc)
    return {"lse": lse, "O": O}
