"""ctypes binding of libfa_back.so: the C ABI under the same names, argument marshalling only."""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfa_back.so")

FA_F32, FA_F16, FA_Q8_0, FA_Q4_0 = 0, 1, 2, 3
STATUS = {0: "FA_OK", 1: "FA_ERR_NULL", 2: "FA_ERR_TYPE", 3: "FA_ERR_SHAPE", 4: "FA_ERR_ALIGN",
          5: "FA_ERR_UNSUPPORTED", 6: "FA_ERR_DEVICE", 7: "FA_ERR_CUDA", 8: "FA_ERR_TIMEOUT",
          9: "FA_ERR_WORKSPACE"}

FA_MASK_F16, FA_MASK_BITS = 0, 1

_lib = None


class fa_strides(ctypes.Structure):
    """struct fa_strides of the header: element strides of Q and dO, byte strides of the K and V
    rows, word strides of the mask."""
    _fields_ = [(n, ctypes.c_int64) for n in ("q_row", "q_head", "q_comp", "do_row", "do_head", "do_comp",
                                             "k_cell", "k_head", "v_cell", "v_head", "mask_head", "mask_row")]


class NativeLibraryMissing(RuntimeError):
    """libfa_back.so is not built or cannot be loaded; there is no fallback path."""


def lib():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise NativeLibraryMissing(
            f"{LIB_PATH} is missing: build it with `python -m flash_attention_backward_gb300.build`")
    try:
        L = ctypes.CDLL(LIB_PATH)
    except OSError as e:  # pragma: no cover - depends on the machine
        raise NativeLibraryMissing(f"cannot load {LIB_PATH}: {e}") from e
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    L.fa_row_bytes.restype = ctypes.c_long
    L.fa_row_bytes.argtypes = [i, i]
    L.fa_back_workspace_size.restype = sz
    L.fa_back_workspace_size.argtypes = [i] * 6
    L.fa_back_workspace_size_min.restype = sz
    L.fa_back_workspace_size_min.argtypes = [i] * 6
    L.fa_back_plan_info.restype = i
    L.fa_back_plan_info.argtypes = [i] * 6 + [sz, vp, vp, vp]
    L.fa_back.restype = i
    L.fa_back.argtypes = [vp, vp, i, vp, i, vp, i, vp, f, i, i, i, i, i, i, i, vp, vp, vp, vp, vp, vp, sz, vp]
    L.fa_back_nocopy.restype = i
    L.fa_back_nocopy.argtypes = [vp, vp, i, vp, i, vp, i, vp, f, i, i, i, i, i, i, i, vp, vp, vp, vp, vp, vp, sz, vp]
    L.fa_back_workspace_size_nocopy.restype = sz
    L.fa_back_workspace_size_nocopy.argtypes = [i] * 6
    L.fa_back_ext.restype = i
    L.fa_back_ext.argtypes = [vp, vp, i, vp, i, vp, i, vp, f, i, i, i, i, i, i, i, vp, f, vp, vp, vp, vp, vp, vp, vp,
                              vp, sz, vp]
    L.fa_back_with_stats.restype = i
    L.fa_back_with_stats.argtypes = [vp, vp, i, vp, i, vp, i, vp, vp, vp, f, i, i, i, i, i, i, i, vp, vp, vp, vp, sz,
                                     vp]
    L.fa_back_batched.restype = i
    L.fa_back_batched.argtypes = [i, vp, vp, i, vp, i, vp, i, i, vp, f, i, i, i, i, i, i, i, vp, vp, vp, vp, vp, vp,
                                  sz, vp]
    L.fa_back_strided_workspace_size.restype = sz
    L.fa_back_strided_workspace_size.argtypes = [i] * 9
    L.fa_back_strided.restype = i
    L.fa_back_strided.argtypes = [vp, vp, i, vp, i, vp, i, i, vp, ctypes.POINTER(fa_strides), f, i, i, i, i, i, i, i,
                                  vp, vp, vp, vp, vp, vp, sz, vp]
    L.fa_forward_workspace_size.restype = sz
    L.fa_forward_workspace_size.argtypes = [i] * 6
    L.fa_forward.restype = i
    L.fa_forward.argtypes = [vp, vp, i, vp, i, vp, i, f, i, i, i, i, i, i, i, vp, vp, vp, sz, vp]
    L.fa_back_get_error.restype = i
    L.fa_back_get_error.argtypes = []
    L.fa_back_status_string.restype = ctypes.c_char_p
    L.fa_back_status_string.argtypes = [i]
    L.fa_back_noalloc.restype = i
    L.fa_back_noalloc.argtypes = [vp, vp, i, vp, i, vp, i, vp, f, i, i, i, i, i, i, i, vp, vp, vp, vp, vp, vp]
    L.fa_back_test_wait_limit.restype = i
    L.fa_back_test_wait_limit.argtypes = [ctypes.c_ulonglong]
    L.fa_back_selftest_timeout.restype = i
    L.fa_back_selftest_timeout.argtypes = [ctypes.c_ulonglong, vp]
    L.fa_back_profile.restype = i
    L.fa_back_profile.argtypes = [i]
    L.fa_back_profile_read.restype = i
    L.fa_back_profile_read.argtypes = [vp, vp, vp, i]
    _lib = L
    return L


def fa_row_bytes(type_: int, D: int) -> int:
    return int(lib().fa_row_bytes(type_, D))


def fa_back_workspace_size(N: int, M: int, H: int, Hkv: int, D: int, Dv: int) -> int:
    return int(lib().fa_back_workspace_size(N, M, H, Hkv, D, Dv))


def fa_back_workspace_size_min(N: int, M: int, H: int, Hkv: int, D: int, Dv: int) -> int:
    return int(lib().fa_back_workspace_size_min(N, M, H, Hkv, D, Dv))


def fa_back_plan_info(N: int, M: int, H: int, Hkv: int, D: int, Dv: int, workspace_bytes: int):
    """(status, level, key_splits, plan_bytes) of the plan fa_back runs with this workspace."""
    level, splits, nbytes = ctypes.c_int(-1), ctypes.c_int(0), ctypes.c_size_t(0)
    rc = int(lib().fa_back_plan_info(N, M, H, Hkv, D, Dv, workspace_bytes, ctypes.byref(level), ctypes.byref(splits),
                                     ctypes.byref(nbytes)))
    return rc, level.value, splits.value, nbytes.value


def fa_back(q, k, k_type, v, v_type, mask, mask_heads, dO, scale, N, M, H, Hkv, D, Dv, causal,
            dQ, dK, dV, lse, delta, workspace, workspace_bytes, stream) -> int:
    """Direct call of the C entry point; pointers are integers (device addresses) or None."""
    return int(lib().fa_back(q, k, k_type, v, v_type, mask, mask_heads, dO, float(scale), N, M, H, Hkv, D, Dv,
                             int(causal), dQ, dK, dV, lse, delta, workspace, workspace_bytes, stream))


def fa_back_nocopy(q, k, k_type, v, v_type, mask, mask_heads, dO, scale, N, M, H, Hkv, D, Dv, causal,
                   dQ, dK, dV, lse, delta, workspace, workspace_bytes, stream) -> int:
    """fa_back restricted to the plans without a decoded copy of the cache (levels 3 and 0)."""
    return int(lib().fa_back_nocopy(q, k, k_type, v, v_type, mask, mask_heads, dO, float(scale), N, M, H, Hkv, D,
                                    Dv, int(causal), dQ, dK, dV, lse, delta, workspace, workspace_bytes, stream))


def fa_back_workspace_size_nocopy(N: int, M: int, H: int, Hkv: int, D: int, Dv: int) -> int:
    return int(lib().fa_back_workspace_size_nocopy(N, M, H, Hkv, D, Dv))


def fa_back_ext(q, k, k_type, v, v_type, mask, mask_heads, dO, scale, N, M, H, Hkv, D, Dv, causal,
                alibi_slopes, softcap, sinks, dsinks, dQ, dK, dV, lse, delta, workspace, workspace_bytes,
                stream) -> int:
    """fa_back with the score extensions (ALiBi slopes, soft cap, sink logits); see the header."""
    return int(lib().fa_back_ext(q, k, k_type, v, v_type, mask, mask_heads, dO, float(scale), N, M, H, Hkv, D, Dv,
                                 int(causal), alibi_slopes, float(softcap), sinks, dsinks, dQ, dK, dV, lse, delta,
                                 workspace, workspace_bytes, stream))


def fa_back_with_stats(q, k, k_type, v, v_type, mask, mask_heads, dO, lse, delta, scale, N, M, H, Hkv, D, Dv,
                       causal, dQ, dK, dV, workspace, workspace_bytes, stream) -> int:
    return int(lib().fa_back_with_stats(q, k, k_type, v, v_type, mask, mask_heads, dO, lse, delta, float(scale), N,
                                        M, H, Hkv, D, Dv, int(causal), dQ, dK, dV, workspace, workspace_bytes,
                                        stream))


def fa_back_batched(B, q, k, k_type, v, v_type, mask, mask_heads, mask_per_batch, dO, scale, N, M, H, Hkv, D, Dv,
                    causal, dQ, dK, dV, lse, delta, workspace, workspace_bytes, stream) -> int:
    return int(lib().fa_back_batched(B, q, k, k_type, v, v_type, mask, mask_heads, int(mask_per_batch), dO,
                                     float(scale), N, M, H, Hkv, D, Dv, int(causal), dQ, dK, dV, lse, delta,
                                     workspace, workspace_bytes, stream))


def fa_back_strided_workspace_size(N: int, M: int, H: int, Hkv: int, D: int, Dv: int, k_type: int, v_type: int,
                                   mask_heads: int) -> int:
    return int(lib().fa_back_strided_workspace_size(N, M, H, Hkv, D, Dv, k_type, v_type, mask_heads))


def fa_back_strided(q, k, k_type, v, v_type, mask, mask_format, mask_heads, dO, strides, scale, N, M, H, Hkv, D, Dv,
                    causal, dQ, dK, dV, lse, delta, workspace, workspace_bytes, stream) -> int:
    """strides: an fa_strides, or None for a NULL pointer."""
    st = None if strides is None else ctypes.byref(strides)
    return int(lib().fa_back_strided(q, k, k_type, v, v_type, mask, mask_format, mask_heads, dO, st, float(scale), N,
                                     M, H, Hkv, D, Dv, int(causal), dQ, dK, dV, lse, delta, workspace,
                                     workspace_bytes, stream))


def fa_forward_workspace_size(N: int, M: int, H: int, Hkv: int, D: int, Dv: int) -> int:
    return int(lib().fa_forward_workspace_size(N, M, H, Hkv, D, Dv))


def fa_forward(q, k, k_type, v, v_type, mask, mask_heads, scale, N, M, H, Hkv, D, Dv, causal, O, lse,
               workspace, workspace_bytes, stream) -> int:
    return int(lib().fa_forward(q, k, k_type, v, v_type, mask, mask_heads, float(scale), N, M, H, Hkv, D, Dv,
                                int(causal), O, lse, workspace, workspace_bytes, stream))


def fa_back_get_error() -> int:
    return int(lib().fa_back_get_error())


def fa_back_status_string(status: int) -> str:
    return lib().fa_back_status_string(status).decode()


def fa_back_profile(enable: bool) -> int:
    return int(lib().fa_back_profile(1 if enable else 0))


def fa_back_profile_read(max_kernels: int = 32) -> dict:
    """{kernel name: (summed ms, launches)} of the recorded fa_back calls; clears the record."""
    ms = (ctypes.c_float * max_kernels)()
    cnt = (ctypes.c_int * max_kernels)()
    names = (ctypes.c_char_p * max_kernels)()
    n = int(lib().fa_back_profile_read(ms, cnt, names, max_kernels))
    return {names[k].decode(): (float(ms[k]), int(cnt[k])) for k in range(n) if cnt[k] > 0}


NOALLOC_SCRATCH_BYTES = 64 << 20


def fa_back_noalloc(q, k, k_type, v, v_type, mask, mask_heads, dO, scale, N, M, H, Hkv, D, Dv, causal,
                    dQ, dK, dV, lse, delta, stream) -> int:
    """fa_back with the library's static scratch instead of a caller workspace (see the header)."""
    return int(lib().fa_back_noalloc(q, k, k_type, v, v_type, mask, mask_heads, dO, float(scale), N, M, H, Hkv,
                                     D, Dv, int(causal), dQ, dK, dV, lse, delta, stream))


def fa_back_selftest_timeout(limit_ns: int, stream=None) -> int:
    return int(lib().fa_back_selftest_timeout(limit_ns, stream))


def fa_back_test_wait_limit(limit_ns: int) -> int:
    """Failure-detection hook: the next call's kernels give up on waits longer than limit_ns."""
    return int(lib().fa_back_test_wait_limit(limit_ns))
