"""Host-side checks of the C ABI: the library loads, exports what the header declares, and
rejects bad arguments before touching a GPU."""
import os
import re

import pytest

import flash_attention_backward_gb300 as fb

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa_back.h")


@pytest.fixture(scope="module")
def L():
    from flash_attention_backward_gb300 import build
    build.build()
    return fb.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    assert declared_functions() == sorted(
        ["fa_back", "fa_back_batched", "fa_back_ext", "fa_back_get_error", "fa_back_noalloc", "fa_back_nocopy",
         "fa_back_plan_info", "fa_back_profile", "fa_back_workspace_size_nocopy",
         "fa_back_profile_read",
         "fa_back_selftest_timeout", "fa_back_status_string", "fa_back_strided", "fa_back_strided_workspace_size",
         "fa_back_test_wait_limit",
         "fa_back_workspace_size",
         "fa_back_with_stats", "fa_back_workspace_size_min", "fa_forward", "fa_forward_workspace_size",
         "fa_row_bytes"])


def test_every_declared_symbol_is_exported(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_row_bytes(L):
    assert fb.fa_row_bytes(fb.FA_F32, 256) == 1024
    assert fb.fa_row_bytes(fb.FA_F16, 128) == 256
    assert fb.fa_row_bytes(fb.FA_Q8_0, 256) == 8 * 34
    assert fb.fa_row_bytes(fb.FA_Q4_0, 256) == 8 * 18
    assert fb.fa_row_bytes(fb.FA_Q8_0, 48) == -1
    assert fb.fa_row_bytes(7, 64) == -1


def test_status_strings(L):
    for code in range(10):
        assert fb.fa_back_status_string(code)
    assert "unknown" in fb.fa_back_status_string(99)


def _call(**kw):
    a = dict(q=0x1000, k=0x2000, k_type=2, v=0x3000, v_type=2, mask=None, mask_heads=0, dO=0x4000, scale=0.1,
             N=8, M=32, H=4, Hkv=2, D=128, Dv=128, causal=0, dQ=0x5000, dK=0x6000, dV=0x7000, lse=0x8000,
             delta=0x9000, workspace=0x10000, workspace_bytes=1 << 30, stream=None)
    a.update(kw)
    return fb.fa_back(**a)


@pytest.mark.parametrize("kw,code", [
    (dict(k_type=9), "FA_ERR_TYPE"),
    (dict(v_type=-1), "FA_ERR_TYPE"),
    (dict(H=6, Hkv=4), "FA_ERR_SHAPE"),
    (dict(N=-1), "FA_ERR_SHAPE"),
    (dict(mask=0xA000, mask_heads=2), "FA_ERR_SHAPE"),
    (dict(D=96, Dv=96), "FA_ERR_UNSUPPORTED"),
    (dict(D=512), "FA_ERR_UNSUPPORTED"),
    (dict(q=None), "FA_ERR_NULL"),
    (dict(dV=None), "FA_ERR_NULL"),
    (dict(dQ=0x5004), "FA_ERR_ALIGN"),
    (dict(k=0x2002), "FA_ERR_ALIGN"),
])
def test_argument_errors_are_reported_before_any_launch(L, kw, code):
    assert fb.STATUS[_call(**kw)] == code


def _ext_call(**kw):
    a = dict(q=0x1000, k=0x2000, k_type=2, v=0x3000, v_type=2, mask=None, mask_heads=0, dO=0x4000, scale=0.1,
             N=8, M=32, H=4, Hkv=2, D=128, Dv=128, causal=0, alibi_slopes=None, softcap=0.0, sinks=None,
             dsinks=None, dQ=0x5000, dK=0x6000, dV=0x7000, lse=0x8000, delta=0x9000, workspace=0x10000,
             workspace_bytes=1 << 30, stream=None)
    a.update(kw)
    return fb.fa_back_ext(**a)


@pytest.mark.parametrize("kw,code", [
    (dict(softcap=-1.0), "FA_ERR_SHAPE"),
    (dict(softcap=float("nan")), "FA_ERR_SHAPE"),
    (dict(softcap=float("inf")), "FA_ERR_SHAPE"),
    (dict(alibi_slopes=0xB001), "FA_ERR_ALIGN"),
    (dict(sinks=0xB002), "FA_ERR_ALIGN"),
    (dict(sinks=0xB000, dsinks=0xC003), "FA_ERR_ALIGN"),
    (dict(k_type=9, softcap=1.0), "FA_ERR_TYPE"),
    (dict(q=None, sinks=0xB000), "FA_ERR_NULL"),
])
def test_ext_argument_errors_are_reported_before_any_launch(L, kw, code):
    assert fb.STATUS[_ext_call(**kw)] == code


def test_workspace_size_grows_with_the_problem(L):
    a = fb.fa_back_workspace_size(64, 512, 8, 2, 128, 128)
    b = fb.fa_back_workspace_size(2048, 75520, 24, 4, 256, 256)
    assert 0 < a < b
    assert fb.fa_back_workspace_size(8, 32, 6, 4, 64, 64) == 0  # H % Hkv != 0


def test_minimum_workspace_leaves_out_the_binary16_cache_copy(L):
    for N, M, H, Hkv, D, Dv in [(64, 512, 8, 2, 128, 128), (2048, 75520, 24, 4, 256, 256), (5, 1, 2, 1, 64, 64)]:
        full = fb.fa_back_workspace_size(N, M, H, Hkv, D, Dv)
        small = fb.fa_back_workspace_size_min(N, M, H, Hkv, D, Dv)
        assert 0 < small < full
        assert full - small >= 2 * Hkv * M * (D + Dv)


def test_with_stats_rejects_missing_or_misaligned_statistics(L):
    a = dict(q=0x1000, k=0x2000, k_type=2, v=0x3000, v_type=2, mask=None, mask_heads=0, dO=0x4000, lse=0x8000,
             delta=0x9000, scale=0.1, N=8, M=32, H=4, Hkv=2, D=128, Dv=128, causal=0, dQ=0x5000, dK=0x6000,
             dV=0x7000, workspace=0x10000, workspace_bytes=1 << 30, stream=None)
    assert fb.STATUS[fb.fa_back_with_stats(**dict(a, lse=None))] == "FA_ERR_NULL"
    assert fb.STATUS[fb.fa_back_with_stats(**dict(a, delta=None))] == "FA_ERR_NULL"
    assert fb.STATUS[fb.fa_back_with_stats(**dict(a, lse=0x8004))] == "FA_ERR_ALIGN"


def test_forward_workspace_and_argument_errors(L):
    assert 0 < fb.fa_forward_workspace_size(64, 512, 8, 2, 128, 128) < fb.fa_back_workspace_size(64, 512, 8, 2, 128, 128)
    a = dict(q=0x1000, k=0x2000, k_type=2, v=0x3000, v_type=2, mask=None, mask_heads=0, scale=0.1, N=8, M=32, H=4,
             Hkv=2, D=128, Dv=128, causal=0, O=0x5000, lse=0x8000, workspace=0x10000, workspace_bytes=1 << 30,
             stream=None)
    assert fb.STATUS[fb.fa_forward(**dict(a, O=None))] == "FA_ERR_NULL"
    assert fb.STATUS[fb.fa_forward(**dict(a, lse=None))] == "FA_ERR_NULL"
    assert fb.STATUS[fb.fa_forward(**dict(a, O=0x5004))] == "FA_ERR_ALIGN"
    assert fb.STATUS[fb.fa_forward(**dict(a, D=96, Dv=96))] == "FA_ERR_UNSUPPORTED"


def test_batched_rejects_a_negative_batch(L):
    rc = fb.fa_back_batched(-1, 0x1000, 0x2000, 2, 0x3000, 2, None, 0, 0, 0x4000, 0.1, 8, 32, 4, 2, 128, 128, 0,
                            0x5000, 0x6000, 0x7000, 0x8000, 0x9000, 0x10000, 1 << 30, None)
    assert fb.STATUS[rc] == "FA_ERR_SHAPE"


def _strided_call(**kw):
    st = fb.fa_strides(q_row=4 * 128, q_head=128, q_comp=1, do_row=4 * 128, do_head=128, do_comp=1, k_cell=2 * 136,
                       k_head=136, v_cell=2 * 136, v_head=136, mask_head=8 * 32, mask_row=32)
    for f in [f for f in kw if f in dict(fb.fa_strides._fields_)]:
        setattr(st, f, kw.pop(f))
    a = dict(q=0x1000, k=0x2000, k_type=2, v=0x3000, v_type=2, mask=None, mask_format=0, mask_heads=0, dO=0x4000,
             strides=st, scale=0.1, N=8, M=32, H=4, Hkv=2, D=128, Dv=128, causal=0, dQ=0x5000, dK=0x6000, dV=0x7000,
             lse=0x8000, delta=0x9000, workspace=0x10000, workspace_bytes=1 << 30, stream=None)
    a.update(kw)
    return fb.STATUS[fb.fa_back_strided(**a)]


@pytest.mark.parametrize("kw,code", [
    (dict(strides=None), "FA_ERR_NULL"),
    (dict(q_comp=-1), "FA_ERR_SHAPE"),
    (dict(k_head=-2), "FA_ERR_SHAPE"),
    (dict(mask=0xA000, mask_heads=4, mask_format=2), "FA_ERR_SHAPE"),
    (dict(mask=0xA000, mask_heads=3), "FA_ERR_SHAPE"),
    (dict(k_type=7), "FA_ERR_TYPE"),
    (dict(D=96, Dv=96), "FA_ERR_UNSUPPORTED"),
    (dict(dO=None), "FA_ERR_NULL"),
    (dict(q=0x1002), "FA_ERR_ALIGN"),
    (dict(k=0x2001), "FA_ERR_ALIGN"),
    (dict(v_cell=273), "FA_ERR_ALIGN"),
    (dict(mask=0xA002, mask_heads=1, mask_format=1), "FA_ERR_ALIGN"),
    (dict(dK=0x6008), "FA_ERR_ALIGN"),
])
def test_strided_argument_errors_are_reported_before_any_launch(L, kw, code):
    assert _strided_call(**kw) == code


def test_strided_accepts_views_that_fa_back_would_reject():
    """Unaligned and strided views pass the host checks; with no GPU here the call then stops at
    the device query (FA_ERR_CUDA), before anything is enqueued."""
    assert _strided_call(q=0x1004, dO=0x4008, k=0x2002, k_cell=3 * 136, q_comp=2) in ("FA_ERR_CUDA", "FA_ERR_DEVICE")
    assert _strided_call(mask=0xA002, mask_heads=4, mask_format=0) in ("FA_ERR_CUDA", "FA_ERR_DEVICE")


def test_strided_workspace_is_the_copies_plus_fa_backs(L):
    for N, M, H, Hkv, D, Dv, kt, vt, hm in [(64, 512, 8, 2, 128, 128, 2, 2, 0), (2048, 75520, 24, 4, 256, 256, 2, 2, 0),
                                            (40, 333, 4, 2, 128, 128, 3, 2, 4), (5, 1, 2, 1, 64, 64, 0, 1, 1)]:
        inner = fb.fa_back_workspace_size(N, M, H, Hkv, D, Dv)
        got = fb.fa_back_strided_workspace_size(N, M, H, Hkv, D, Dv, kt, vt, hm)
        copies = (4 * N * H * (D + Dv) + M * Hkv * (fb.fa_row_bytes(kt, D) + fb.fa_row_bytes(vt, Dv))
                  + 2 * hm * N * M)
        assert copies <= got - inner < copies + 5 * 256
    assert fb.fa_back_strided_workspace_size(8, 32, 4, 2, 48, 48, 2, 2, 0) == 0  # not a whole q8_0 block


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    """No CPU fallback: without libfa_back.so every entry point raises NativeLibraryMissing."""
    from flash_attention_backward_gb300 import _native
    monkeypatch.setattr(_native, "LIB_PATH", str(tmp_path / "libfa_back.so"))
    monkeypatch.setattr(_native, "_lib", None)
    with pytest.raises(_native.NativeLibraryMissing):
        _native.fa_back_workspace_size(8, 32, 4, 2, 128, 128)
    with pytest.raises(_native.NativeLibraryMissing):
        _native.fa_back(0x1000, 0x2000, 2, 0x3000, 2, None, 0, 0x4000, 0.1, 8, 32, 4, 2, 128, 128, 0, 0x5000,
                        0x6000, 0x7000, 0x8000, 0x9000, 0x10000, 1 << 30, None)


def test_product_path_imports_nothing_from_the_oracle():
    """The package and its sources never name the oracle: the CPU oracle is test infrastructure."""
    pkg = os.path.join(ROOT, "flash_attention_backward_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "fa_oracle" not in text and "liboracle" not in text, f


PLAN_SHAPES = [(2048, 75520, 24, 4, 256, 256), (64, 512, 8, 2, 128, 128), (40, 17000, 4, 2, 128, 128),
               (5, 1, 2, 1, 64, 64), (100, 40, 4, 1, 64, 64)]


@pytest.mark.parametrize("shape", PLAN_SHAPES)
def test_plan_levels_follow_the_workspace(L, shape):
    full = fb.fa_back_workspace_size(*shape)
    small = fb.fa_back_workspace_size_min(*shape)
    assert fb.fa_back_plan_info(*shape, full)[:2] == (0, 2) and fb.fa_back_plan_info(*shape, full)[3] == full
    assert fb.fa_back_plan_info(*shape, small) == (0, 0, 1, small)
    assert fb.STATUS[fb.fa_back_plan_info(*shape, small - 1)[0]] == "FA_ERR_WORKSPACE"
    # more workspace never gives a slower plan level, and a plan never uses more than it is given
    # (levels from slowest to fastest: 0, 1, 3, 2)
    speed = {0: 0, 1: 1, 3: 2, 2: 3}
    last = -1
    for f in [i / 16 for i in range(17)]:
        ws = int(small + f * (full - small))
        rc, level, splits, used = fb.fa_back_plan_info(*shape, ws)
        assert rc == 0 and speed[level] >= last and used <= ws and splits >= 1
        last = speed[level]
    # the plan without the cache copy needs less than the fastest plan and more than the smallest
    assert small < fb.fa_back_workspace_size_nocopy(*shape) < full


def test_plan_of_the_long_context_shape(L):
    shape = (2048, 75520, 24, 4, 256, 256)
    N, M, H, Hkv, D, Dv = shape
    copies = 2 * Hkv * M * (D + Dv)  # binary16 K'/V'
    ds = 2 * N * H * ((M + 63) // 64 * 64)  # binary16 dS
    _, level, _, used = fb.fa_back_plan_info(*shape, 2 << 30)  # room for the copies, not for dS
    assert level == 1 and copies <= used < ds
    _, level, _, used = fb.fa_back_plan_info(*shape, 1 << 40)
    assert level == 2 and used >= copies + ds
    # room for dS but not for the copies as well: dS stored, the raw cache decoded in every pass
    nocopy = fb.fa_back_workspace_size_nocopy(*shape)
    _, level, _, used = fb.fa_back_plan_info(*shape, nocopy)
    assert level == 3 and ds <= used == nocopy < ds + copies


def test_plan_info_argument_errors(L):
    assert fb.STATUS[fb.fa_back_plan_info(8, 32, 6, 4, 64, 64, 1 << 30)[0]] == "FA_ERR_SHAPE"
    assert fb.STATUS[fb.fa_back_plan_info(8, 32, 4, 2, 96, 96, 1 << 30)[0]] == "FA_ERR_UNSUPPORTED"
