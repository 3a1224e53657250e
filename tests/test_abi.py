"""CPU checks of the C ABI: the library loads without a GPU, exports every
entry point include/fa.h declares, and rejects invalid arguments before it
touches the device."""

import ctypes
import os
import re

import pytest

from exact_attention_16_gb300 import api

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    text = open(os.path.join(ROOT, "include", "fa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\*?(fa_\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(api.library_path()):
        from exact_attention_16_gb300 import build
        build.build()
    return api.lib()


def test_header_declares_the_boundary():
    names = header_functions()
    assert {"fa_fwd", "fa_status", "fa_status_string", "fa_version"} <= set(names)


def test_library_exports_every_declared_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), name
        assert name in api.EXPORTED_SYMBOLS, name


def test_version_and_status_strings(lib):
    assert api.fa_version() >= 100
    assert api.fa_status_string(0) == "FA_OK"
    assert api.fa_status_string(4) == "FA_ERR_TIMEOUT"
    assert api.fa_status_string(99) == "FA_ERR_UNKNOWN"


def _call(lib, **kw):
    args = dict(q=16, k=16, v=16, o=16, lse=None, B=1, Sq=4, Sk=4, Hq=2, Hkv=1, D=128,
                scale=0.125, causal=0, dtype=1, stream=None)
    args.update(kw)
    return lib.fa_fwd(args["q"], args["k"], args["v"], args["o"], args["lse"], args["B"], args["Sq"],
                      args["Sk"], args["Hq"], args["Hkv"], args["D"], ctypes.c_float(args["scale"]),
                      args["causal"], args["dtype"], args["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(B=-1), api.FA_ERR_INVALID_ARG),
    (dict(Sq=-3), api.FA_ERR_INVALID_ARG),
    (dict(Sk=-1), api.FA_ERR_INVALID_ARG),
    (dict(Hq=3, Hkv=2), api.FA_ERR_INVALID_ARG),
    (dict(Hkv=0), api.FA_ERR_INVALID_ARG),
    (dict(dtype=2), api.FA_ERR_INVALID_ARG),
    (dict(causal=2), api.FA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), api.FA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), api.FA_ERR_INVALID_ARG),
    (dict(scale=3.0e38), api.FA_ERR_UNSUPPORTED),   # scale * log2(e) is not a finite float
    (dict(scale=-3.0e38), api.FA_ERR_UNSUPPORTED),
    (dict(scale=0.0, B=0), api.FA_OK),          # any finite scale passes the checks (B = 0: no launch)
    (dict(scale=-0.5, B=0), api.FA_OK),
    (dict(scale=-2.0e38, B=0), api.FA_OK),
    (dict(q=None), api.FA_ERR_INVALID_ARG),
    (dict(o=None), api.FA_ERR_INVALID_ARG),
    (dict(k=None), api.FA_ERR_INVALID_ARG),
    (dict(q=24), api.FA_ERR_INVALID_ARG),       # not 16-byte aligned
    (dict(v=8), api.FA_ERR_INVALID_ARG),
    (dict(lse=2), api.FA_ERR_INVALID_ARG),      # not 4-byte aligned
    (dict(D=40), api.FA_ERR_UNSUPPORTED),    # not a multiple of 16
    (dict(D=8), api.FA_ERR_UNSUPPORTED),
    (dict(D=272), api.FA_ERR_UNSUPPORTED),
    (dict(D=256, Hq=258, Hkv=1), api.FA_ERR_UNSUPPORTED),   # D = 256 takes at most 128 heads per KV head
    (dict(B=0), api.FA_OK),                     # nothing to do: no device call
    (dict(Sq=0), api.FA_OK),
    (dict(Hq=0, Hkv=1), api.FA_OK),
])
def test_invalid_arguments_are_rejected_before_any_launch(lib, kw, code):
    assert _call(lib, **kw) == code


def test_sk_zero_needs_no_kv_pointers_but_still_validates(lib):
    assert _call(lib, Sk=0, k=None, v=None, D=72) == api.FA_ERR_UNSUPPORTED


def test_debug_fault_hook_validates(lib):
    assert api.fa_debug_set_fault(-2) == api.FA_ERR_INVALID_ARG
    assert api.fa_debug_set_fault(-1) == api.FA_OK


def test_debug_schedule_hook_validates(lib):
    assert api.fa_debug_set_schedule(2) == api.FA_ERR_INVALID_ARG
    assert api.fa_debug_set_schedule(-2) == api.FA_ERR_INVALID_ARG
    for mode in (1, 0, -1):
        assert api.fa_debug_set_schedule(mode) == api.FA_OK


def _call_strided(lib, qs=None, ks=None, vs=None, os_=None, **kw):
    args = dict(q=16, k=16, v=16, o=16, lse=None, B=2, Sq=4, Sk=4, Hq=2, Hkv=1, D=128,
                scale=0.125, causal=0, dtype=1, stream=None)
    args.update(kw)
    arr = lambda x: None if x is None else (ctypes.c_longlong * 3)(*x)
    nat_q = (args["Sq"] * args["Hq"] * 128, args["Hq"] * 128, 128)
    nat_k = (args["Sk"] * args["Hkv"] * 128, args["Hkv"] * 128, 128)
    return lib.fa_fwd_strided(args["q"], args["k"], args["v"], args["o"], args["lse"], args["B"], args["Sq"],
                              args["Sk"], args["Hq"], args["Hkv"], args["D"],
                              arr(nat_q if qs is None else qs), arr(nat_k if ks is None else ks),
                              arr(nat_k if vs is None else vs), arr(nat_q if os_ is None else os_),
                              ctypes.c_float(args["scale"]), args["causal"], args["dtype"], args["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(qs=(1024, 256, 100)), api.FA_ERR_INVALID_ARG),     # head stride not a 16-byte multiple
    (dict(ks=(0, 128, 128)), api.FA_ERR_INVALID_ARG),        # zero batch stride with B > 1
    (dict(os_=(1024, -256, 128)), api.FA_ERR_INVALID_ARG),   # negative stride
    (dict(B=0), api.FA_OK),
])
def test_strided_entry_validates_strides(lib, kw, code):
    assert _call_strided(lib, **kw) == code


def test_strided_entry_rejects_null_strides(lib):
    rc = lib.fa_fwd_strided(16, 16, 16, 16, None, 1, 4, 4, 2, 1, 128, None, None, None, None,
                            ctypes.c_float(0.125), 0, 1, None)
    assert rc == api.FA_ERR_INVALID_ARG


@pytest.mark.parametrize("args,code", [
    ((16, 16, 0, 16, None, 1, 4, 2, 128, 1), api.FA_ERR_INVALID_ARG),   # n_parts = 0
    ((16, 16, 2, 16, None, 1, 4, 2, 124, 1), api.FA_ERR_UNSUPPORTED),   # D not a multiple of 16
    ((16, 16, 2, 16, None, 1, 4, 2, 128, 3), api.FA_ERR_INVALID_ARG),   # dtype
    ((None, 16, 2, 16, None, 1, 4, 2, 128, 1), api.FA_ERR_INVALID_ARG),
    ((24, 16, 2, 16, None, 1, 4, 2, 128, 1), api.FA_ERR_INVALID_ARG),   # misaligned parts
    ((16, 16, 2, 16, None, 0, 4, 2, 128, 1), api.FA_OK),                # nothing to merge
])
def test_merge_validates_before_any_launch(lib, args, code):
    assert lib.fa_merge(*args, None) == code


def test_decode_workspace_size_formula(lib):
    out = ctypes.c_ulonglong(7)
    # explicit 4 splits of 2048 keys (16 tiles): 4 x rows x (D + 1) floats, LSE part padded to 16 bytes
    assert lib.fa_decode_workspace_size(2, 1, 2048, 32, 4, 128, 4, ctypes.byref(out)) == api.FA_OK
    rows = 2 * 1 * 32
    assert out.value == 4 * rows * 128 * 4 + (4 * rows * 4 + 15) // 16 * 16
    # one split: no workspace
    assert lib.fa_decode_workspace_size(2, 1, 2048, 32, 4, 128, 1, ctypes.byref(out)) == api.FA_OK
    assert out.value == 0
    # more splits than key tiles are clamped to the tile count (2 tiles)
    assert lib.fa_decode_workspace_size(1, 1, 200, 8, 8, 64, 9, ctypes.byref(out)) == api.FA_OK
    assert out.value == 2 * 8 * 64 * 4 + (2 * 8 * 4 + 15) // 16 * 16


@pytest.mark.parametrize("args,code", [
    ((1, 17, 100, 256, 1, 128, 0), api.FA_ERR_UNSUPPORTED),   # 256 query heads per KV head > 128 rows
    ((1, 1, 100, 6, 4, 128, 0), api.FA_ERR_INVALID_ARG),      # Hq not a multiple of Hkv
    ((1, 1, 100, 8, 8, 72, 0), api.FA_ERR_UNSUPPORTED),       # D not a multiple of 16
])
def test_decode_size_checks(lib, args, code):
    out = ctypes.c_ulonglong(0)
    assert lib.fa_decode_workspace_size(*args, ctypes.byref(out)) == code


def test_decode_rejects_before_any_launch(lib):
    c = lambda **kw: lib.fa_fwd_decode(16, 16, 16, 16, None, kw.get("B", 1), kw.get("Sq", 1), 64, kw.get("Hq", 8),
                                       kw.get("Hkv", 2), 128, ctypes.c_float(kw.get("scale", 0.1)),
                                       kw.get("causal", 0), kw.get("dtype", 1), 0, None, 0, None)
    assert c(dtype=5) == api.FA_ERR_INVALID_ARG
    assert c(causal=3) == api.FA_ERR_INVALID_ARG
    assert c(scale=float("nan")) == api.FA_ERR_INVALID_ARG
    assert c(scale=3.0e38) == api.FA_ERR_UNSUPPORTED
    assert c(scale=0.0, B=0) == api.FA_OK          # zero and negative scales are valid
    assert c(scale=-1.0, B=0) == api.FA_OK
    assert c(Hq=258, Hkv=2) == api.FA_ERR_UNSUPPORTED
    assert c(B=0) == api.FA_OK


def test_host_workspace_size_formula(lib):
    # device copy of q, k, v, o (16-bit) and lse (fp32), each rounded up to 256 bytes
    B, Sq, Sk, Hq, Hkv, D = 2, 300, 257, 8, 2, 128
    up = lambda x: (x + 255) // 256 * 256
    q = B * Sq * Hq * D * 2
    kv = B * Sk * Hkv * D * 2
    want = up(q) + 2 * up(kv) + up(q) + up(B * Hq * Sq * 4)
    assert api.fa_fwd_host_workspace_size(B, Sq, Sk, Hq, Hkv, D) == want
    with pytest.raises(api.FAError):
        api.fa_fwd_host_workspace_size(-1, Sq, Sk, Hq, Hkv, D)


@pytest.mark.parametrize("kw,code", [
    (dict(dtype=7), api.FA_ERR_INVALID_ARG),
    (dict(Hq=3, Hkv=2), api.FA_ERR_INVALID_ARG),
    (dict(D=72), api.FA_ERR_UNSUPPORTED),
    (dict(q=None), api.FA_ERR_INVALID_ARG),
    (dict(workspace=None), api.FA_ERR_INVALID_ARG),
    (dict(workspace_bytes=16), api.FA_ERR_INVALID_ARG),
    (dict(workspace=256 + 16), api.FA_ERR_INVALID_ARG),      # not 256-byte aligned
    (dict(B=0), api.FA_OK),
])
def test_host_entry_validates_before_any_copy(lib, kw, code):
    args = dict(q=64, k=64, v=64, o=64, lse=None, B=1, Sq=4, Sk=4, Hq=2, Hkv=1, D=128, scale=0.125, causal=0,
                dtype=1, workspace=256, workspace_bytes=1 << 30, stream=None)
    args.update(kw)
    rc = lib.fa_fwd_host(args["q"], args["k"], args["v"], args["o"], args["lse"], args["B"], args["Sq"], args["Sk"],
                         args["Hq"], args["Hkv"], args["D"], args["scale"], args["causal"], args["dtype"],
                         args["workspace"], args["workspace_bytes"], args["stream"])
    assert rc == code
