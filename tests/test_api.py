"""Host-side checks of the C ABI and the Python binding (no GPU needed).

Argument validation in attn_fwd runs before any CUDA call, so invalid calls can
be exercised on a machine without a GPU: the fake pointer values below are
never dereferenced.
"""
import ctypes
import os
import re

import pytest
import torch

import scaled_dot_product_tcgen05_gb300 as pkg
from scaled_dot_product_tcgen05_gb300 import build_lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")


@pytest.fixture(scope="module")
def lib():
    build_lib.build()
    return pkg.load_library()


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\*?(attn_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    fns = header_functions()
    assert "attn_fwd" in fns and "attn_check" in fns and "attn_status_string" in fns
    assert set(fns) == set(pkg.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), name
    # also check the dynamic symbol table directly
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", build_lib.LIB_PATH], capture_output=True,
                         text=True).stdout
    for name in header_functions():
        assert re.search(rf"\bT {name}$", out, flags=re.M), name


def test_status_strings(lib):
    for code, name in [(0, "ATTN_OK"), (-1, "ATTN_ERR_INVALID_ARG"), (-2, "ATTN_ERR_UNSUPPORTED"),
                       (-3, "ATTN_ERR_MISALIGNED"), (-4, "ATTN_ERR_CUDA"),
                       (-5, "ATTN_ERR_DEVICE_TIMEOUT"), (-6, "ATTN_ERR_BAD_SEQLENS")]:
        assert lib.attn_status_string(code).decode() == name
    assert lib.attn_status_string(123).decode() == "ATTN_ERR_UNKNOWN"


A = 0x10000  # fake, 16-byte aligned addresses: validation fails before any use


def call(lib, **kw):
    args = dict(q=A, k=A + 0x100, v=A + 0x200, o=A + 0x300, lse=A + 0x400, B=1, H=2, Sq=128,
                Sk=128, D=64, scale=0.125, causal=0, cq=0, ck=0, dtype=0)
    args.update(kw)
    return pkg.attn_fwd_raw(args["q"], args["k"], args["v"], args["o"], args["lse"], args["B"],
                            args["H"], args["Sq"], args["Sk"], args["D"], args["scale"],
                            args["causal"], args["cq"], args["ck"], args["dtype"], 0)


@pytest.mark.parametrize("kw,code", [
    (dict(D=96), pkg.ATTN_ERR_UNSUPPORTED),
    (dict(D=256), pkg.ATTN_ERR_UNSUPPORTED),
    (dict(dtype=2), pkg.ATTN_ERR_UNSUPPORTED),
    (dict(B=-1), pkg.ATTN_ERR_INVALID_ARG),
    (dict(H=0), pkg.ATTN_ERR_INVALID_ARG),
    (dict(Sq=-5), pkg.ATTN_ERR_INVALID_ARG),
    (dict(Sk=0), pkg.ATTN_ERR_INVALID_ARG),
    (dict(scale=float("nan")), pkg.ATTN_ERR_INVALID_ARG),
    (dict(scale=float("inf")), pkg.ATTN_ERR_INVALID_ARG),
    (dict(cq=A + 0x500), pkg.ATTN_ERR_INVALID_ARG),
    (dict(ck=A + 0x500), pkg.ATTN_ERR_INVALID_ARG),
    (dict(q=0), pkg.ATTN_ERR_INVALID_ARG),
    (dict(lse=0), pkg.ATTN_ERR_INVALID_ARG),
    (dict(q=A + 8), pkg.ATTN_ERR_MISALIGNED),
    (dict(o=A + 2), pkg.ATTN_ERR_MISALIGNED),
    (dict(lse=A + 2), pkg.ATTN_ERR_MISALIGNED),
    (dict(cq=A + 0x502, ck=A + 0x600), pkg.ATTN_ERR_MISALIGNED),
    (dict(B=1 << 16, Sq=1 << 16), pkg.ATTN_ERR_INVALID_ARG),
])
def test_invalid_arguments_rejected_before_launch(lib, kw, code):
    assert call(lib, **kw) == code


def test_empty_problem_is_a_noop(lib):
    assert call(lib, B=0) == pkg.ATTN_OK
    assert call(lib, Sq=0) == pkg.ATTN_OK
    assert call(lib, B=0, q=0, k=0, v=0, o=0, lse=0) == pkg.ATTN_OK


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU behaviour")
def test_no_device_fails_loudly(lib):
    st = call(lib)
    assert st in (pkg.ATTN_ERR_CUDA, pkg.ATTN_ERR_UNSUPPORTED)
    assert lib.attn_num_sms() < 0
    with pytest.raises(ValueError):
        pkg.attn_fwd(torch.zeros(1, 128, 2, 64, dtype=torch.float16),
                     torch.zeros(1, 128, 2, 64, dtype=torch.float16),
                     torch.zeros(1, 128, 2, 64, dtype=torch.float16))


def test_missing_library_raises(tmp_path):
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        pkg.load_library(str(tmp_path / "missing.so"))


def test_product_path_does_not_import_the_oracle():
    pkg_dir = os.path.join(ROOT, "scaled_dot_product_tcgen05_gb300")
    pat = re.compile(r"^\s*(import\s+oracle|from\s+oracle)|sdpa_oracle|#include.*oracle", re.M)
    for dirpath, _, files in os.walk(pkg_dir):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp", ".c")):
                text = open(os.path.join(dirpath, f), encoding="utf-8").read()
                assert not pat.search(text), f


def call_window(lib, wl, wr, g, **kw):
    args = dict(q=A, k=A + 0x100, v=A + 0x200, o=A + 0x300, lse=A + 0x400, B=1, H=2, Sq=128,
                Sk=128, D=64, scale=0.125, causal=0, cq=0, ck=0, dtype=0)
    args.update(kw)
    return pkg.attn_fwd_window_raw(args["q"], args["k"], args["v"], args["o"], args["lse"],
                                   args["B"], args["H"], args["Sq"], args["Sk"], args["D"],
                                   args["scale"], args["causal"], wl, wr, g, args["cq"],
                                   args["ck"], args["dtype"], 0)


@pytest.mark.parametrize("wl,wr,g,causal", [
    (-2, 0, 0, 0), (0, -2, 0, 0), (5, 5, -1, 0), (5, 1, 0, 1), (-1, 3, 0, 1),
])
def test_window_arguments_rejected_before_launch(lib, wl, wr, g, causal):
    assert call_window(lib, wl, wr, g, causal=causal) == pkg.ATTN_ERR_INVALID_ARG


def test_window_entry_point_shares_attn_fwd_checks(lib):
    assert call_window(lib, 4, 0, 0, causal=1, D=96) == pkg.ATTN_ERR_UNSUPPORTED
    assert call_window(lib, 4, 0, 0, causal=1, q=A + 8) == pkg.ATTN_ERR_MISALIGNED
    assert call_window(lib, 4, 0, 0, causal=1, B=0) == pkg.ATTN_OK
    assert call_window(lib, -1, -1, 0, Sq=0) == pkg.ATTN_OK


def test_bwd_rejects_zero_scale_and_bad_sizes(lib):
    a = dict(q=A, k=A + 0x100, v=A + 0x200, o=A + 0x300, do=A + 0x400, lse=A + 0x500,
             dq=A + 0x600, dk=A + 0x700, dv=A + 0x800, ws=A + 0x1000, cq=None, ck=None)
    def bwd(scale=0.125, D=64, B=1, Sq=128, Sk=128, dtype=0, ws_bytes=1 << 30, **kw):
        x = dict(a, **kw)
        return lib.attn_bwd(x["q"], x["k"], x["v"], x["o"], x["do"], x["lse"], x["dq"], x["dk"],
                            x["dv"], B, 2, Sq, Sk, D, ctypes.c_float(scale), 1, x["cq"], x["ck"],
                            x["ws"], ws_bytes, dtype, None)
    assert bwd(scale=0.0) == pkg.ATTN_ERR_UNSUPPORTED
    assert bwd(scale=float("nan")) == pkg.ATTN_ERR_INVALID_ARG
    assert bwd(D=96) == pkg.ATTN_ERR_UNSUPPORTED
    assert bwd(Sk=0) == pkg.ATTN_ERR_INVALID_ARG
    assert bwd(ws=A + 0x1010) == pkg.ATTN_ERR_MISALIGNED
    assert bwd(ws_bytes=16) == pkg.ATTN_ERR_INVALID_ARG
    assert bwd(B=0) == pkg.ATTN_OK
    # packed sequences: both bounds arrays or neither, 4-byte aligned
    assert bwd(cq=A + 0x900) == pkg.ATTN_ERR_INVALID_ARG
    assert bwd(ck=A + 0x900) == pkg.ATTN_ERR_INVALID_ARG
    assert bwd(cq=A + 0x902, ck=A + 0x980) == pkg.ATTN_ERR_MISALIGNED
    assert bwd(cq=A + 0x900, ck=A + 0x980, ws_bytes=16) == pkg.ATTN_ERR_INVALID_ARG
    n = ctypes.c_size_t(0)
    assert lib.attn_bwd_workspace(1, 2, 300, 128, 0, ctypes.byref(n)) == pkg.ATTN_OK
    # dense: fp32 accumulator + 8 KiB per 128-query tile and head
    assert n.value == ((2 * 300 * 128 * 4 + 255) // 256) * 256 + 2 * 3 * 8192
    # packed, 5 sequences over 300 rows: at most (300 + 127 * 5) // 128 = 7 tiles per head,
    # plus 4 * (5 + 2) bytes of tile offsets rounded up to 256
    assert lib.attn_bwd_workspace(5, 2, 300, 128, 1, ctypes.byref(n)) == pkg.ATTN_OK
    assert n.value == ((2 * 300 * 128 * 4 + 255) // 256) * 256 + 2 * 7 * 8192 + 256
    assert lib.attn_bwd_workspace(1, 2, 300, 96, 0, ctypes.byref(n)) == pkg.ATTN_ERR_UNSUPPORTED

def test_fp8_workspace_is_the_transposed_v_with_keys_padded_to_16(lib):
    n = ctypes.c_size_t(0)
    for B, H, Sk, keys in ((1, 2, 16, 16), (2, 3, 17, 32), (1, 32, 65536, 65536), (3, 1, 1, 16)):
        assert lib.attn_fwd_fp8_workspace(B, H, Sk, 128, ctypes.byref(n)) == pkg.ATTN_OK
        assert n.value == H * 128 * B * keys  # V^T [H, 128, B * round16(Sk)], one byte each
    assert lib.attn_fwd_fp8_workspace(1, 2, 16, 64, ctypes.byref(n)) == pkg.ATTN_ERR_UNSUPPORTED
    assert n.value == 0
    assert lib.attn_fwd_fp8_workspace(1, 0, 16, 128, ctypes.byref(n)) == pkg.ATTN_ERR_INVALID_ARG
    assert lib.attn_fwd_fp8_workspace(1, 2, 0, 128, ctypes.byref(n)) == pkg.ATTN_ERR_INVALID_ARG
    assert lib.attn_fwd_fp8_workspace(1, 2, 16, 128, None) == pkg.ATTN_ERR_INVALID_ARG
