"""The C ABI without a GPU: the library builds, loads, exports every entry point the
header declares, and rejects bad arguments on the host before any launch."""
import ctypes
import os
import re
import shutil

import pytest
import torch

import bf16_forward_attention_gb300 as attn
from bf16_forward_attention_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn_fwd.h")


@pytest.fixture(scope="module")
def lib():
    if not build.up_to_date():
        if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
            pytest.skip("library not built and nvcc not available")
        build.build()
    return attn.load_library()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(attn_\w+)\s*\(", text, flags=re.M)


def test_header_declares_entry_points():
    names = _declared_functions()
    assert {"attn_fwd", "attn_status_str", "attn_fwd_last_error", "attn_fwd_version"} <= set(names)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for st in range(0, -13, -1):
        s = attn.status_str(st)
        assert s and s != "unknown status", st
    assert attn.status_str(-1234) == "unknown status"
    assert lib.attn_fwd_version() >= 100


A = 1 << 20  # fake, 16-byte aligned addresses: never dereferenced on these paths


def _call(q=A, k=2 * A, v=3 * A, o=4 * A, layout=0, B=1, H=2, Sq=256, Sk=256, d=128,
          scale=0.088, mode=0):
    return attn.attn_fwd_raw(q, k, v, o, layout, B, H, Sq, Sk, d, scale, mode, 0)


@pytest.mark.parametrize("kw,status", [
    (dict(q=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(o=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(B=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(H=-1), attn.ATTN_ERR_INVALID_ARG),
    (dict(Sq=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(Sk=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(scale=float("nan")), attn.ATTN_ERR_INVALID_ARG),
    (dict(scale=float("inf")), attn.ATTN_ERR_INVALID_ARG),
    (dict(d=64), attn.ATTN_ERR_UNSUPPORTED),
    (dict(d=256), attn.ATTN_ERR_UNSUPPORTED),
    (dict(layout=2), attn.ATTN_ERR_UNSUPPORTED),
    (dict(mode=3), attn.ATTN_ERR_UNSUPPORTED),
    (dict(mode=-1), attn.ATTN_ERR_UNSUPPORTED),
    (dict(q=A + 8), attn.ATTN_ERR_MISALIGNED),
    (dict(o=4 * A + 2), attn.ATTN_ERR_MISALIGNED),
    (dict(o=A), attn.ATTN_ERR_ALIASING),
    (dict(o=3 * A + 4096), attn.ATTN_ERR_ALIASING),
    (dict(Sq=1 << 31), attn.ATTN_ERR_TOO_LARGE),
    (dict(H=1 << 20, Sq=1 << 20, Sk=1 << 20), attn.ATTN_ERR_TOO_LARGE),
])
def test_host_validation(lib, kw, status):
    assert _call(**kw) == status


def test_timeout_selftest_validation(lib):
    args = (A, 2 * A, 3 * A, 4 * A, 0, 1, 2, 256, 256, 128, 0.088, 0)
    assert attn.attn_fwd_timeout_selftest_raw(*args, 0, 0) == attn.ATTN_ERR_INVALID_ARG
    assert attn.attn_fwd_timeout_selftest_raw(*args, 0, 3_000_000_000) == attn.ATTN_ERR_INVALID_ARG
    bad = (0,) + args[1:]
    assert attn.attn_fwd_timeout_selftest_raw(*bad, 0, 10_000_000) == attn.ATTN_ERR_INVALID_ARG
    # Flags: the tail split only (the causal mask is not a mode of this test entry).
    assert (attn.attn_fwd_timeout_selftest_raw(*args, 0, 10_000_000, attn.ATTN_FLAG_CAUSAL)
            == attn.ATTN_ERR_UNSUPPORTED)
    assert (attn.attn_fwd_timeout_selftest_raw(*args, 0, 10_000_000, attn.ATTN_FLAG_SPLIT_TAIL)
            == attn.ATTN_ERR_NO_DEVICE)


def _split(q=A, k=2 * A, v=3 * A, o=4 * A, B=1, H=2, Sq=256, Sk=1000, splits=2, ws=8 * A,
           ws_bytes=1 << 24):
    return attn.attn_fwd_splitkv_raw(q, k, v, o, 0, B, H, Sq, Sk, 128, 0.088, 0, splits, ws, ws_bytes, 0)


def test_split_tail_items_validation(lib):
    assert attn.split_tail_items(0, 1, 256, 256) == attn.ATTN_ERR_INVALID_ARG
    assert attn.split_tail_items(1 << 31, 1, 256, 256) == attn.ATTN_ERR_TOO_LARGE
    assert attn.split_tail_items(1 << 20, 1 << 20, 256, 256) == attn.ATTN_ERR_TOO_LARGE
    assert attn.split_tail_items(1, 8, 4096, 32768) == attn.ATTN_ERR_NO_DEVICE  # valid; no GPU


def test_splitkv_workspace_bytes(lib):
    assert attn.splitkv_workspace_bytes(1, 2, 256, 1000, 1) == 0
    # splits x B x H x rows (padded to 256) x (128 + 2) fp32
    assert attn.splitkv_workspace_bytes(1, 2, 256, 1000, 2) == 2 * 2 * 256 * 130 * 4
    assert attn.splitkv_workspace_bytes(3, 1, 300, 1000, 8) == 8 * 3 * 512 * 130 * 4
    for bad in [(1, 2, 256, 1000, 0), (1, 2, 256, 1000, 9), (0, 2, 256, 1000, 2)]:
        with pytest.raises(attn.AttnError):
            attn.splitkv_workspace_bytes(*bad)
    assert attn.splitkv_num_splits(2, 16, 8192, 8192) == 1
    assert 1 <= attn.splitkv_num_splits(1, 1, 100, 4096) <= 8


@pytest.mark.parametrize("B,H,Sq,Sk,splits", [
    (1 << 31, 1 << 21, 1, 384, 3),       # each size below the per-size check, product huge
    ((1 << 31) - 1, 2, 1, 384, 3),       # more than 2^31 - 1 CTAs
    (1, (1 << 30), 512, 384, 3),
    (1 << 40, 1, 1, 384, 2),             # one size beyond 2^31 - 1
])
def test_splitkv_workspace_bytes_never_overflows(lib, B, H, Sq, Sk, splits):
    n = lib.attn_fwd_splitkv_workspace_bytes(B, H, Sq, Sk, 128, splits)
    assert n == attn.ATTN_ERR_TOO_LARGE
    # The no-allocation entry point passes the status on (it sizes its scratch
    # with the same function) and launches nothing; the pointers are never used.
    st = attn.attn_fwd_splitkv_noalloc_raw(A, 2 * A, 3 * A, 4 * A, 0, B, H, Sq, Sk, 128, 0.088, 0,
                                           splits, 0)
    assert st == attn.ATTN_ERR_TOO_LARGE


@pytest.mark.parametrize("kw,status", [
    (dict(splits=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(splits=9), attn.ATTN_ERR_INVALID_ARG),          # 1000 keys = 8 tiles
    (dict(ws=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(ws_bytes=1000), attn.ATTN_ERR_INVALID_ARG),
    (dict(ws=8 * A + 4), attn.ATTN_ERR_MISALIGNED),
    (dict(ws=4 * A + 256), attn.ATTN_ERR_ALIASING),       # overlaps out
    (dict(ws=2 * A), attn.ATTN_ERR_ALIASING),             # overlaps k
])
def test_splitkv_validation(lib, kw, status):
    assert _split(**kw) == status


@pytest.mark.skipif(torch.cuda.is_available(), reason="fake pointers must never reach a GPU")
def test_splitkv_valid_call_without_gpu_reports_no_device(lib):
    assert _split() == attn.ATTN_ERR_NO_DEVICE


@pytest.mark.parametrize("Hq,Hkv,flags,status", [
    (8, 3, 0, attn.ATTN_ERR_INVALID_ARG),     # Hq not a multiple of Hkv
    (8, 0, 0, attn.ATTN_ERR_INVALID_ARG),
    (8, 2, 4, attn.ATTN_ERR_UNSUPPORTED),     # unknown flag
    (8, 2, attn.ATTN_FLAG_SPLIT_TAIL, attn.ATTN_ERR_NO_DEVICE),  # accepted; no GPU here
    (8, 2, attn.ATTN_FLAG_SPLIT_TAIL | attn.ATTN_FLAG_CAUSAL, attn.ATTN_ERR_NO_DEVICE),
])
def test_ex_validation(lib, Hq, Hkv, flags, status):
    assert attn.attn_fwd_ex_raw(A, 2 * A, 3 * A, 4 * A, 0, 1, Hq, Hkv, 256, 256, 128, 0.088, 0,
                                flags, 0) == status


def _varlen(q=A, k=2 * A, v=3 * A, o=4 * A, cq=5 * A, ck=6 * A, B=2, Hq=4, Hkv=2, tq=300, tk=500,
            maxq=200, d=128, scale=0.088, mode=0, flags=0):
    return attn.attn_fwd_varlen_raw(q, k, v, o, cq, ck, B, Hq, Hkv, tq, tk, maxq, d, scale, mode,
                                    flags, 0)


@pytest.mark.parametrize("kw,status", [
    (dict(cq=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(ck=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(B=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(Hkv=3), attn.ATTN_ERR_INVALID_ARG),
    (dict(tq=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(tk=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(maxq=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(maxq=301), attn.ATTN_ERR_INVALID_ARG),
    (dict(scale=float("nan")), attn.ATTN_ERR_INVALID_ARG),
    (dict(flags=4), attn.ATTN_ERR_UNSUPPORTED),
    (dict(d=64), attn.ATTN_ERR_UNSUPPORTED),
    (dict(mode=3), attn.ATTN_ERR_UNSUPPORTED),
    (dict(q=A + 8), attn.ATTN_ERR_MISALIGNED),
    (dict(cq=5 * A + 2), attn.ATTN_ERR_MISALIGNED),
    (dict(o=A), attn.ATTN_ERR_ALIASING),
    (dict(o=5 * A - 256), attn.ATTN_ERR_ALIASING),   # out runs over cu_seqlens_q
])
def test_varlen_validation(lib, kw, status):
    assert _varlen(**kw) == status


@pytest.mark.skipif(torch.cuda.is_available(), reason="fake pointers must never reach a GPU")
def test_varlen_valid_call_without_gpu_reports_no_device(lib):
    assert _varlen(flags=attn.ATTN_FLAG_CAUSAL) == attn.ATTN_ERR_NO_DEVICE


def _host(q=A, k=2 * A, v=3 * A, o=4 * A, layout=1, B=2, Hq=16, Hkv=16, Sq=8192, Sk=8192, d=128,
          scale=0.088, mode=0, flags=0, ws=8 * A, wsb=None):
    need = attn.host_workspace_bytes(B, Hq, Hkv, Sq, Sk, d) if wsb is None else wsb
    return attn.attn_fwd_host_raw(q, k, v, o, layout, B, Hq, Hkv, Sq, Sk, d, scale, mode, flags, ws,
                                  max(need, 0), 0)


def test_varlen_host_workspace_bytes(lib):
    n = lib.attn_fwd_varlen_host_workspace_bytes(3, 8, 2, 1000, 1500, 128)
    assert n == 2 * 1000 * 8 * 256 + 2 * 1500 * 2 * 256 + 2 * 256
    assert lib.attn_fwd_varlen_host_workspace_bytes(3, 8, 3, 1000, 1500, 128) == attn.ATTN_ERR_INVALID_ARG
    assert lib.attn_fwd_varlen_host_workspace_bytes(3, 8, 2, 0, 1500, 128) == attn.ATTN_ERR_INVALID_ARG


def test_host_buffer_workspace_bytes(lib):
    assert attn.host_workspace_bytes(2, 16, 4, 8192, 1000) == 2 * 2 * 16 * 8192 * 256 + 2 * 2 * 4 * 1000 * 256
    assert attn.host_workspace_bytes(1, 1, 1, 1, 1) == 4 * 256
    assert attn.host_workspace_bytes(1, 6, 4, 10, 10) == attn.ATTN_ERR_INVALID_ARG
    assert attn.host_workspace_bytes(1, 2, 2, 10, 10, 64) == attn.ATTN_ERR_UNSUPPORTED


@pytest.mark.parametrize("kw,status", [
    (dict(q=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(ws=0), attn.ATTN_ERR_INVALID_ARG),
    (dict(wsb=1000), attn.ATTN_ERR_INVALID_ARG),       # workspace too small
    (dict(Hkv=3), attn.ATTN_ERR_INVALID_ARG),
    (dict(scale=float("inf")), attn.ATTN_ERR_INVALID_ARG),
    (dict(flags=2), attn.ATTN_ERR_UNSUPPORTED),
    (dict(d=64), attn.ATTN_ERR_UNSUPPORTED),
    (dict(layout=5), attn.ATTN_ERR_UNSUPPORTED),
    (dict(mode=7), attn.ATTN_ERR_UNSUPPORTED),
    (dict(ws=8 * A + 16), attn.ATTN_ERR_MISALIGNED),    # workspace must be 256-byte aligned
])
def test_host_buffer_validation(lib, kw, status):
    assert _host(**kw) == status


@pytest.mark.skipif(torch.cuda.is_available(), reason="fake pointers must never reach a GPU")
def test_host_buffer_call_without_gpu_reports_no_device(lib):
    assert _host(flags=attn.ATTN_FLAG_CAUSAL) == attn.ATTN_ERR_NO_DEVICE


@pytest.mark.skipif(torch.cuda.is_available(), reason="fake pointers must never reach a GPU")
def test_ex_valid_call_without_gpu_reports_no_device(lib):
    assert attn.attn_fwd_ex_raw(A, 2 * A, 3 * A, 4 * A, 1, 1, 8, 2, 256, 300, 128, 0.088, 0,
                                attn.ATTN_FLAG_CAUSAL, 0) == attn.ATTN_ERR_NO_DEVICE


@pytest.mark.skipif(torch.cuda.is_available(), reason="fake pointers must never reach a GPU")
def test_valid_call_without_gpu_reports_no_device(lib):
    assert _call() == attn.ATTN_ERR_NO_DEVICE


def test_release_build_has_no_debug_checks(lib):
    assert lib.attn_fwd_debug_build() == 0
    # The release build refuses the debug self-test before touching any pointer.
    assert lib.attn_fwd_debug_selftest(A, 2 * A, 3 * A, 4 * A, 0, 1, 2, 256, 256, 128, 0.088, 0,
                                       0) == attn.ATTN_ERR_UNSUPPORTED


def test_debug_flavour_builds_and_loads():
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available")
    build.build(debug=True)
    dbg = attn.load_library(debug=True)
    assert dbg.attn_fwd_debug_build() == 1
    for name in _declared_functions():
        assert hasattr(dbg, name), name


def test_python_binding_checks(lib):
    x = torch.zeros(1, 1, 4, 128, dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        attn.attn_fwd(x, x, x)  # CPU tensors are refused before any call
    with pytest.raises(ValueError):
        attn.attn_fwd(x, x, x, layout="sbhd")
    with pytest.raises(ValueError):
        attn.attn_fwd(x, x, x, rounding="rtp")
    # attn_fwd_host takes host tensors; a wrongly shaped or typed out is refused
    # before the library writes through its pointer.
    with pytest.raises(ValueError):
        attn.attn_fwd_host(x, x, x, out=torch.zeros(1, 1, 3, 128, dtype=torch.bfloat16))
    with pytest.raises(ValueError):
        attn.attn_fwd_host(x, x, x, out=torch.zeros(1, 1, 4, 128, dtype=torch.float32))
    with pytest.raises(ValueError):
        attn.attn_fwd_host(x, x[:, :, :2].repeat(1, 2, 1, 1)[:, :1], x)  # k, v shapes differ
    with pytest.raises(TypeError):
        attn.attn_fwd_host(x.float(), x, x)


def test_product_package_does_not_import_oracle():
    pkg = os.path.join(ROOT, "bf16_forward_attention_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(from|import)\s+oracle\b", src, flags=re.M), f
                assert "oracle/" not in src, f
