"""The C ABI: the built library loads and exports every entry point that
include/fgm.h declares, and its host-side argument checks reject bad calls
before touching a GPU. No kernel runs here."""

import ctypes
import os
import re

import pytest

import fine_grained_moe_gb300 as fgm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fgm.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fgm_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(fgm.LIB_PATH):
        from fine_grained_moe_gb300 import build
        build.build()
    return fgm.lib()


def test_header_declares_the_four_step_calls():
    names = _declared()
    for n in ("fgm_moe_layer_fwd", "fgm_moe_stack_fwd", "fgm_lm_head_argmax", "fgm_spec_verify"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_workspace_bytes_host_only(lib):
    n = lib.fgm_workspace_bytes(5, 262144)
    assert n > 0 and n % 256 == 0
    assert lib.fgm_workspace_bytes(0, 0) == 0 and lib.fgm_workspace_bytes(9, 0) == 0
    assert lib.fgm_version() >= 100


def test_argument_checks_fail_before_launch(lib):
    L = fgm.fgm_layer()
    buf = (ctypes.c_uint8 * 4096)()
    # M out of range
    assert lib.fgm_moe_layer_fwd(ctypes.byref(L), buf, buf, 0, None, None, buf, 4096, None) == -1
    assert lib.fgm_moe_layer_fwd(ctypes.byref(L), buf, buf, 9, None, None, buf, 4096, None) == -1
    # null weights
    assert lib.fgm_moe_layer_fwd(ctypes.byref(L), buf, buf, 1, None, None, buf, 4096, None) == -1
    assert b"NULL" in lib.fgm_last_error()
    # stack: bad layer count
    arr = (fgm.fgm_layer * 1)()
    assert lib.fgm_moe_stack_fwd(arr, 0, buf, buf, 1, None, buf, 4096, None) == -1
    assert lib.fgm_moe_stack_fwd(arr, 49, buf, buf, 1, None, buf, 4096, None) == -1
    # lm_head: V out of range, misaligned embedding
    assert lib.fgm_lm_head_argmax(buf, 0, buf, 1, buf, None, buf, 4096, None) == -1
    assert lib.fgm_lm_head_argmax(ctypes.c_void_p(ctypes.addressof(buf) + 1), 10, buf, 1, buf, None,
                                  buf, 4096, None) == -1
    # FP8 lm_head: NULL or misaligned codes / scales, V out of range
    assert lib.fgm_lm_head_argmax_fp8(None, buf, 10, buf, 1, buf, None, buf, 4096, None) == -1
    assert lib.fgm_lm_head_argmax_fp8(buf, ctypes.c_void_p(ctypes.addressof(buf) + 2), 10, buf, 1, buf,
                                      None, buf, 4096, None) == -1
    assert lib.fgm_lm_head_argmax_fp8(buf, buf, 0, buf, 1, buf, None, buf, 4096, None) == -1
    assert b"V = 0" in lib.fgm_last_error()
    assert lib.fgm_verify_step_fp8_head(arr, 1, buf, buf, 10, buf, None, 2, None, buf, buf, 4096,
                                        None) == -1
    # spec_verify: draft missing with M > 1
    assert lib.fgm_spec_verify(buf, None, 3, buf, None) == -1
    # workspace too small / misaligned
    big = (ctypes.c_uint8 * (1 << 22))()
    base = (ctypes.addressof(big) + 255) // 256 * 256
    assert lib.fgm_read_status(ctypes.c_void_p(base), 16, 0, buf, None) == -2
    assert lib.fgm_read_status(ctypes.c_void_p(base + 8), 1 << 21, 0, buf, None) == -2


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(fgm, "_lib", None)
    monkeypatch.setattr(fgm, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(fgm.FgmError):
        fgm.lib()


def test_dense_stack_argument_checks(lib):
    """The dense stack and verify step reject a missing MLP table and a width
    that is not a multiple of 704 before any launch."""
    arr = (fgm.fgm_layer * 1)()
    buf = (ctypes.c_uint8 * 4096)()
    assert lib.fgm_moe_stack_dense_fwd(arr, None, 1, buf, buf, 1, None, buf, 4096, None) == -1
    mlps = (fgm.fgm_mlp * 1)()
    mlps[0].width = 700
    # (the layer struct is checked first: fill it with aligned dummies)
    for name in ("router_w", "gate_q", "gate_s", "up_q", "up_s", "down_q", "down_s"):
        setattr(arr[0], name, ctypes.addressof(buf))
    assert lib.fgm_moe_stack_dense_fwd(arr, mlps, 1, buf, buf, 1, None, buf, 4096, None) == -1
    assert b"width 700" in lib.fgm_last_error()
    assert lib.fgm_verify_step_dense(arr, None, 1, buf, 16, buf, None, 1, None, buf, buf, 4096, None) == -1
