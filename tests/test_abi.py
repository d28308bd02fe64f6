"""The C-ABI library without a GPU: it builds for sm_103a, loads, exports every
symbol include/spec_verify.h declares, and rejects bad arguments on the host
before touching the device.  The binding refuses to run without the library."""
import ctypes
import os
import re
import shutil

import pytest

import speculative_decoding_verification_68_gb300 as sv
from speculative_decoding_verification_68_gb300 import _native

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "spec_verify.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(spec_verify\w*)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    if shutil.which(_native.nvcc()) is None and not os.path.exists(_native.nvcc()):
        pytest.skip("nvcc not available")
    _native.build()
    return _native.load()


def test_header_declares_the_interface():
    names = declared_functions()
    for need in ("spec_verify_init", "spec_verify", "spec_verify_tv", "spec_verify_get_error",
                 "spec_verify_destroy", "spec_verify_strerror"):
        assert need in names


def test_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_host_side_argument_checks(lib):
    h = ctypes.c_void_p()
    assert lib.spec_verify_init(None, 1, 7, 100, 0, 0) == sv.SV_ERR_ARG
    assert lib.spec_verify_init(ctypes.byref(h), 1, 0, 100, 0, 0) == 3      # k = 0
    assert lib.spec_verify_init(ctypes.byref(h), 1, 32, 100, 0, 0) == 3     # k above 31
    assert lib.spec_verify_init(ctypes.byref(h), 1, 7, 100, 9, 0) == 2      # dtype
    assert lib.spec_verify_init(ctypes.byref(h), 1, 7, 400000, 1, 0) == 3   # vocabulary too large
    assert lib.spec_verify_init(ctypes.byref(h), 1, 7, 327681, 1, 0) == 3   # bf16: V <= 327,680
    assert lib.spec_verify_init(ctypes.byref(h), 1, 7, 163841, 0, 0) == 3   # fp32: V <= 163,840
    assert lib.spec_verify_init(ctypes.byref(h), -1, 7, 100, 0, 0) == sv.SV_ERR_ARG
    assert lib.spec_verify_init(ctypes.byref(h), 1 << 28, 7, 100, 0, 0) == 3   # B*(k+1) reaches 2^31
    assert lib.spec_verify_ex(None, 1, *([None] * 13)) == sv.SV_ERR_ARG
    assert lib.spec_verify_loss_grad(None, 1, None, None, None, 0, None, None, None, None) == sv.SV_ERR_ARG
    assert lib.spec_verify_lazy(None, 1, *([None] * 8)) == sv.SV_ERR_ARG
    assert lib.spec_verify(None, 1, *([None] * 11)) == sv.SV_ERR_ARG
    assert lib.spec_verify_tv(None, 1, *([None] * 5)) == sv.SV_ERR_ARG
    assert lib.spec_verify_get_error(None, None) == sv.SV_ERR_ARG
    assert lib.spec_verify_selftest_wait(None, 1, None) == sv.SV_ERR_ARG
    lib.spec_verify_destroy(None)
    assert lib.spec_verify_strerror(0) == b"ok"
    assert b"invalid" in lib.spec_verify_strerror(6)


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(_native, "LIB", str(tmp_path / "missing.so"))
    monkeypatch.setattr(_native, "_lib", None)
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        _native.load()
