"""The C ABI without a GPU: the library builds for sm_103a, loads, exports every function
include/softmax_rows.h declares, and rejects bad arguments on the host before touching CUDA."""
import ctypes
import os
import re

import pytest

import row_wise_online_gb300 as rwo
from row_wise_online_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "softmax_rows.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return rwo.capi()


def declared_functions():
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*([a-z_0-9]+)\s*\(", text, flags=re.M)))


def test_header_declares_the_named_calls():
    names = declared_functions()
    for n in ("softmax_rows", "softmax_rows_ex", "softmax_row_state", "merge_states"):
        assert n in names
    assert set(rwo.EXPORTED) >= set(names), set(names) - set(rwo.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_build_targets_sm_103a_only():
    flags = " ".join(_build.NVCC_FLAGS)
    assert "arch=compute_103a,code=sm_103a" in flags and flags.count("-gencode") == 1


NULL = None
X = ctypes.c_void_p(0x1000)  # never dereferenced: every call below fails validation first


@pytest.mark.parametrize("args,expect", [
    ((NULL, X, 4, 4, 0, NULL), rwo.ERR_INVALID_ARG),       # x NULL
    ((X, NULL, 4, 4, 0, NULL), rwo.ERR_INVALID_ARG),       # y NULL
    ((X, X, 4, 0, 0, NULL), rwo.ERR_INVALID_ARG),          # N = 0
    ((X, X, -1, 4, 0, NULL), rwo.ERR_INVALID_ARG),         # M < 0
    ((X, X, 4, 4, 7, NULL), rwo.ERR_INVALID_ARG),          # unknown dtype
    ((X, X, 2**62, 2**3, 0, NULL), rwo.ERR_INVALID_ARG),   # M*N*4 overflows int64
    ((X, X, 0, 4, 0, NULL), rwo.OK),                        # M = 0: no-op
    ((NULL, NULL, 0, 4, 0, NULL), rwo.OK),                  # M = 0 with the NULL data of an empty tensor
    ((NULL, NULL, 0, 0, 0, NULL), rwo.ERR_INVALID_ARG),     # ... but N is still checked
])
def test_softmax_rows_argument_checks(lib, args, expect):
    assert lib.softmax_rows(*args) == expect


def test_other_calls_argument_checks(lib):
    assert lib.softmax_rows_ex(X, X, None, None, None, 4, 4, 0, 99, None) == rwo.ERR_INVALID_ARG
    assert lib.softmax_rows_ex(X, X, None, None, None, 4, 4, 0, -1, None) == rwo.ERR_INVALID_ARG
    assert lib.softmax_row_state(X, None, None, None, 4, 4, 0, None) == rwo.ERR_INVALID_ARG  # no output
    assert lib.softmax_row_state(X, X, None, None, 0, 4, 0, None) == rwo.OK
    assert lib.merge_states(X, X, X, None, X, X, None, 4, None) == rwo.ERR_INVALID_ARG
    assert lib.merge_states(X, X, X, X, X, None, None, 4, None) == rwo.ERR_INVALID_ARG
    assert lib.merge_states(X, X, X, X, X, X, None, 0, None) == rwo.OK
    assert lib.softmax_rows_host(X, NULL, 4, 4, 0, None) == rwo.ERR_INVALID_ARG
    assert lib.softmax_rows_causal(X, X, None, None, None, 4, 4, 0, 0, 0, None) == rwo.ERR_INVALID_ARG  # period 0
    assert lib.softmax_rows_causal(X, NULL, None, None, None, 4, 4, 4, 0, 0, None) == rwo.ERR_INVALID_ARG
    assert lib.softmax_rows_causal(NULL, NULL, None, None, None, 0, 4, 4, 0, 0, None) == rwo.OK  # M = 0
    assert lib.log_softmax_rows(X, NULL, None, None, None, 4, 4, 0, 0, None) == rwo.ERR_INVALID_ARG  # no y
    assert lib.log_softmax_rows(X, X, None, None, None, 4, 4, 0, 6, None) == rwo.ERR_INVALID_ARG  # variant
    assert lib.log_softmax_rows(NULL, NULL, None, None, None, 0, 4, 1, 0, None) == rwo.OK  # M = 0
    assert lib.cross_entropy_rows(X, NULL, X, None, 4, 4, 0, None) == rwo.ERR_INVALID_ARG  # no labels
    assert lib.cross_entropy_rows(X, X, None, None, 4, 4, 0, None) == rwo.ERR_INVALID_ARG  # no loss
    assert lib.cross_entropy_rows(X, X, X, None, 4, 0, 0, None) == rwo.ERR_INVALID_ARG  # N = 0
    assert lib.cross_entropy_rows(NULL, NULL, NULL, None, 0, 4, 0, None) == rwo.OK  # M = 0
    st = lib.softmax_rows_strided
    assert st(X, 3, X, 4, None, None, None, 4, 4, 0, 1.0, 0, 0, None) == rwo.ERR_INVALID_ARG  # ldx < N
    assert st(X, 4, X, 3, None, None, None, 4, 4, 0, 1.0, 0, 0, None) == rwo.ERR_INVALID_ARG  # ldy < N
    assert st(X, 4, X, 4, None, None, None, 4, 4, 0, 0.0, 0, 0, None) == rwo.ERR_INVALID_ARG  # scale 0
    assert st(X, 4, X, 4, None, None, None, 4, 4, 0, -2.0, 0, 0, None) == rwo.ERR_INVALID_ARG
    assert st(X, 4, X, 4, None, None, None, 4, 4, 0, float("inf"), 0, 0, None) == rwo.ERR_INVALID_ARG
    assert st(X, 4, X, 4, None, None, None, 4, 4, 0, float("nan"), 0, 0, None) == rwo.ERR_INVALID_ARG
    assert st(X, 4, X, 4, None, None, None, 4, 4, 0, 1.0, 2, 0, None) == rwo.ERR_INVALID_ARG  # unknown flag
    assert st(X, 4, X, 4, None, None, None, 4, 4, 3, 1.0, 0, 0, None) == rwo.ERR_INVALID_ARG  # dtype
    assert st(X, 4, NULL, 4, None, None, None, 4, 4, 0, 1.0, 0, 0, None) == rwo.ERR_INVALID_ARG  # no y
    assert st(X, 2**62, X, 4, None, None, None, 4, 4, 0, 1.0, 0, 0, None) == rwo.ERR_INVALID_ARG  # overflow
    assert st(NULL, 0, NULL, 0, None, None, None, 0, 4, 0, 1.0, 0, 0, None) == rwo.OK  # M = 0
    at = lib.attention_forward  # (q, k, v, o, lse, BH, Sq, Sk, d, scale, causal, dtype, stream)
    assert at(X, X, X, X, None, 1, 16, 16, 96, 1.0, 0, 1, None) == rwo.ERR_UNSUPPORTED  # d = 96
    assert at(X, X, X, X, None, 1, 16, 16, 128, 1.0, 0, 0, None) == rwo.ERR_UNSUPPORTED  # fp32
    assert at(X, X, X, X, None, 1, 16, 16, 128, -1.0, 0, 1, None) == rwo.ERR_INVALID_ARG  # scale
    assert at(X, X, X, X, None, 1, 16, 16, 128, float("inf"), 0, 1, None) == rwo.ERR_INVALID_ARG
    assert at(NULL, NULL, NULL, NULL, None, 1, 16, 16, 128, 0.0, 0, 1, None) == rwo.ERR_INVALID_ARG  # 0: default
    assert at(X, X, X, X, None, 1, 16, 16, 128, 1.0, 2, 1, None) == rwo.ERR_INVALID_ARG  # causal flag
    assert at(X, X, X, X, None, 1, 0, 16, 128, 1.0, 0, 1, None) == rwo.ERR_INVALID_ARG  # Sq = 0
    assert at(X, X, X, X, None, 65536, 16, 16, 128, 1.0, 0, 1, None) == rwo.ERR_UNSUPPORTED  # BH
    assert at(X, X, X, X, None, 1, 2**31, 16, 128, 1.0, 0, 1, None) == rwo.ERR_UNSUPPORTED  # 32-bit rows
    assert at(X, X, X, X, None, 1, 16, 2**31, 128, 1.0, 0, 1, None) == rwo.ERR_UNSUPPORTED
    assert at(X, X, X, X, None, 1, 2**31 - 255, 16, 128, 1.0, 1, 1, None) == rwo.ERR_UNSUPPORTED  # causal rows
    assert at(NULL, NULL, NULL, NULL, None, 1, 16, 16, 128, 1.0, 0, 1, None) == rwo.ERR_INVALID_ARG  # pointers
    assert at(NULL, NULL, NULL, NULL, None, 0, 16, 16, 128, 1.0, 0, 1, None) == rwo.OK  # BH = 0


def test_status_strings(lib):
    for s in range(6):
        assert rwo.status_string(s)
    assert rwo.status_string(42) == "unknown status"


def test_debug_hooks_roundtrip(lib):
    old = rwo.debug_set_fault(1)
    assert rwo.debug_set_fault(old) == 1
    prev = rwo.debug_set_wait_limit_ns(12345)
    assert rwo.debug_set_wait_limit_ns(prev) == 12345


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(rwo, "_lib", None)
    monkeypatch.setattr(rwo, "_LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        rwo.capi()
