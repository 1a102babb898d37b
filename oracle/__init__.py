"""fp64 CPU oracle for row-wise softmax -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline / reference leg may import this package.  The CUDA library and its
Python binding never do; the two sides share no code.

The arithmetic lives in ``oracle.c`` (plain C, double precision):

* ``softmax_rows`` -- the three-pass safe softmax of each row, the definition
  in "5.2 CUDA Online Softmax 实现优化" §1.1 and "Softmax 数值稳定性与
  IO-Aware Attention" §三, plus LSE = m + log d ("从原始Softmax到在线Softmax",
  section "softmax形式推导").
* ``log_softmax_rows`` -- log_probs = x - max - log(sum exp(x - max)), and
  ``cross_entropy_rows`` -- the per-row loss -log_probs[r, label_r]
  ("从原始Softmax到在线Softmax", section "softmax实际代码实现").
* ``attention_rows`` -- attention forward O = softmax(scale Q K^T) V (and LSE) for selected query
  rows, the plain definition of the worked example "标准 Attention 中的 Softmax"
  ("从原始Softmax到在线Softmax"); ``attention_online`` -- the same page's blocked (m, l, o~)
  recurrence for one query.
* ``online_state`` -- the element-by-element (m, d) recurrence,
  "5.2 CUDA Online Softmax 实现优化" §2.1.
* ``merge_state`` -- the merge of two partial states,
  "5.2 CUDA Online Softmax 实现优化" §4.1.

Readings where the pages are silent (also listed in the C source): the empty
state (-inf, 0) is the merge identity (exp(-inf - b) := 0); an all -inf row
gives y = 0, m = -inf, d = 0, LSE = -inf.

Every function is pinned by ``tests/test_oracle.py`` to values the pages print,
closed forms, mpmath brute force and library special cases.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

F32 = 0
BF16 = 1
F16 = 2


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (plain gcc, -O2)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", tmp, _SRC, "-lm"]
        )
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, dp, vp = ctypes.c_int64, ctypes.POINTER(ctypes.c_double), ctypes.c_void_p
            lib.oracle_softmax_rows_scaled.argtypes = [vp, ctypes.c_int, i64, vp, i64, ctypes.c_double, vp, vp, vp,
                                                       vp, ctypes.c_int]
            lib.oracle_softmax_rows_scaled.restype = ctypes.c_int
            lib.oracle_online_state.argtypes = [vp, i64, dp, dp]
            lib.oracle_online_state.restype = None
            lib.oracle_merge_state.argtypes = [ctypes.c_double] * 4 + [dp, dp]
            lib.oracle_merge_state.restype = None
            lib.oracle_log_softmax_rows.argtypes = [vp, ctypes.c_int, i64, vp, i64, ctypes.c_double, vp, ctypes.c_int]
            lib.oracle_log_softmax_rows.restype = ctypes.c_int
            lib.oracle_cross_entropy_rows.argtypes = [vp, ctypes.c_int, i64, vp, i64, vp, ctypes.c_int]
            lib.oracle_cross_entropy_rows.restype = ctypes.c_int
            lib.oracle_attention_rows.argtypes = [vp, vp, vp, ctypes.c_int, i64, i64, i64, ctypes.c_double,
                                                  ctypes.c_int, vp, i64, vp, vp, ctypes.c_int]
            lib.oracle_attention_rows.restype = ctypes.c_int
            lib.oracle_attention_online.argtypes = [vp, vp, i64, i64, i64, vp]
            lib.oracle_attention_online.restype = None
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def softmax_rows(x: np.ndarray, dtype: int | None = None, rows=None, *, want_y: bool = True,
                 nthreads: int | None = None, scale: float = 1.0):
    """Three-pass fp64 softmax of rows of a row-major matrix (of scale * x; exact in fp64).

    ``x`` is a 2-D float32 array, or a 2-D uint16 array of bf16 bit patterns.
    ``rows`` selects rows (default: all).  Returns ``(y, m, d, lse)`` as
    float64 arrays; ``y`` is None when ``want_y`` is False.
    """
    x = np.ascontiguousarray(x)
    if x.ndim != 2:
        raise ValueError("x must be 2-D")
    if dtype is None:
        dtype = F32 if x.dtype == np.float32 else BF16 if x.dtype == np.uint16 else None
    if dtype is None or (dtype == F32 and x.dtype != np.float32) or (dtype in (BF16, F16) and x.dtype != np.uint16):
        raise TypeError("x must be float32 (F32) or uint16 bf16 / fp16 bits (BF16 / F16, dtype given)")
    M, N = x.shape
    if rows is None:
        idx = None
        nrows = M
    else:
        idx = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        if idx.size and (idx.min() < 0 or idx.max() >= M):
            raise IndexError("row index out of range")
        nrows = idx.size
    y = np.empty((nrows, N), np.float64) if want_y else None
    m = np.empty(nrows, np.float64)
    d = np.empty(nrows, np.float64)
    lse = np.empty(nrows, np.float64)
    if nrows == 0:
        return y, m, d, lse
    if not scale > 0:
        raise ValueError("scale must be > 0")
    rc = _load().oracle_softmax_rows_scaled(_ptr(x), dtype, N, _ptr(idx), nrows, float(scale), _ptr(y), _ptr(m),
                                            _ptr(d), _ptr(lse), nthreads or default_threads())
    if rc != 0:
        raise RuntimeError("oracle_softmax_rows rejected its arguments")
    return y, m, d, lse


def _matrix(x, dtype):
    x = np.ascontiguousarray(x)
    if x.ndim != 2:
        raise ValueError("x must be 2-D")
    if dtype is None:
        dtype = F32 if x.dtype == np.float32 else BF16 if x.dtype == np.uint16 else None
    if dtype is None or (dtype == F32 and x.dtype != np.float32) or (dtype in (BF16, F16) and x.dtype != np.uint16):
        raise TypeError("x must be float32 (F32) or uint16 bf16 / fp16 bits (BF16 / F16, dtype given)")
    return x, dtype


def log_softmax_rows(x: np.ndarray, dtype: int | None = None, rows=None, *, nthreads: int | None = None,
                     scale: float = 1.0):
    """fp64 log softmax of rows of a row-major matrix (all -inf row: -inf).  Returns (nrows, N) float64."""
    x, dtype = _matrix(x, dtype)
    M, N = x.shape
    idx = None if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    if idx is not None and idx.size and (idx.min() < 0 or idx.max() >= M):
        raise IndexError("row index out of range")
    nrows = M if idx is None else idx.size
    ly = np.empty((nrows, N), np.float64)
    if nrows == 0:
        return ly
    rc = _load().oracle_log_softmax_rows(_ptr(x), dtype, N, _ptr(idx), nrows, float(scale), _ptr(ly),
                                         nthreads or default_threads())
    if rc != 0:
        raise RuntimeError("oracle_log_softmax_rows rejected its arguments")
    return ly


def cross_entropy_rows(x: np.ndarray, labels, dtype: int | None = None, *, nthreads: int | None = None):
    """fp64 per-row cross-entropy loss against int labels (negative: 0; >= N: NaN).  Returns (M,) float64."""
    x, dtype = _matrix(x, dtype)
    M, N = x.shape
    lab = np.ascontiguousarray(np.asarray(labels, dtype=np.int64).reshape(-1))
    if lab.size != M:
        raise ValueError("one label per row")
    loss = np.empty(M, np.float64)
    if M == 0:
        return loss
    rc = _load().oracle_cross_entropy_rows(_ptr(x), dtype, N, _ptr(lab), M, _ptr(loss), nthreads or default_threads())
    if rc != 0:
        raise RuntimeError("oracle_cross_entropy_rows rejected its arguments")
    return loss


def attention_rows(q, k, v, rows, *, dtype: int | None = None, scale: float | None = None, causal: bool = False,
                   nthreads: int | None = None):
    """fp64 attention forward for selected query rows: O = softmax(scale Q K^T) V, and LSE.

    q: [BH, Sq, d], k and v: [BH, Sk, d] (float32, or uint16 bf16 / fp16 bits with dtype given);
    rows: sequence of (head, query row).  scale defaults to 1/sqrt(d); causal: row i sees keys
    j <= i + Sk - Sq.  Returns (o [nrows, d], lse [nrows]) as float64."""
    q, k, v = (np.ascontiguousarray(a) for a in (q, k, v))
    if q.ndim != 3 or k.shape != v.shape or k.ndim != 3 or q.shape[0] != k.shape[0] or q.shape[2] != k.shape[2]:
        raise ValueError("q [BH, Sq, d], k and v [BH, Sk, d]")
    if dtype is None:
        dtype = F32 if q.dtype == np.float32 else BF16
    BH, Sq, d = q.shape
    Sk = k.shape[1]
    sel = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 2))
    if sel.size and (sel[:, 0].min() < 0 or sel[:, 0].max() >= BH or sel[:, 1].min() < 0 or sel[:, 1].max() >= Sq):
        raise IndexError("row out of range")
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    o = np.empty((len(sel), d), np.float64)
    lse = np.empty(len(sel), np.float64)
    if len(sel) == 0:
        return o, lse
    rc = _load().oracle_attention_rows(_ptr(q), _ptr(k), _ptr(v), dtype, Sq, Sk, d, float(scale), int(bool(causal)),
                                       _ptr(sel), len(sel), _ptr(o), _ptr(lse), nthreads or default_threads())
    if rc != 0:
        raise RuntimeError("oracle_attention_rows rejected its arguments")
    return o, lse


def attention_online(scores, v, block: int):
    """The blocked (m, l, o~) recurrence for one query: scores [n], v [n, d] (float64)."""
    s = np.ascontiguousarray(np.asarray(scores, dtype=np.float64).reshape(-1))
    vv = np.ascontiguousarray(np.asarray(v, dtype=np.float64).reshape(len(s), -1))
    o = np.empty(vv.shape[1], np.float64)
    _load().oracle_attention_online(_ptr(s), _ptr(vv), len(s), vv.shape[1], int(block), _ptr(o))
    return o


def online_state(xs) -> tuple[float, float]:
    """The (m, d) recurrence over a 1-D sequence, starting from (-inf, 0)."""
    a = np.ascontiguousarray(np.asarray(xs, dtype=np.float64).reshape(-1))
    m, d = ctypes.c_double(), ctypes.c_double()
    _load().oracle_online_state(_ptr(a) if a.size else None, a.size, ctypes.byref(m), ctypes.byref(d))
    return m.value, d.value


def merge_state(a, b) -> tuple[float, float]:
    """Merge two partial states ``a = (m_a, d_a)`` and ``b = (m_b, d_b)``."""
    m, d = ctypes.c_double(), ctypes.c_double()
    _load().oracle_merge_state(float(a[0]), float(a[1]), float(b[0]), float(b[1]), ctypes.byref(m),
                               ctypes.byref(d))
    return m.value, d.value
