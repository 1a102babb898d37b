"""Seeded synthetic inputs for the row-wise softmax workloads.

This module is shared by both sides of every parity check: the CUDA path's
tests and benchmark, and the fp64 oracle, read the same bytes.  It holds no
softmax arithmetic -- only a counter-based random source (splitmix64), value
distributions and structural edits, all in ``synth.c``.

The workloads follow the shapes of the pages' problem ("5.2 CUDA Online
Softmax 实现优化" §2.4 measures M = N = 4096 in fp32) and of the logits /
attention-score uses they describe:

=============================  =========  =========================================================
name                           M x N      recipe
=============================  =========  =========================================================
fp32_64x1024                   64x1024    fp32, x ~ N(0, 1), seed 0
fp32_4096x4096                 4096x4096  fp32, x = 3 * N(0, 1), seed 1
bf16_logits_16384x32768        16384x...  bf16, x ~ N(0, sd 2), seed 2; rows r % 100 == 0 get one +80 and
                                          one -80 entry at two hashed distinct columns
fp32_longrow_32x4194304        32x4Mi     fp32, x ~ U[-20, 20), seed 3; each row's unique max 20.0 sits in its
                                          last quarter at a hashed column
bf16_causal_4x32x4096x4096     524288x4k  bf16, x = bf16(z / sqrt(128)), z ~ N(0, 1), seed 4; row r is query
                                          q = r % 4096 and keys j > q are -inf
fp32_rows_600x262144           600x256Ki  fp32, x = 3 * N(0, 1), seed 5 (many 1 MiB rows: more than L2
                                          holds at a row per SM; not one of the pages' shapes)
=============================  =========  =========================================================

Every value depends only on (seed, global row, column), so any row range can
be generated alone (``row0``/``nrows``), which is how large workloads are
sharded across ranks and sampled for parity.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "libsynth.so")
_lock = threading.Lock()
_lib = None

F32 = 0
BF16 = 1
F16 = 2
NORMAL = 0
UNIFORM = 1


def build(force: bool = False) -> str:
    """Compile synth.c into libsynth.so next to it."""
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
            i64, u64, vp, ci, cd = ctypes.c_int64, ctypes.c_uint64, ctypes.c_void_p, ctypes.c_int, ctypes.c_double
            lib.synth_fill.argtypes = [vp, ci, i64, i64, i64, ci, cd, cd, u64, ci]
            lib.synth_stress_rows.argtypes = [vp, ci, i64, i64, i64, i64, cd, cd, u64]
            lib.synth_late_max.argtypes = [vp, ci, i64, i64, i64, cd, u64]
            lib.synth_late_max_col.argtypes = [i64, i64, u64]
            lib.synth_late_max_col.restype = i64
            lib.synth_causal_mask.argtypes = [vp, ci, i64, i64, i64, i64]
            for f in (lib.synth_fill, lib.synth_stress_rows, lib.synth_late_max, lib.synth_causal_mask):
                f.restype = ci
            _lib = lib
    return _lib


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise RuntimeError(f"{what} rejected its arguments")


def np_dtype(dtype: int):
    return np.float32 if dtype == F32 else np.uint16


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    dtype: int  # F32, BF16 or F16
    M: int
    N: int
    seed: int
    dist: int
    p0: float
    p1: float
    stress_period: int = 0  # rows r % period == 0 get (+hi, lo) entries; 0 = none
    stress_hi: float = 80.0
    stress_lo: float = -80.0
    late_max: float | None = None  # value placed in the last quarter of each row
    causal_q: int = 0  # rows are queries r % causal_q; keys beyond them are -inf; 0 = none

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == F32 else 2

    @property
    def min_bytes(self) -> int:
        """Read x once + write y once."""
        return 2 * self.M * self.N * self.elem_bytes

    def with_rows(self, M: int) -> "Workload":
        return dataclasses.replace(self, M=M)

    def late_max_col(self, r: int) -> int:
        return int(_load().synth_late_max_col(self.N, r, self.seed))


WORKLOADS = {
    w.name: w
    for w in (
        Workload("fp32_64x1024", F32, 64, 1024, 0, NORMAL, 0.0, 1.0),
        Workload("fp32_4096x4096", F32, 4096, 4096, 1, NORMAL, 0.0, 3.0),
        Workload("bf16_logits_16384x32768", BF16, 16384, 32768, 2, NORMAL, 0.0, 2.0, stress_period=100),
        Workload("fp32_longrow_32x4194304", F32, 32, 4194304, 3, UNIFORM, -20.0, 20.0, late_max=20.0),
        Workload("bf16_causal_4x32x4096x4096", BF16, 4 * 32 * 4096, 4096, 4, NORMAL, 0.0, 1.0 / np.sqrt(128.0),
                 causal_q=4096),
        Workload("fp32_rows_600x262144", F32, 600, 262144, 5, NORMAL, 0.0, 3.0),
    )
}


def custom(name: str, dtype: int, M: int, N: int, seed: int, dist: int = NORMAL, p0: float = 0.0,
           p1: float = 1.0, **kw) -> Workload:
    return Workload(name, dtype, M, N, seed, dist, p0, p1, **kw)


def fill(w: Workload, out_ptr: int, row0: int = 0, nrows: int | None = None, nthreads: int | None = None) -> None:
    """Write rows [row0, row0 + nrows) of workload ``w`` to host memory at ``out_ptr``
    (row-major, nrows x N, elements of w's dtype)."""
    if nrows is None:
        nrows = w.M - row0
    lib = _load()
    nt = nthreads or max(1, os.cpu_count() or 1)
    p = ctypes.c_void_p(out_ptr)
    _check(lib.synth_fill(p, w.dtype, w.N, row0, nrows, w.dist, w.p0, w.p1, w.seed, nt), "synth_fill")
    if w.stress_period:
        _check(lib.synth_stress_rows(p, w.dtype, w.N, row0, nrows, w.stress_period, w.stress_hi, w.stress_lo,
                                     w.seed), "synth_stress_rows")
    if w.late_max is not None:
        _check(lib.synth_late_max(p, w.dtype, w.N, row0, nrows, w.late_max, w.seed), "synth_late_max")
    if w.causal_q:
        _check(lib.synth_causal_mask(p, w.dtype, w.N, row0, nrows, w.causal_q), "synth_causal_mask")


def generate(w: Workload, row0: int = 0, nrows: int | None = None, nthreads: int | None = None) -> np.ndarray:
    """Rows [row0, row0 + nrows) of workload ``w`` as a numpy array (float32, or uint16 bf16 bits)."""
    if nrows is None:
        nrows = w.M - row0
    out = np.empty((nrows, w.N), dtype=np_dtype(w.dtype))
    if nrows:
        fill(w, out.ctypes.data, row0, nrows, nthreads)
    return out


def generate_rows(w: Workload, rows, nthreads: int | None = None) -> np.ndarray:
    """Selected (possibly scattered) global rows of ``w``, stacked in the given order."""
    rows = [int(r) for r in rows]
    out = np.empty((len(rows), w.N), dtype=np_dtype(w.dtype))
    for i, r in enumerate(rows):
        fill(w, out[i:i + 1].ctypes.data, r, 1, nthreads=1)
    return out


def f16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen fp16 bit patterns (uint16) to float32 exactly."""
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float32)


def f32_to_f16(a: np.ndarray) -> np.ndarray:
    """Round float32 to fp16 bit patterns, round-to-nearest-even (input encoding only)."""
    return np.ascontiguousarray(a, dtype=np.float32).astype(np.float16).view(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to float32 exactly (a bit shift)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16(a: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 bit patterns, round-to-nearest-even (input encoding only)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    nan = (u & 0x7F800000) == 0x7F800000
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    keep = (u >> 16).astype(np.uint16) | np.where((u & 0x7FFFFF) != 0, 0x40, 0).astype(np.uint16)
    return np.where(nan, keep, r).astype(np.uint16)
