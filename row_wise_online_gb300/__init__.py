"""GB300-native row-wise online softmax: a thin Python binding of ``libsoftmax_rows.so``.

The library (C ABI in ``include/softmax_rows.h``, CUDA kernels in ``csrc/``) computes, for
each row of a row-major M x N matrix, the safe softmax with the online (m, d) recurrence
("5.2 CUDA Online Softmax 实现优化", §2) and the per-row state m, d, LSE.  This module only
marshals arguments: it turns torch tensors into device pointers and the current CUDA stream
into a ``cudaStream_t``.  Every step of the computation runs in the library's kernels; there
is no CPU fallback, and importing fails loudly if the library has not been built
(``python -m row_wise_online_gb300._build``).

PyTorch supplies device memory and streams only.
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "F32", "BF16", "VARIANT_AUTO", "VARIANT_ONEREAD_REG", "VARIANT_ONEREAD_SMEM", "VARIANT_TWOPASS",
    "VARIANT_SPLITROW", "VARIANT_SPLITROW_STREAM", "VARIANT_NAMES", "SoftmaxError", "softmax_rows", "softmax_rows_ex",
    "softmax_row_state", "merge_states", "softmax_rows_host", "get_status", "status_string",
    "last_variant", "debug_set_fault", "debug_set_wait_limit_ns", "capi", "library_path",
    "softmax_rows_splitrow_noalloc", "softmax_rows_causal",
]

F32, BF16, F16 = 0, 1, 2
(VARIANT_AUTO, VARIANT_ONEREAD_REG, VARIANT_ONEREAD_SMEM, VARIANT_TWOPASS, VARIANT_SPLITROW,
 VARIANT_SPLITROW_STREAM) = range(6)
VARIANT_NAMES = {VARIANT_AUTO: "auto", VARIANT_ONEREAD_REG: "oneread_reg",
                 VARIANT_ONEREAD_SMEM: "oneread_smem", VARIANT_TWOPASS: "twopass",
                 VARIANT_SPLITROW: "splitrow", VARIANT_SPLITROW_STREAM: "splitrow_stream"}

OK, ERR_INVALID_ARG, ERR_MISALIGNED, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT = range(6)

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "lib", "libsoftmax_rows.so")
_lib = None

EXPORTED = (
    "softmax_rows", "softmax_rows_ex", "softmax_row_state", "merge_states", "softmax_rows_host",
    "softmax_get_status", "softmax_status_string", "softmax_last_cuda_error", "softmax_last_variant",
    "softmax_debug_set_fault", "softmax_debug_set_wait_limit_ns", "softmax_rows_splitrow_noalloc",
    "softmax_rows_causal", "log_softmax_rows", "cross_entropy_rows", "softmax_rows_strided", "attention_forward",
)


class SoftmaxError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        msg = status_string(status)
        if status == ERR_CUDA:
            msg += ": " + capi().softmax_last_cuda_error().decode()
        super().__init__(f"{what}: {msg}" if what else msg)


def library_path() -> str:
    return _LIB_PATH


def capi() -> ctypes.CDLL:
    """The loaded C library with argument types declared (raises if it is not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise ImportError(
                f"{_LIB_PATH} is missing: build the CUDA library first "
                "(python -m row_wise_online_gb300._build); there is no fallback")
        lib = ctypes.CDLL(_LIB_PATH)
        vp, i64, ci, fp = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
        lib.softmax_rows.argtypes = [vp, vp, i64, i64, ci, vp]
        lib.softmax_rows_ex.argtypes = [vp, vp, fp, fp, fp, i64, i64, ci, ci, vp]
        lib.softmax_row_state.argtypes = [vp, fp, fp, fp, i64, i64, ci, vp]
        lib.merge_states.argtypes = [fp, fp, fp, fp, fp, fp, fp, i64, vp]
        lib.softmax_rows_host.argtypes = [vp, vp, i64, i64, ci, vp]
        lib.softmax_get_status.argtypes = [vp]
        lib.softmax_status_string.argtypes = [ci]
        lib.softmax_status_string.restype = ctypes.c_char_p
        lib.softmax_last_cuda_error.argtypes = []
        lib.softmax_last_cuda_error.restype = ctypes.c_char_p
        lib.softmax_last_variant.argtypes = []
        lib.softmax_debug_set_fault.argtypes = [ci]
        lib.softmax_debug_set_wait_limit_ns.argtypes = [i64]
        lib.softmax_rows_splitrow_noalloc.argtypes = [vp, vp, fp, fp, fp, i64, i64, ci, vp]
        lib.softmax_rows_causal.argtypes = [vp, vp, fp, fp, fp, i64, i64, i64, i64, ci, vp]
        lib.log_softmax_rows.argtypes = [vp, vp, fp, fp, fp, i64, i64, ci, ci, vp]
        lib.cross_entropy_rows.argtypes = [vp, vp, fp, fp, i64, i64, ci, vp]
        lib.softmax_rows_strided.argtypes = [vp, i64, vp, i64, fp, fp, fp, i64, i64, ci, ctypes.c_float, ci, ci, vp]
        lib.attention_forward.argtypes = [vp, vp, vp, vp, fp, i64, i64, i64, i64, ctypes.c_float, ci, ci, vp]
        lib.softmax_debug_set_wait_limit_ns.restype = i64
        for name in ("softmax_rows", "softmax_rows_ex", "softmax_row_state", "merge_states",
                     "softmax_rows_host", "softmax_get_status", "softmax_last_variant",
                     "softmax_debug_set_fault", "softmax_rows_splitrow_noalloc", "softmax_rows_causal",
                     "log_softmax_rows", "cross_entropy_rows", "softmax_rows_strided", "attention_forward"):
            getattr(lib, name).restype = ci
        _lib = lib
    return _lib


def status_string(status: int) -> str:
    return capi().softmax_status_string(int(status)).decode()


def _check(status: int, what: str) -> None:
    if status != OK:
        raise SoftmaxError(status, what)


def _stream(stream):
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream))


def _dtype_code(t) -> int:
    import torch

    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float16:
        return F16
    raise TypeError(f"unsupported dtype {t.dtype}: float32, bfloat16 or float16")


def _rows(t):
    """(M, N) of a contiguous tensor whose last dimension is the softmax axis."""
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous (row-major rows)")
    if t.dim() == 0:
        raise ValueError("tensor must have at least one dimension")
    N = int(t.shape[-1])
    M = int(t.numel() // N) if N else 0
    return M, N


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _state_out(t, M, name):
    import torch

    if t is None:
        return None
    if t.dtype != torch.float32 or t.numel() != M or not t.is_contiguous() or not t.is_cuda:
        raise ValueError(f"{name} must be a contiguous CUDA float32 tensor of {M} entries")
    return t


def softmax_rows_ex(x, y=None, m_out=None, d_out=None, lse_out=None, variant: int = VARIANT_AUTO,
                    stream=None):
    """y = softmax(x) along the last dimension, optionally with per-row m, d, LSE (fp32)."""
    import torch

    if not x.is_cuda:
        raise ValueError("x must be a CUDA tensor (use softmax_rows_host for host buffers)")
    M, N = _rows(x)
    if y is None:
        y = torch.empty_like(x)
    if y.shape != x.shape or y.dtype != x.dtype or not y.is_cuda or not y.is_contiguous():
        raise ValueError("y must be a contiguous CUDA tensor with x's shape and dtype")
    st = capi().softmax_rows_ex(_ptr(x), _ptr(y), _ptr(_state_out(m_out, M, "m_out")),
                                _ptr(_state_out(d_out, M, "d_out")), _ptr(_state_out(lse_out, M, "lse_out")),
                                M, N, _dtype_code(x), int(variant), _stream(stream))
    _check(st, "softmax_rows_ex")
    return y


def softmax_rows(x, y=None, stream=None):
    """y = softmax(x) along the last dimension (float32 or bfloat16 CUDA tensors)."""
    import torch

    if not x.is_cuda:
        raise ValueError("x must be a CUDA tensor (use softmax_rows_host for host buffers)")
    M, N = _rows(x)
    if y is None:
        y = torch.empty_like(x)
    if y.shape != x.shape or y.dtype != x.dtype or not y.is_cuda or not y.is_contiguous():
        raise ValueError("y must be a contiguous CUDA tensor with x's shape and dtype")
    _check(capi().softmax_rows(_ptr(x), _ptr(y), M, N, _dtype_code(x), _stream(stream)), "softmax_rows")
    return y


def softmax_rows_causal(x, q_period: int, key_offset: int = 0, y=None, m_out=None, d_out=None, lse_out=None,
                        stream=None):
    """Softmax of rows masked by position: row r keeps its first clamp(r % q_period + 1 + key_offset, 0, N)
    entries; the rest count as -inf, are never read, and give y = 0."""
    import torch

    if not x.is_cuda:
        raise ValueError("x must be a CUDA tensor")
    M, N = _rows(x)
    if y is None:
        y = torch.empty_like(x)
    if y.shape != x.shape or y.dtype != x.dtype or not y.is_cuda or not y.is_contiguous():
        raise ValueError("y must be a contiguous CUDA tensor with x's shape and dtype")
    st = capi().softmax_rows_causal(_ptr(x), _ptr(y), _ptr(_state_out(m_out, M, "m_out")),
                                    _ptr(_state_out(d_out, M, "d_out")), _ptr(_state_out(lse_out, M, "lse_out")),
                                    M, N, int(q_period), int(key_offset), _dtype_code(x), _stream(stream))
    _check(st, "softmax_rows_causal")
    return y


FLAG_LOG = 1


def _rows_strided(t):
    """(M, N, row pitch) of a 2-D tensor whose rows are contiguous (stride(1) == 1)."""
    if t.dim() != 2 or t.stride(1) != 1 or (t.shape[0] > 1 and t.stride(0) < t.shape[1]):
        raise ValueError("expected a 2-D tensor with contiguous rows (stride(1) == 1, stride(0) >= N)")
    return int(t.shape[0]), int(t.shape[1]), int(t.stride(0)) if t.shape[0] > 1 else int(t.shape[1])


def softmax_rows_strided(x, y=None, m_out=None, d_out=None, lse_out=None, scale: float = 1.0, log: bool = False,
                         variant: int = VARIANT_AUTO, stream=None):
    """softmax(scale * x) (or its log) along the last dimension of a 2-D tensor whose rows may be
    pitched (e.g. x[:, a:b] of a wider matrix).  y defaults to a new contiguous tensor."""
    import torch

    if not x.is_cuda:
        raise ValueError("x must be a CUDA tensor")
    M, N, ldx = _rows_strided(x)
    if y is None:
        y = torch.empty((M, N), dtype=x.dtype, device=x.device)
    if tuple(y.shape) != (M, N) or y.dtype != x.dtype or not y.is_cuda:
        raise ValueError("y must be a CUDA tensor with x's shape and dtype")
    _, _, ldy = _rows_strided(y)
    st = capi().softmax_rows_strided(_ptr(x), ldx, _ptr(y), ldy, _ptr(_state_out(m_out, M, "m_out")),
                                     _ptr(_state_out(d_out, M, "d_out")), _ptr(_state_out(lse_out, M, "lse_out")),
                                     M, N, _dtype_code(x), float(scale), FLAG_LOG if log else 0, int(variant),
                                     _stream(stream))
    _check(st, "softmax_rows_strided")
    return y


def attention_forward(q, k, v, o=None, lse_out=None, scale: float | None = None, causal: bool = False, stream=None):
    """O = softmax(scale Q K^T) V for q [BH, Sq, d], k and v [BH, Sk, d] (contiguous CUDA tensors; bf16 or
    fp16, d = 64 or 128).  scale defaults to 1/sqrt(d).  Returns o (and fills lse_out [BH, Sq] fp32 if given)."""
    import torch

    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        if not t.is_cuda or t.dim() != 3 or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous 3-D CUDA tensor")
    BH, Sq, d = (int(s) for s in q.shape)
    if k.shape != v.shape or k.shape[0] != BH or k.shape[2] != d or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("k and v must be [BH, Sk, d] with q's dtype")
    Sk = int(k.shape[1])
    if o is None:
        o = torch.empty_like(q)
    if lse_out is not None and (lse_out.dtype != torch.float32 or lse_out.numel() != BH * Sq or not lse_out.is_cuda):
        raise ValueError("lse_out must be a CUDA float32 tensor of BH * Sq entries")
    st = capi().attention_forward(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse_out), BH, Sq, Sk, d,
                                  0.0 if scale is None else float(scale),  # 0: the library's 1/sqrt(d)
                                  1 if causal else 0, _dtype_code(q), _stream(stream))
    _check(st, "attention_forward")
    return o


def log_softmax_rows(x, y=None, m_out=None, d_out=None, lse_out=None, variant: int = VARIANT_AUTO, stream=None):
    """y = log softmax(x) = x - LSE along the last dimension, optionally with per-row m, d, LSE (fp32)."""
    import torch

    if not x.is_cuda:
        raise ValueError("x must be a CUDA tensor")
    M, N = _rows(x)
    if y is None:
        y = torch.empty_like(x)
    if y.shape != x.shape or y.dtype != x.dtype or not y.is_cuda or not y.is_contiguous():
        raise ValueError("y must be a contiguous CUDA tensor with x's shape and dtype")
    st = capi().log_softmax_rows(_ptr(x), _ptr(y), _ptr(_state_out(m_out, M, "m_out")),
                                 _ptr(_state_out(d_out, M, "d_out")), _ptr(_state_out(lse_out, M, "lse_out")),
                                 M, N, _dtype_code(x), int(variant), _stream(stream))
    _check(st, "log_softmax_rows")
    return y


def cross_entropy_rows(x, labels, loss=None, lse_out=None, stream=None):
    """Per-row cross-entropy loss LSE_r - x[r, labels[r]] (fp32); labels int64, negative = ignored row (loss 0)."""
    import torch

    if not x.is_cuda:
        raise ValueError("x must be a CUDA tensor")
    M, N = _rows(x)
    if labels.dtype != torch.int64 or labels.numel() != M or not labels.is_contiguous() or not labels.is_cuda:
        raise ValueError(f"labels must be a contiguous CUDA int64 tensor of {M} entries")
    if loss is None:
        loss = torch.empty(M, dtype=torch.float32, device=x.device)
    st = capi().cross_entropy_rows(_ptr(x), _ptr(labels), _ptr(_state_out(loss, M, "loss")),
                                   _ptr(_state_out(lse_out, M, "lse_out")), M, N, _dtype_code(x), _stream(stream))
    _check(st, "cross_entropy_rows")
    return loss


def softmax_row_state(x, m_out=None, d_out=None, lse_out=None, stream=None):
    """Per-row (m, d, LSE) of x without writing y.  Returns (m_out, d_out, lse_out)."""
    import torch

    M, N = _rows(x)
    if m_out is None and d_out is None and lse_out is None:
        m_out = torch.empty(M, dtype=torch.float32, device=x.device)
        d_out = torch.empty(M, dtype=torch.float32, device=x.device)
        lse_out = torch.empty(M, dtype=torch.float32, device=x.device)
    st = capi().softmax_row_state(_ptr(x), _ptr(_state_out(m_out, M, "m_out")), _ptr(_state_out(d_out, M, "d_out")),
                                  _ptr(_state_out(lse_out, M, "lse_out")), M, N, _dtype_code(x), _stream(stream))
    _check(st, "softmax_row_state")
    return m_out, d_out, lse_out


def merge_states(m_a, d_a, m_b, d_b, m_out=None, d_out=None, lse_out=None, stream=None):
    """Elementwise merge of two state arrays.  Returns (m_out, d_out, lse_out)."""
    import torch

    M = int(m_a.numel())
    for t, n in ((m_a, "m_a"), (d_a, "d_a"), (m_b, "m_b"), (d_b, "d_b")):
        _state_out(t, M, n)
    if m_out is None:
        m_out = torch.empty_like(m_a)
    if d_out is None:
        d_out = torch.empty_like(d_a)
    st = capi().merge_states(_ptr(m_a), _ptr(d_a), _ptr(m_b), _ptr(d_b), _ptr(_state_out(m_out, M, "m_out")),
                             _ptr(_state_out(d_out, M, "d_out")), _ptr(_state_out(lse_out, M, "lse_out")), M,
                             _stream(stream))
    _check(st, "merge_states")
    return m_out, d_out, lse_out


def softmax_rows_host(x_host, y_host, stream=None):
    """softmax of a HOST tensor (ideally pinned) into a host tensor; synchronises before returning."""
    if x_host.is_cuda or y_host.is_cuda:
        raise ValueError("softmax_rows_host takes host tensors")
    M, N = _rows(x_host)
    if y_host.shape != x_host.shape or y_host.dtype != x_host.dtype or not y_host.is_contiguous():
        raise ValueError("y_host must be a contiguous host tensor with x_host's shape and dtype")
    _check(capi().softmax_rows_host(_ptr(x_host), _ptr(y_host), M, N, _dtype_code(x_host), _stream(stream)),
           "softmax_rows_host")
    return y_host


def softmax_rows_splitrow_noalloc(x, y=None, m_out=None, d_out=None, lse_out=None, stream=None):
    """Split-row softmax that allocates no device memory inside the library, for callers that
    cannot let a library allocate (see the C header: M x clusters <= 40960 slots; calls that
    overlap on the GPU race on the shared scratch)."""
    import torch

    if not x.is_cuda:
        raise ValueError("x must be a CUDA tensor")
    M, N = _rows(x)
    if y is None:
        y = torch.empty_like(x)
    if y.shape != x.shape or y.dtype != x.dtype or not y.is_cuda or not y.is_contiguous():
        raise ValueError("y must be a contiguous CUDA tensor with x's shape and dtype")
    st = capi().softmax_rows_splitrow_noalloc(_ptr(x), _ptr(y), _ptr(_state_out(m_out, M, "m_out")),
                                              _ptr(_state_out(d_out, M, "d_out")),
                                              _ptr(_state_out(lse_out, M, "lse_out")), M, N, _dtype_code(x),
                                              _stream(stream))
    _check(st, "softmax_rows_splitrow_noalloc")
    return y


def get_status(stream=None) -> int:
    """Synchronise the stream; return and clear the device status word (OK or ERR_TIMEOUT)."""
    return int(capi().softmax_get_status(_stream(stream)))


def last_variant() -> int:
    return int(capi().softmax_last_variant())


def debug_set_fault(fault: int) -> int:
    return int(capi().softmax_debug_set_fault(int(fault)))


def debug_set_wait_limit_ns(ns: int) -> int:
    return int(capi().softmax_debug_set_wait_limit_ns(int(ns)))
