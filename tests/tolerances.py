"""Parity tolerances between the CUDA path and the fp64 oracle, and the checks that apply them.

Tolerances (per element, against the oracle's exact fp64 result y_ref):
  * fp32 output: |y - y_ref| <= 1e-5 * |y_ref| + 2^-126
  * bf16 output: |y - y_ref| <= ulp_bf16(y_ref) + 2^-126, ulp_bf16(v) = 2^(floor(log2|v|) - 7)
    (one unit in the last place of bf16's 8-bit significand)
  * fp16 output: |y - y_ref| <= ulp_f16(y_ref) + 2^-126, ulp_f16(v) = 2^(max(floor(log2|v|), -14) - 10)
    (one unit in the last place of fp16's 11-bit significand; subnormal spacing below 2^-14)
  * row sums:    |sum_j y_j - 1| <= 1e-5 (fp32) / 4e-3 (bf16) / 1e-3 (fp16), rows not fully masked
  * m:           bit-exact (as fp32; -0 == +0)
  * d:           |d - d_ref| <= 1e-5 * d_ref
  * LSE:         |LSE - LSE_ref| <= 1e-5 * max(1, |LSE_ref|)
The 2^-126 floor admits results below the smallest normal fp32, which the hardware exponential
flushes to zero.  Fully masked rows (all -inf) must give y = 0, m = -inf, d = 0, LSE = -inf.

Log softmax and cross-entropy loss (values x_j - LSE and LSE - x_label; same arithmetic as LSE):
  * fp32 log y:  |v - v_ref| <= 1e-5 * max(1, |v_ref|)
  * bf16 log y:  |v - v_ref| <= ulp_bf16(v_ref) + 1e-5 * max(1, |v_ref|)
  * loss (fp32): |l - l_ref| <= 1e-5 * max(1, |l_ref|)
  -inf references (masked entries, log 0) must be -inf exactly; NaN references must be NaN.
"""
from __future__ import annotations

import numpy as np

import synth

TINY = 2.0 ** -126
Y_REL_F32 = 1e-5
ROWSUM_F32 = 1e-5
ROWSUM_BF16 = 4e-3
ROWSUM_F16 = 1e-3
D_REL = 1e-5
LSE_REL = 1e-5


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    a = np.abs(v)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.exp2(e - 7), 0.0)


def f16_ulp(v: np.ndarray) -> np.ndarray:
    """Spacing of fp16 at |v|: 2^(floor(log2|v|) - 10), 2^-24 in the subnormal range."""
    a = np.abs(v)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.exp2(np.maximum(e, -14.0) - 10)


def output_as_f64(y: np.ndarray, dtype: int) -> np.ndarray:
    if dtype == synth.BF16:
        return synth.bf16_to_f32(y).astype(np.float64)
    if dtype == synth.F16:
        return synth.f16_to_f32(y).astype(np.float64)
    return y.astype(np.float64)


def check_y(y: np.ndarray, y_ref: np.ndarray, dtype: int, what: str = "") -> dict:
    """Element-wise check; returns error statistics; raises AssertionError on a violation."""
    yg = output_as_f64(y, dtype)
    assert yg.shape == y_ref.shape, (yg.shape, y_ref.shape)
    err = np.abs(yg - y_ref)
    if dtype == synth.F32:
        bound = Y_REL_F32 * np.abs(y_ref) + TINY
    elif dtype == synth.F16:
        bound = f16_ulp(y_ref) + TINY
    else:
        bound = bf16_ulp(y_ref) + TINY
    bad = ~(err <= bound)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} elements out of tolerance; first at {tuple(i)}: "
                             f"y={yg[tuple(i)]!r} y_ref={y_ref[tuple(i)]!r} bound={bound[tuple(i)]!r}")
    nz = y_ref > TINY
    rel = err[nz] / y_ref[nz] if nz.any() else np.zeros(1)
    stats = {"max_abs": float(err.max()) if err.size else 0.0, "max_rel": float(rel.max()) if rel.size else 0.0}
    if dtype == synth.BF16:
        stats["n_above_2^-8_rel"] = int(np.count_nonzero(rel > 2.0 ** -8))
    return stats


def check_rowsums(y: np.ndarray, dtype: int, masked_rows=None, what: str = "") -> float:
    yg = output_as_f64(y, dtype)
    s = yg.sum(axis=1)
    keep = np.ones(len(s), bool) if masked_rows is None else ~np.asarray(masked_rows, bool)
    tol = ROWSUM_F32 if dtype == synth.F32 else ROWSUM_F16 if dtype == synth.F16 else ROWSUM_BF16
    dev = np.abs(s[keep] - 1.0)
    assert np.all(dev <= tol), f"{what}: row sum off by {dev.max()}"
    if masked_rows is not None:
        assert np.all(yg[~keep] == 0.0), f"{what}: fully masked rows must be zero"
    return float(dev.max()) if dev.size else 0.0


def check_state(m, d, lse, m_ref, d_ref, lse_ref, what: str = "") -> None:
    if m is not None:
        m32 = np.asarray(m, np.float32)
        ref32 = np.asarray(m_ref).astype(np.float32)
        assert np.all((m32 == ref32) | (np.isneginf(m32) & np.isneginf(ref32))), f"{what}: m not bit-exact"
    if d is not None:
        d = np.asarray(d, np.float64)
        ok = np.abs(d - d_ref) <= D_REL * d_ref
        ok |= (d_ref == 0) & (d == 0)
        assert np.all(ok), f"{what}: d off, max rel {np.max(np.abs(d - d_ref) / np.where(d_ref > 0, d_ref, 1))}"
    if lse is not None:
        lse = np.asarray(lse, np.float64)
        fin = np.isfinite(lse_ref)
        assert np.all(np.isneginf(lse[~fin])), f"{what}: LSE of fully masked rows must be -inf"
        ok = np.abs(lse[fin] - lse_ref[fin]) <= LSE_REL * np.maximum(1.0, np.abs(lse_ref[fin]))
        assert np.all(ok), f"{what}: LSE off"


def check_log_values(v: np.ndarray, v_ref: np.ndarray, dtype: int, what: str = "") -> float:
    """Log-softmax values (dtype output) or losses (fp32) against fp64 references; returns max abs error."""
    vg = output_as_f64(v, dtype)
    assert vg.shape == v_ref.shape, (vg.shape, v_ref.shape)
    ninf = np.isneginf(v_ref)
    pinf = np.isposinf(v_ref)
    nan = np.isnan(v_ref)
    assert np.all(np.isneginf(vg[ninf])), f"{what}: -inf references must give -inf"
    assert np.all(np.isposinf(vg[pinf])), f"{what}: +inf references must give +inf"
    assert np.all(np.isnan(vg[nan])), f"{what}: NaN references must give NaN"
    fin = ~(ninf | pinf | nan)
    err = np.abs(vg[fin] - v_ref[fin])
    bound = LSE_REL * np.maximum(1.0, np.abs(v_ref[fin]))
    if dtype == synth.BF16:
        bound = bound + bf16_ulp(v_ref[fin])
    elif dtype == synth.F16:
        bound = bound + f16_ulp(v_ref[fin])
    bad = ~(err <= bound)
    if bad.any():
        k = int(np.argmax(bad))
        idx = tuple(np.argwhere(fin)[k])
        raise AssertionError(f"{what}: {bad.sum()} values out of tolerance; first at {idx}: "
                             f"v={vg[idx]!r} v_ref={v_ref[idx]!r}")
    return float(err.max()) if err.size else 0.0
