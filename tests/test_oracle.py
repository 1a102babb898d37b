"""Pins of the fp64 oracle to things other than itself (CPU only).

Each test ties one part of the oracle to a value the pages print, a closed
form, an exact invariant, a library special case, or a 50-digit brute force,
so that a dropped term, a wrong sign, a wrong row index or a transposed
operand fails at least one of them.
"""
import itertools
import math
import os
import random

import mpmath
import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "p3_worked_examples.txt")


def _parse_golden():
    cases = []
    with open(GOLDEN, encoding="utf-8") as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            kind, *fields = line.split()
            kv = {}
            for f in fields:
                k, v = f.split("=", 1)
                kv[k] = v
            cases.append((kind, kv))
    return cases


def _vec(s):
    return [float(t) for t in s.split(",")]


def _f32(rows):
    return np.asarray(rows, dtype=np.float32).reshape(len(rows), -1)


def test_golden_worked_examples():
    """Every worked example of "从原始Softmax到在线Softmax" (section "手推小例子")."""
    cases = _parse_golden()
    assert len(cases) >= 10
    for kind, kv in cases:
        tol = float(kv["tol"])
        if kind == "softmax":
            x = np.asarray(_vec(kv["x"]), dtype=np.float64)
            # the printed inputs are decimal; feed the fp32 nearest (what a kernel would see)
            y, m, d, lse = oracle.softmax_rows(_f32([x]))
            assert np.allclose(y[0], _vec(kv["p"]), rtol=0, atol=tol), (kv, y)
            if "sum" in kv:
                assert abs(y[0].sum() - float(kv["sum"])) <= tol
        elif kind == "cross_entropy":
            x = _vec(kv["x"])
            label = int(kv["label"])
            y, m, d, lse = oracle.softmax_rows(_f32([x]))
            xl = float(np.float32(x[label]))
            assert abs((lse[0] - xl) - float(kv["loss"])) <= tol
            assert abs(-math.log(y[0][label]) - float(kv["loss"])) <= tol
            # the oracle's own cross-entropy and log-softmax functions
            assert abs(oracle.cross_entropy_rows(_f32([x]), [label])[0] - float(kv["loss"])) <= tol
            assert abs(-oracle.log_softmax_rows(_f32([x]))[0, label] - float(kv["loss"])) <= tol
        elif kind == "state":
            x = _vec(kv["x"])
            m, d = oracle.online_state(x)
            assert m == float(kv["m"])
            assert abs(d - float(kv["d"])) <= tol
            _, m3, d3, _ = oracle.softmax_rows(np.asarray([x], dtype=np.float32), want_y=False)
            assert abs(d3[0] - float(kv["d"])) <= tol
        elif kind == "attention":
            mat = lambda t: np.array([[float(x) for x in r.split(",")] for r in t.split(";")], np.float32)
            q, k, v, o_page = mat(kv["q"]), mat(kv["k"]), mat(kv["v"]), mat(kv["o"])
            o, _ = oracle.attention_rows(q[None], k[None], v[None], [(0, i) for i in range(len(q))],
                                         scale=1.0 / math.sqrt(q.shape[1]))
            assert np.allclose(o, o_page, rtol=0, atol=tol), (o, o_page)
        elif kind == "attention_online":
            sc = _vec(kv["s"])
            v = np.array([[float(x) for x in r.split(",")] for r in kv["v"].split(";")])
            o = oracle.attention_online(sc, v, int(kv["block"]))
            assert np.allclose(o, _vec(kv["o"]), rtol=0, atol=tol) and np.allclose(o, _vec(kv["o_online"]), rtol=0, atol=tol)
        elif kind == "merge":
            a = _vec(kv["a"])
            b = _vec(kv["b"])
            m, d = oracle.merge_state(a, b)
            assert m == float(kv["m"])
            assert abs(d - float(kv["d"])) <= tol
            if "scale_old" in kv:
                assert abs(math.exp(a[0] - m) - float(kv["scale_old"])) <= tol
        else:  # pragma: no cover
            raise AssertionError(f"unknown golden kind {kind}")


def _mp_softmax(row):
    """50-digit softmax of one row of finite values (brute force, independent of the oracle)."""
    with mpmath.workdps(50):
        xs = [mpmath.mpf(float(v)) for v in row]
        m = max(xs)
        es = [mpmath.e ** (v - m) for v in xs]
        d = mpmath.fsum(es)
        return [float(e / d) for e in es], float(m), float(d), float(m + mpmath.log(d))


def test_mpmath_brute_force_rectangular():
    """Non-square random inputs, each row against a 50-digit brute force (catches transposes and row indexing)."""
    rng = np.random.default_rng(7)
    for M, N in [(3, 5), (5, 3), (4, 17), (1, 1), (2, 64)]:
        x = (rng.standard_normal((M, N)) * 4).astype(np.float32)
        y, m, d, lse = oracle.softmax_rows(x)
        for r in range(M):
            ym, mm, dm, lm = _mp_softmax(x[r])
            np.testing.assert_allclose(y[r], ym, rtol=1e-14, atol=0)
            assert m[r] == mm
            assert abs(d[r] - dm) <= 1e-14 * dm
            assert abs(lse[r] - lm) <= 1e-14 * max(1.0, abs(lm))


def test_row_sum_is_one():
    x = synth.generate(synth.WORKLOADS["fp32_64x1024"])
    y, m, d, lse = oracle.softmax_rows(x)
    assert np.all(np.abs(y.sum(axis=1) - 1.0) <= 1e-12)
    assert np.all(y >= 0)


def test_shift_invariance_exact_shift():
    """softmax(x + c) = softmax(x); m shifts by c, d is unchanged ("Softmax 数值稳定性与 IO-Aware Attention" §2.1)."""
    rng = np.random.default_rng(1)
    base = (np.round(rng.uniform(-8, 8, size=(6, 257)) * 1024) / 1024).astype(np.float32)
    y0, m0, d0, l0 = oracle.softmax_rows(base)
    for c in (1024.0, -1024.0):
        shifted = (base.astype(np.float64) + c).astype(np.float32)
        assert np.array_equal(shifted.astype(np.float64) - c, base.astype(np.float64))  # shift is exact
        y1, m1, d1, l1 = oracle.softmax_rows(shifted)
        np.testing.assert_allclose(y1, y0, rtol=1e-12, atol=0)
        assert np.array_equal(m1, m0 + c)
        np.testing.assert_allclose(d1, d0, rtol=1e-12)
        np.testing.assert_allclose(l1, l0 + c, rtol=1e-14)


def test_uniform_row_closed_form():
    for N in (1, 2, 64, 1024, 4096):
        x = np.full((2, N), 3.25, dtype=np.float32)
        y, m, d, lse = oracle.softmax_rows(x)
        assert np.all(y == 1.0 / N)
        assert np.all(m == 3.25) and np.all(d == N)
        np.testing.assert_allclose(lse, 3.25 + math.log(N), rtol=1e-15)


def test_two_elements_logistic():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((50, 2)).astype(np.float32) * 5
    y, _, _, _ = oracle.softmax_rows(x)
    x64 = x.astype(np.float64)
    expect = 1.0 / (1.0 + np.exp(x64[:, 1] - x64[:, 0]))
    np.testing.assert_allclose(y[:, 0], expect, rtol=1e-14)
    np.testing.assert_allclose(y[:, 1], 1.0 / (1.0 + np.exp(x64[:, 0] - x64[:, 1])), rtol=1e-14)


def test_one_huge_value_is_one_hot_without_overflow():
    """A single huge entry ("5.2 CUDA Online Softmax 实现优化" §2.3: exponents stay <= 0)."""
    rng = np.random.default_rng(4)
    for big in (1e4, 1e30):
        x = rng.standard_normal((3, 100)).astype(np.float32)
        x[:, 37] = big
        y, m, d, lse = oracle.softmax_rows(x)
        assert np.all(np.isfinite(y)) and np.all(np.isfinite(d))
        assert np.all(y[:, 37] == 1.0)
        assert np.all(np.delete(y, 37, axis=1) == 0.0)
        assert np.all(m == np.float32(big)) and np.all(d == 1.0)


def test_huge_negative_rows():
    """Very negative entries ("Softmax 数值稳定性与 IO-Aware Attention" §9.2): behaves like the shifted row."""
    x = np.full((1, 33), -1e30, dtype=np.float32)
    y, m, d, lse = oracle.softmax_rows(x)
    assert np.all(y == 1.0 / 33) and d[0] == 33.0
    rng = np.random.default_rng(5)
    z = (np.round(rng.uniform(-4, 4, size=(2, 40)) * 256) / 256).astype(np.float32)
    shifted = (z.astype(np.float64) - 30000.0).astype(np.float32)
    assert np.array_equal(shifted.astype(np.float64) + 30000.0, z.astype(np.float64))
    y1, _, d1, _ = oracle.softmax_rows(shifted)
    y0, _, d0, _ = oracle.softmax_rows(z)
    np.testing.assert_allclose(y1, y0, rtol=1e-10)
    np.testing.assert_allclose(d1, d0, rtol=1e-10)


def test_masked_entries_reduce_to_shorter_row():
    """-inf entries carry zero weight; the rest is the softmax of the unmasked entries."""
    rng = np.random.default_rng(6)
    x = rng.standard_normal((4, 20)).astype(np.float32)
    mask = rng.random((4, 20)) < 0.4
    mask[:, 3] = False
    xm = np.where(mask, -np.inf, x).astype(np.float32)
    y, m, d, lse = oracle.softmax_rows(xm)
    for r in range(4):
        keep = ~mask[r]
        ym, mm, dm, lm = _mp_softmax(x[r][keep])
        assert np.all(y[r][mask[r]] == 0.0)
        np.testing.assert_allclose(y[r][keep], ym, rtol=1e-14)
        assert m[r] == mm and abs(d[r] - dm) <= 1e-14 * dm


def test_fully_masked_row_reading():
    x = np.full((2, 7), -np.inf, dtype=np.float32)
    x[1, 2] = 0.5
    y, m, d, lse = oracle.softmax_rows(x)
    assert np.all(y[0] == 0.0) and m[0] == -np.inf and d[0] == 0.0 and lse[0] == -np.inf
    assert y[1, 2] == 1.0 and np.sum(y[1]) == 1.0 and d[1] == 1.0 and lse[1] == 0.5


def test_log_softmax_identity():
    """log y_j = x_j - LSE ("从原始Softmax到在线Softmax", log-softmax)."""
    x = synth.generate(synth.WORKLOADS["fp32_64x1024"], nrows=8)
    y, m, d, lse = oracle.softmax_rows(x)
    np.testing.assert_allclose(np.log(y), x.astype(np.float64) - lse[:, None], rtol=0, atol=1e-12)


def test_library_special_case_torch_and_scipy():
    import scipy.special
    import torch

    x = synth.generate(synth.WORKLOADS["fp32_4096x4096"], row0=10, nrows=6)
    y, m, d, lse = oracle.softmax_rows(x)
    ref = torch.softmax(torch.from_numpy(x).double(), dim=-1).numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-13, atol=1e-300)
    np.testing.assert_allclose(y, scipy.special.softmax(x.astype(np.float64), axis=1), rtol=1e-13, atol=1e-300)
    np.testing.assert_allclose(lse, scipy.special.logsumexp(x.astype(np.float64), axis=1), rtol=1e-14)


def test_online_recurrence_equals_three_pass():
    """"5.2 CUDA Online Softmax 实现优化" §2.3: the online d equals the three-pass d."""
    x = synth.generate(synth.WORKLOADS["fp32_64x1024"])
    _, m3, d3, _ = oracle.softmax_rows(x, want_y=False)
    for r in range(x.shape[0]):
        m, d = oracle.online_state(x[r].astype(np.float64))
        assert m == m3[r]
        assert abs(d - d3[r]) <= 1e-13 * d3[r]
    rng = np.random.default_rng(8)
    for n in range(1, 65):
        row = (rng.standard_normal(n) * 10).astype(np.float32)
        m, d = oracle.online_state(row.astype(np.float64))
        _, mm, dm, _ = _mp_softmax(row)
        assert m == mm and abs(d - dm) <= 1e-13 * dm


def test_online_state_of_empty_and_masked_sequences():
    assert oracle.online_state([]) == (-math.inf, 0.0)
    assert oracle.online_state([-math.inf, -math.inf]) == (-math.inf, 0.0)
    m, d = oracle.online_state([-math.inf, 1.0, -math.inf])
    assert m == 1.0 and d == 1.0


def _bracketings(states):
    """Every full binary bracketing of the sequence, each merged with the oracle merge."""
    if len(states) == 1:
        yield states[0]
        return
    for k in range(1, len(states)):
        for left in _bracketings(states[:k]):
            for right in _bracketings(states[k:]):
                yield oracle.merge_state(left, right)


def test_merge_of_random_chunks_equals_whole_row():
    """"Softmax 数值稳定性与 IO-Aware Attention" §4.1: cut a row at random, merge the chunk states in any
    bracketing and either order; the result is the whole-row state."""
    rng = random.Random(11)
    nprng = np.random.default_rng(11)
    for trial in range(60):
        n = rng.randint(1, 40)
        row = (nprng.standard_normal(n) * rng.choice([1.0, 5.0, 30.0])).astype(np.float64)
        if trial % 5 == 0:
            row[: n // 2] = -np.inf  # an all -inf chunk
        _, mw, dw, _ = oracle.softmax_rows(row.astype(np.float32)[None, :], want_y=False)
        row = row.astype(np.float32).astype(np.float64)
        nchunks = rng.randint(1, 8 if trial % 2 else 5)
        cuts = sorted(rng.randint(0, n) for _ in range(nchunks - 1))  # repeated cuts = empty chunks
        bounds = [0] + cuts + [n]
        states = [oracle.online_state(row[a:b]) for a, b in zip(bounds[:-1], bounds[1:])]
        if all(s[0] == -math.inf for s in states):
            continue
        results = list(_bracketings(states)) if len(states) <= 5 else []
        # left fold, right fold, and reversed order
        acc = (-math.inf, 0.0)
        for s in states:
            acc = oracle.merge_state(acc, s)
        results.append(acc)
        acc = (-math.inf, 0.0)
        for s in reversed(states):
            acc = oracle.merge_state(s, acc)
        results.append(acc)
        for m, d in results:
            assert m == mw[0]
            assert abs(d - dw[0]) <= 1e-13 * dw[0], (trial, d, dw[0])


def test_merge_identity_and_commutativity():
    e = (-math.inf, 0.0)
    assert oracle.merge_state(e, e) == e
    assert oracle.merge_state(e, (2.0, 3.5)) == (2.0, 3.5)
    assert oracle.merge_state((2.0, 3.5), e) == (2.0, 3.5)
    a, b = (1.25, 2.0), (-0.5, 7.0)
    assert oracle.merge_state(a, b) == oracle.merge_state(b, a)
    m, d = oracle.merge_state(a, b)
    assert m == 1.25 and abs(d - (2.0 + 7.0 * math.exp(-1.75))) <= 1e-15 * d


def test_bf16_input_is_widened_exactly():
    rng = np.random.default_rng(9)
    f = (rng.standard_normal((5, 300)) * 3).astype(np.float32)
    bits = synth.f32_to_bf16(f)
    widened = synth.bf16_to_f32(bits)
    yb, mb, db, lb = oracle.softmax_rows(bits)
    yf, mf, df, lf = oracle.softmax_rows(widened)
    assert np.array_equal(yb, yf) and np.array_equal(mb, mf) and np.array_equal(db, df)


def test_row_selection_matches_full_computation():
    x = synth.generate(synth.WORKLOADS["fp32_64x1024"])
    y, m, d, lse = oracle.softmax_rows(x)
    sel = [63, 0, 17, 17, 5]
    ys, ms, ds, ls = oracle.softmax_rows(x, rows=sel)
    assert np.array_equal(ys, y[sel]) and np.array_equal(ms, m[sel]) and np.array_equal(ds, d[sel])


def test_threads_do_not_change_results():
    x = synth.generate(synth.WORKLOADS["fp32_64x1024"])
    a = oracle.softmax_rows(x, nthreads=1)
    b = oracle.softmax_rows(x, nthreads=7)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


def test_bad_arguments_are_rejected():
    with pytest.raises(TypeError):
        oracle.softmax_rows(np.zeros((2, 2), np.float64))
    with pytest.raises(IndexError):
        oracle.softmax_rows(np.zeros((2, 2), np.float32), rows=[2])


# ---------------------------------------------------------------------------------------------
# log softmax and cross entropy ("从原始Softmax到在线Softmax", section "softmax实际代码实现")
# ---------------------------------------------------------------------------------------------


def _mp_log_softmax(row):
    """50-digit log softmax with no max subtraction: x_j - log(sum_k exp(x_k))."""
    with mpmath.workdps(50):
        xs = [mpmath.mpf(float(v)) for v in row]
        lse = mpmath.log(mpmath.fsum(mpmath.exp(v) for v in xs))
        return np.array([float(v - lse) for v in xs])


def test_log_softmax_mpmath_brute_force():
    rng = np.random.default_rng(11)
    for M, N in [(3, 5), (5, 3), (4, 33), (1, 1), (2, 64)]:
        x = (rng.standard_normal((M, N)) * 6).astype(np.float32)
        ly = oracle.log_softmax_rows(x)
        assert ly.shape == (M, N)
        for r in range(M):
            ref = _mp_log_softmax(x[r])
            np.testing.assert_allclose(ly[r], ref, rtol=1e-14, atol=1e-14)


def test_log_softmax_closed_forms():
    # uniform row of 2^k entries: -ln(2^k) everywhere
    for k in (0, 3, 10):
        ly = oracle.log_softmax_rows(np.full((1, 1 << k), 1.25, np.float32))
        np.testing.assert_allclose(ly, -k * math.log(2.0), rtol=0, atol=1e-15)
    # two elements: log y_0 = -log1p(exp(x_1 - x_0)) (softplus)
    for a, b in [(0.0, 0.0), (3.0, -1.5), (-2.0, 7.0), (40.0, -40.0)]:
        ly = oracle.log_softmax_rows(np.array([[a, b]], np.float32))
        assert abs(ly[0, 0] + math.log1p(math.exp(b - a))) <= 1e-15 * max(1.0, abs(b - a))
        assert abs(ly[0, 1] + math.log1p(math.exp(a - b))) <= 1e-15 * max(1.0, abs(b - a))
    # shift invariance, with values on a 1/64 grid so that x + c is exact in fp32
    x = (np.round(np.random.default_rng(2).standard_normal((3, 50)) * 3 * 64) / 64).astype(np.float32)
    for c in (1024.0, -1024.0):
        np.testing.assert_allclose(oracle.log_softmax_rows(x + np.float32(c)), oracle.log_softmax_rows(x),
                                   rtol=0, atol=1e-12)


def test_log_softmax_masked_rows_and_selection():
    x = np.array([[1.0, -np.inf, 2.0, -np.inf], [-np.inf] * 4, [0.5, 0.5, -np.inf, 3.0]], np.float32)
    ly = oracle.log_softmax_rows(x)
    assert np.all(np.isneginf(ly[1]))                       # all -inf row: log 0
    assert np.isneginf(ly[0, 1]) and np.isneginf(ly[0, 3])  # masked entries: log 0
    np.testing.assert_allclose(ly[0, [0, 2]], _mp_log_softmax([1.0, 2.0]), rtol=1e-15)
    np.testing.assert_allclose(oracle.log_softmax_rows(x, rows=[2, 0]), ly[[2, 0]], rtol=0, atol=0)
    # bf16 bits are widened exactly
    xb = synth.f32_to_bf16(x)
    np.testing.assert_array_equal(oracle.log_softmax_rows(xb), ly)


def test_cross_entropy_against_brute_force_and_label_rules():
    rng = np.random.default_rng(4)
    x = (rng.standard_normal((6, 19)) * 5).astype(np.float32)
    labels = np.array([0, 18, 7, -1, 19, -100])
    loss = oracle.cross_entropy_rows(x, labels)
    for r in (0, 1, 2):
        assert abs(loss[r] + _mp_log_softmax(x[r])[labels[r]]) <= 1e-14 * max(1.0, abs(loss[r]))
    assert loss[3] == 0.0 and loss[5] == 0.0   # negative label: ignored row
    assert math.isnan(loss[4])                  # label >= N
    # loss >= 0, and equals the page's -log p of the labelled class
    y, *_ = oracle.softmax_rows(x[:3])
    np.testing.assert_allclose(loss[:3], -np.log(y[np.arange(3), labels[:3]]), rtol=1e-13)
    # masked labelled entry: -log 0 = +inf; all -inf row: NaN
    xm = np.array([[1.0, -np.inf], [-np.inf, -np.inf]], np.float32)
    lm = oracle.cross_entropy_rows(xm, [1, 0])
    assert np.isposinf(lm[0]) and math.isnan(lm[1])


def test_f16_input_is_widened_exactly():
    """Every finite fp16 bit pattern: the oracle's widening equals numpy's float16 -> float64 (a
    one-element row's m is the value itself); and a softmax of fp16 data equals the softmax of
    the same values given as fp32."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = bits.view(np.float16)
    fin = np.isfinite(vals)
    rows = bits[fin].reshape(-1, 1)
    _, m, d, lse = oracle.softmax_rows(rows, dtype=oracle.F16, want_y=False)
    np.testing.assert_array_equal(m, vals[fin].astype(np.float64))
    assert np.all(d == 1.0)
    rng = np.random.default_rng(5)
    x16 = (rng.standard_normal((6, 77)) * 6).astype(np.float16)
    y16, m16, d16, l16 = oracle.softmax_rows(x16.view(np.uint16), dtype=oracle.F16)
    y32, m32, d32, l32 = oracle.softmax_rows(x16.astype(np.float32))
    for a, b in ((y16, y32), (m16, m32), (d16, d32), (l16, l32)):
        np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(oracle.log_softmax_rows(x16.view(np.uint16), dtype=oracle.F16),
                                  oracle.log_softmax_rows(x16.astype(np.float32)))


def test_scaled_softmax_pins():
    """softmax(scale * x): a power-of-two scale equals the pre-multiplied input exactly; any other
    scale (here fp32(1/sqrt(128)), attention's 1/sqrt(d)) against a 50-digit brute force."""
    rng = np.random.default_rng(21)
    x = (rng.standard_normal((5, 40)) * 4).astype(np.float32)
    for k in (-3, 1, 4):
        a = oracle.softmax_rows(x, scale=2.0 ** k)
        b = oracle.softmax_rows((x * np.float32(2.0 ** k)).astype(np.float32))
        for u, v in zip(a, b):
            np.testing.assert_array_equal(u, v)
        np.testing.assert_array_equal(oracle.log_softmax_rows(x, scale=2.0 ** k),
                                      oracle.log_softmax_rows((x * np.float32(2.0 ** k)).astype(np.float32)))
    s = float(np.float32(1.0 / np.sqrt(128.0)))
    y, m, d, lse = oracle.softmax_rows(x, scale=s)
    ly = oracle.log_softmax_rows(x, scale=s)
    for r in range(x.shape[0]):
        with mpmath.workdps(50):
            z = [mpmath.mpf(s) * mpmath.mpf(float(v)) for v in x[r]]
            mz = max(z)
            dz = mpmath.fsum(mpmath.exp(t - mz) for t in z)
            for j in range(x.shape[1]):
                assert abs(y[r, j] - float(mpmath.exp(z[j] - mz) / dz)) <= 1e-15 * y[r, j] + 1e-300
                assert abs(ly[r, j] - float(z[j] - mz - mpmath.log(dz))) <= 1e-14 * max(1.0, abs(ly[r, j]))
            assert m[r] == float(mz)
            assert abs(d[r] - float(dz)) <= 1e-14 * float(dz)
    with pytest.raises(ValueError):
        oracle.softmax_rows(x, scale=0.0)


# ---------------------------------------------------------------------------------------------
# attention forward ("从原始Softmax到在线Softmax": the attention example and the blocked recurrence)
# ---------------------------------------------------------------------------------------------


def _mp_attention(q, k, v, scale, nk):
    with mpmath.workdps(40):
        s = [mpmath.mpf(scale) * mpmath.fsum(mpmath.mpf(float(a)) * mpmath.mpf(float(b)) for a, b in zip(q, k[j]))
             for j in range(nk)]
        m = max(s)
        p = [mpmath.exp(t - m) for t in s]
        l = mpmath.fsum(p)
        o = [float(mpmath.fsum(p[j] * mpmath.mpf(float(v[j][c])) for j in range(nk)) / l) for c in range(v.shape[1])]
        return np.array(o), float(m + mpmath.log(l))


def test_attention_brute_force_and_causal_rule():
    rng = np.random.default_rng(40)
    BH, Sq, Sk, d = 2, 5, 7, 6
    q = rng.standard_normal((BH, Sq, d)).astype(np.float32)
    k = rng.standard_normal((BH, Sk, d)).astype(np.float32)
    v = rng.standard_normal((BH, Sk, d)).astype(np.float32)
    rows = [(h, i) for h in range(BH) for i in range(Sq)]
    for causal in (False, True):
        o, lse = oracle.attention_rows(q, k, v, rows, scale=0.3, causal=causal)
        for t, (h, i) in enumerate(rows):
            nk = min(Sk, i + Sk - Sq + 1) if causal else Sk
            om, lm = _mp_attention(q[h, i], k[h], v[h], float(np.float64(0.3)), nk)
            np.testing.assert_allclose(o[t], om, rtol=1e-13, atol=1e-14)
            assert abs(lse[t] - lm) <= 1e-13 * max(1.0, abs(lm))


def test_attention_closed_forms():
    rng = np.random.default_rng(41)
    d = 8
    v = rng.standard_normal((1, 9, d)).astype(np.float32)
    q = rng.standard_normal((1, 9, d)).astype(np.float32)
    # causal row 0 sees only key 0: o = v_0, lse = s_00
    k = rng.standard_normal((1, 9, d)).astype(np.float32)
    o, lse = oracle.attention_rows(q, k, v, [(0, 0)], causal=True, scale=0.5)
    np.testing.assert_array_equal(o[0], v[0, 0].astype(np.float64))
    assert abs(lse[0] - 0.5 * float(np.dot(q[0, 0].astype(np.float64), k[0, 0].astype(np.float64)))) <= 1e-15
    # identical keys: uniform weights, o = mean of v, lse = s + log n
    kk = np.repeat(k[:, :1], 9, axis=1)
    o, lse = oracle.attention_rows(q, kk, v, [(0, 4)], scale=0.5)
    np.testing.assert_allclose(o[0], v[0].astype(np.float64).mean(axis=0), rtol=1e-14, atol=1e-15)
    # one dominant key: o = its value row
    k2 = np.zeros((1, 9, d), np.float32)
    k2[0, 3] = 40.0 * q[0, 2] / np.linalg.norm(q[0, 2])
    o, _ = oracle.attention_rows(q, k2, v, [(0, 2)], scale=1.0)
    np.testing.assert_allclose(o[0], v[0, 3].astype(np.float64), rtol=0, atol=1e-12)


def test_attention_online_equals_direct():
    rng = np.random.default_rng(42)
    for n, block in ((1, 1), (7, 3), (64, 16), (100, 128), (33, 1)):
        s = rng.standard_normal(n) * 5
        v = rng.standard_normal((n, 5))
        p = np.exp(s - s.max())
        direct = (p[:, None] * v).sum(axis=0) / p.sum()
        np.testing.assert_allclose(oracle.attention_online(s, v, block), direct, rtol=1e-13, atol=1e-14)
