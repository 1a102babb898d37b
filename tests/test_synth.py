"""The seeded input generator (CPU only): determinism, row-range consistency, recipes."""
import numpy as np
import torch

import synth


def test_deterministic_and_row_ranges_consistent():
    w = synth.WORKLOADS["fp32_64x1024"]
    a = synth.generate(w)
    b = synth.generate(w, nthreads=3)
    assert np.array_equal(a, b)
    assert np.array_equal(synth.generate(w, row0=17, nrows=9), a[17:26])
    assert np.array_equal(synth.generate_rows(w, [40, 3]), a[[40, 3]])


def test_distribution_moments():
    w = synth.WORKLOADS["fp32_4096x4096"]
    x = synth.generate(w, nrows=64).astype(np.float64)
    assert abs(x.mean()) < 0.02 and abs(x.std() - 3.0) < 0.02
    u = synth.generate(synth.custom("u", synth.F32, 8, 100000, 3, synth.UNIFORM, -20.0, 20.0))
    assert u.min() >= -20.0 and u.max() < 20.0 and abs(u.mean()) < 0.1


def test_bf16_rounding_matches_torch_rne():
    rng = np.random.default_rng(0)
    f = (rng.standard_normal(100000) * 7).astype(np.float32)
    ours = synth.f32_to_bf16(f)
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    assert np.array_equal(synth.bf16_to_f32(ours), torch.from_numpy(f).to(torch.bfloat16).float().numpy())


def test_generated_bf16_matches_rounded_fp32():
    wb = synth.custom("b", synth.BF16, 4, 333, 5, synth.NORMAL, 0.0, 2.0)
    wf = synth.custom("f", synth.F32, 4, 333, 5, synth.NORMAL, 0.0, 2.0)
    assert np.array_equal(synth.generate(wb), synth.f32_to_bf16(synth.generate(wf)))


def test_logits_stress_rows():
    w = synth.WORKLOADS["bf16_logits_16384x32768"].with_rows(201)
    x = synth.bf16_to_f32(synth.generate(w))
    for r in range(201):
        hi = np.count_nonzero(x[r] == 80.0)
        lo = np.count_nonzero(x[r] == -80.0)
        if r % 100 == 0:
            assert hi == 1 and lo == 1
        else:
            assert hi == 0 and lo == 0


def test_long_row_late_unique_max():
    w = synth.WORKLOADS["fp32_longrow_32x4194304"]
    for r in (0, 31):
        x = synth.generate(w, row0=r, nrows=1)[0]
        p = w.late_max_col(r)
        assert p >= 3 * w.N // 4
        assert x[p] == 20.0 and np.count_nonzero(x == 20.0) == 1 and x.max() == 20.0


def test_causal_mask():
    w = synth.WORKLOADS["bf16_causal_4x32x4096x4096"]
    rows = [0, 1, 127, 4095, 4096, 4096 * 37 + 200]
    x = synth.bf16_to_f32(synth.generate_rows(w, rows))
    for i, r in enumerate(rows):
        q = r % 4096
        assert np.all(np.isneginf(x[i, q + 1:]))
        assert np.all(np.isfinite(x[i, : q + 1]))


def test_generated_f16_matches_rounded_fp32():
    """fp16 workloads hold the fp32 draw rounded to nearest even (numpy's float16 conversion)."""
    w32 = synth.custom("g", synth.F32, 7, 333, seed=9, p1=5.0)
    w16 = synth.custom("g", synth.F16, 7, 333, seed=9, p1=5.0)
    a = synth.generate(w32)
    b = synth.generate(w16)
    assert b.dtype == np.uint16
    np.testing.assert_array_equal(b, a.astype(np.float16).view(np.uint16))
    np.testing.assert_array_equal(synth.f16_to_f32(b), a.astype(np.float16).astype(np.float32))
    assert w16.elem_bytes == 2
