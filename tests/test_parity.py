"""GPU parity: the CUDA path against the fp64 oracle on the seeded workloads.

Small and medium cases are compared element by element in full (several tiles, grid-stride
tails, ragged rows).  The full-size workloads run in the launch configuration the benchmark
uses (AUTO) and are compared on sampled rows element by element, plus properties checked on
every row (row sums, m = exact row max).
"""
import numpy as np
import pytest
import torch

import oracle
import row_wise_online_gb300 as rwo
import synth
from gpu_util import run_softmax, to_device, to_host
from tolerances import check_log_values, check_rowsums, check_state, check_y

pytestmark = pytest.mark.gpu

V = rwo


@pytest.fixture(scope="module", autouse=True)
def _built():
    from row_wise_online_gb300 import _build

    _build.build()
    torch.cuda.set_device(0)


def _full_check(x_host, dtype, variant, what):
    x = to_device(x_host)
    y, m, d, lse = run_softmax(x, variant)
    y_ref, m_ref, d_ref, lse_ref = oracle.softmax_rows(x_host)
    stats = check_y(to_host(y), y_ref, dtype, what)
    masked = ~np.isfinite(m_ref)
    check_rowsums(to_host(y), dtype, masked, what)
    check_state(m.cpu().numpy(), d.cpu().numpy(), lse.cpu().numpy(), m_ref, d_ref, lse_ref, what)
    return stats


@pytest.mark.parametrize("variant", [V.VARIANT_AUTO, V.VARIANT_ONEREAD_REG, V.VARIANT_ONEREAD_SMEM,
                                     V.VARIANT_TWOPASS])
def test_fp32_64x1024(variant):
    w = synth.WORKLOADS["fp32_64x1024"]
    _full_check(synth.generate(w), w.dtype, variant, f"{w.name}/{V.VARIANT_NAMES[variant]}")


@pytest.mark.parametrize("variant", [V.VARIANT_AUTO, V.VARIANT_ONEREAD_SMEM, V.VARIANT_TWOPASS])
def test_fp32_4096x4096(variant):
    w = synth.WORKLOADS["fp32_4096x4096"]
    _full_check(synth.generate(w), w.dtype, variant, f"{w.name}/{V.VARIANT_NAMES[variant]}")


# Medium shapes: many rows per CTA with a ragged grid-stride tail, rows spanning several vectors
# per thread, and a row length that is not a power of two.
MEDIUM = [
    (synth.F32, 1000, 1000), (synth.F32, 777, 4100), (synth.F32, 300, 16384), (synth.F32, 129, 20000),
    (synth.BF16, 1000, 1000), (synth.BF16, 517, 4104), (synth.BF16, 300, 32768), (synth.BF16, 65, 40000),
]


@pytest.mark.parametrize("dtype,M,N", MEDIUM)
@pytest.mark.parametrize("variant", [V.VARIANT_AUTO, V.VARIANT_ONEREAD_REG, V.VARIANT_ONEREAD_SMEM,
                                     V.VARIANT_TWOPASS])
def test_medium_shapes(dtype, M, N, variant):
    w = synth.custom("medium", dtype, M, N, seed=100 + N, p1=3.0)
    x_host = synth.generate(w)
    x = to_device(x_host)
    try:
        y, m, d, lse = run_softmax(x, variant)
    except rwo.SoftmaxError as e:
        assert variant != V.VARIANT_AUTO and e.status == rwo.ERR_UNSUPPORTED
        return
    y_ref, m_ref, d_ref, lse_ref = oracle.softmax_rows(x_host)
    what = f"{M}x{N}/{V.VARIANT_NAMES[variant]}"
    check_y(to_host(y), y_ref, dtype, what)
    check_rowsums(to_host(y), dtype, None, what)
    check_state(m.cpu().numpy(), d.cpu().numpy(), lse.cpu().numpy(), m_ref, d_ref, lse_ref, what)


def _sampled_check(w, variant, sample_rows, chunk=None):
    """Full-size run; every row checked for row sum and exact max; sampled rows against the oracle."""
    x_host = synth.generate(w)
    x = to_device(x_host)
    y, m, d, lse = run_softmax(x, variant)
    what = f"{w.name}/{V.VARIANT_NAMES[rwo.last_variant()]}"
    # every row: m is the exact row max, rows sum to 1
    assert torch.equal(m, x.amax(dim=1).float()), f"{what}: m != row max"
    sums = torch.sum(y, dim=1, dtype=torch.float64)
    tol = 1e-5 if w.dtype == synth.F32 else 4e-3
    assert float((sums - 1).abs().max()) <= tol, f"{what}: row sums"
    del sums
    # sampled rows in full against the oracle
    rows = np.unique(np.asarray(sample_rows, dtype=np.int64))
    y_ref, m_ref, d_ref, lse_ref = oracle.softmax_rows(x_host, rows=rows)
    idx = torch.from_numpy(rows).cuda()
    ys = to_host(y.index_select(0, idx))
    stats = check_y(ys, y_ref, w.dtype, what)
    check_state(m[idx].cpu().numpy(), d[idx].cpu().numpy(), lse[idx].cpu().numpy(), m_ref, d_ref, lse_ref, what)
    return stats


def test_bf16_logits_16384x32768():
    w = synth.WORKLOADS["bf16_logits_16384x32768"]
    rng = np.random.default_rng(0)
    rows = list(rng.integers(0, w.M, 40)) + [0, 100, 200, 16300, w.M - 1]  # stress rows r % 100 == 0
    _sampled_check(w, V.VARIANT_AUTO, rows)


def test_bf16_logits_twopass_sampled():
    w = synth.WORKLOADS["bf16_logits_16384x32768"].with_rows(2048)
    rng = np.random.default_rng(1)
    _sampled_check(w, V.VARIANT_TWOPASS, list(rng.integers(0, w.M, 24)) + [0, 100, 2047])


def test_bf16_causal_524288x4096():
    w = synth.WORKLOADS["bf16_causal_4x32x4096x4096"]
    rng = np.random.default_rng(2)
    qs = [0, 1, 2, 127, 128, 129, 255, 256, 1000, 4095]
    rows = list(rng.integers(0, w.M, 48)) + [h * 4096 + q for h in (0, 57, 127) for q in qs]
    _sampled_check(w, V.VARIANT_AUTO, rows)


@pytest.mark.parametrize("variant", [V.VARIANT_ONEREAD_REG, V.VARIANT_ONEREAD_SMEM, V.VARIANT_TWOPASS])
def test_bf16_causal_variants_one_head(variant):
    w = synth.WORKLOADS["bf16_causal_4x32x4096x4096"].with_rows(4096)
    x_host = synth.generate(w)
    _full_check(x_host, w.dtype, variant, f"causal-head/{V.VARIANT_NAMES[variant]}")


@pytest.mark.parametrize("variant", [V.VARIANT_AUTO, V.VARIANT_TWOPASS])
def test_fp32_longrow_32x4194304(variant):
    w = synth.WORKLOADS["fp32_longrow_32x4194304"]
    x_host = synth.generate(w)
    x = to_device(x_host)
    y, m, d, lse = run_softmax(x, variant)
    what = f"{w.name}/{V.VARIANT_NAMES[rwo.last_variant()]}"
    yh = to_host(y)
    mh, dh, lh = m.cpu().numpy(), d.cpu().numpy(), lse.cpu().numpy()
    for r0 in range(0, w.M, 4):  # four rows at a time keeps the fp64 reference at 128 MiB
        sel = np.arange(r0, r0 + 4)
        y_ref, m_ref, d_ref, lse_ref = oracle.softmax_rows(x_host, rows=sel)
        check_y(yh[sel], y_ref, w.dtype, what)
        check_rowsums(yh[sel], w.dtype, None, what)
        check_state(mh[sel], dh[sel], lh[sel], m_ref, d_ref, lse_ref, what)
    assert np.all(mh == 20.0)


def test_in_place():
    w = synth.custom("inplace", synth.BF16, 333, 4096, seed=9, p1=2.0)
    x_host = synth.generate(w)
    x = to_device(x_host)
    rwo.softmax_rows(x, x)
    y_ref, *_ = oracle.softmax_rows(x_host)
    check_y(to_host(x), y_ref, w.dtype, "in place")


def test_host_buffers_staged_pipeline():
    """Pageable host memory, and pinned rows too long for the direct path, go through staging."""
    w = synth.custom("host-pageable", synth.F32, 3000, 4096, seed=11, p1=3.0)
    x_host = synth.generate(w)
    xt = torch.from_numpy(x_host)
    yt = torch.empty_like(xt)
    rwo.softmax_rows_host(xt, yt)
    y_ref, *_ = oracle.softmax_rows(x_host)
    check_y(yt.numpy(), y_ref, w.dtype, "host pipeline, pageable")
    w = synth.custom("host-long", synth.BF16, 700, 32768, seed=12, p1=2.0)
    x_host = synth.generate(w)
    xt = torch.from_numpy(x_host.view(np.int16)).pin_memory()
    yt = torch.empty_like(xt).pin_memory()
    rwo.softmax_rows_host(xt.view(torch.bfloat16), yt.view(torch.bfloat16))
    assert rwo.last_variant() == rwo.VARIANT_ONEREAD_SMEM
    y_ref, *_ = oracle.softmax_rows(x_host)
    check_y(yt.numpy().view(np.uint16), y_ref, w.dtype, "host pipeline, long rows")


@pytest.mark.parametrize("dtype,N,want", [
    (synth.F32, 8192, V.VARIANT_ONEREAD_REG),     # 32 KiB fp32 rows: one read into registers
    (synth.BF16, 16384, V.VARIANT_ONEREAD_SMEM),  # 32 KiB 16-bit rows: one read through shared memory
    (synth.F32, 12288, V.VARIANT_ONEREAD_REG),    # 48 KiB fp32 rows: registers
    (synth.F32, 16384, V.VARIANT_ONEREAD_REG),    # 64 KiB fp32 rows: registers (12 or 16 vectors a thread)
    (synth.BF16, 24576, V.VARIANT_ONEREAD_SMEM),  # 48 KiB 16-bit rows: shared memory
    (synth.BF16, 32768, V.VARIANT_ONEREAD_SMEM),  # 64 KiB 16-bit rows: one read
    (synth.F32, 16388, V.VARIANT_ONEREAD_SMEM),   # just over 64 KiB of fp32: bulk copy, 16 warps a row
    (synth.BF16, 32776, V.VARIANT_ONEREAD_SMEM),  # just over 64 KiB of bf16: bulk copy, x kept packed
    (synth.BF16, 61448, V.VARIANT_TWOPASS),       # just over 120 KiB of bf16: past every one-read kernel
])
def test_auto_choice_around_64kib(dtype, N, want):
    w = synth.custom("auto64", dtype, 300, N, seed=N % 101, p1=3.0)
    x_host = synth.generate(w)
    y, *_ = run_softmax(to_device(x_host), V.VARIANT_AUTO, state=False)
    assert rwo.last_variant() == want
    y_ref, *_ = oracle.softmax_rows(x_host)
    check_y(to_host(y), y_ref, dtype, f"auto {N}")


@pytest.mark.parametrize("dtype,N,want", [
    (synth.F32, 1536, V.VARIANT_ONEREAD_REG),     # 6 KiB fp32 rows: registers (warp kernel slower)
    (synth.F32, 2048, V.VARIANT_ONEREAD_REG),     # 8 KiB fp32 rows: registers
    (synth.BF16, 2048, V.VARIANT_ONEREAD_REG),    # 4 KiB 16-bit rows: registers (two warps a row)
    (synth.F16, 1600, V.VARIANT_ONEREAD_REG),     # 3.1 KiB 16-bit rows: the same, ragged
    (synth.BF16, 4096, V.VARIANT_ONEREAD_SMEM),   # 8 KiB 16-bit rows, many of them: a warp per row
    (synth.BF16, 6144, V.VARIANT_ONEREAD_SMEM),   # 12 KiB 16-bit rows: CTA bulk copy, x kept packed
    (synth.F16, 8192, V.VARIANT_ONEREAD_SMEM),    # 16 KiB 16-bit rows: the same
])
def test_auto_choice_short_rows(dtype, N, want):
    w = synth.custom("auto-short", dtype, 700, N, seed=N % 103, p1=3.0)
    x_host = synth.generate(w)
    x = to_device(x_host, dtype)
    y = rwo.softmax_rows_ex(x)
    assert rwo.get_status() == rwo.OK and rwo.last_variant() == want
    odt = {synth.F32: oracle.F32, synth.BF16: oracle.BF16, synth.F16: oracle.F16}[dtype]
    y_ref, *_ = oracle.softmax_rows(x_host, dtype=odt)
    check_y(to_host(y), y_ref, dtype, f"auto short {N}")


@pytest.mark.parametrize("dtype,N", [(synth.F32, 8196), (synth.F32, 10244), (synth.F32, 12288),
                                     (synth.F32, 16380), (synth.F32, 16384), (synth.BF16, 16392),
                                     (synth.BF16, 32768)])
def test_register_kernel_rows_of_32_to_64_kib(dtype, N):
    """Rows past 32 KiB forced into registers (12 or 16 vectors a thread over 8 warps): ragged last
    vectors, full rows, fp32 and bf16 (fp16 in its own file), with per-row state."""
    w = synth.custom("reg64", dtype, 77, N, seed=N % 97, p1=4.0)
    x_host = synth.generate(w)
    _full_check(x_host, dtype, V.VARIANT_ONEREAD_REG, f"reg {N}")
    assert rwo.last_variant() == V.VARIANT_ONEREAD_REG


@pytest.mark.parametrize("N", [16388, 17404, 18432, 20480, 20484, 24576, 24580, 30720, 32764, 32768])
def test_bulk_copy_fp32_rows_of_64_to_128_kib(N):
    """fp32 rows of 64 - 128 KiB on the CTA bulk-copy kernel, forced and through AUTO: 16 consumer
    warps with 10, 12 or 16 vectors a thread (ragged rows straddle those), one row slot from 68 KiB
    (each CTA takes several rows, so the slot is refilled while the previous row is normalised)."""
    w = synth.custom("tma128", synth.F32, 400, N, seed=N % 89, p1=3.0)
    x_host = synth.generate(w)
    _full_check(x_host, synth.F32, V.VARIANT_ONEREAD_SMEM, f"bulk copy {N}")
    assert rwo.last_variant() == V.VARIANT_ONEREAD_SMEM
    if N in (20484, 32768):
        _full_check(x_host, synth.F32, V.VARIANT_AUTO, f"auto {N}")
        assert rwo.last_variant() == V.VARIANT_ONEREAD_SMEM


@pytest.mark.parametrize("dtype,N", [(synth.BF16, 4104), (synth.BF16, 5120), (synth.F16, 6152), (synth.BF16, 7176),
                                     (synth.BF16, 8192),
                                     (synth.BF16, 16384), (synth.BF16, 18440), (synth.F16, 22536),
                                     (synth.BF16, 27648),
                                     (synth.BF16, 32776), (synth.BF16, 40000), (synth.BF16, 45064),
                                     (synth.BF16, 53760), (synth.F16, 36872), (synth.BF16, 61440),
                                     (synth.F16, 57352)])
def test_bulk_copy_16bit_rows_kept_packed(dtype, N):
    """16-bit rows of 8 - 16 KiB (4 consumer warps, 8 vectors a thread, 2 - 4 CTAs per SM), of 32 -
    54 KiB (8 consumer warps, 8 - 14 vectors a thread) and of 64 - 120 KiB (15
    consumer warps, 10 - 16 vectors; one row slot above 80 KiB) on the CTA bulk-copy kernel with x
    kept packed in registers, ragged rows among them: softmax with the
    state, forced and through AUTO, and log softmax, against the fp64 oracle."""
    w = synth.custom("tma16", dtype, 400, N, seed=N % 79, p1=4.0)
    x_host = synth.generate(w)
    odt = oracle.F16 if dtype == synth.F16 else oracle.BF16
    x = to_device(x_host, dtype)
    for variant in (V.VARIANT_ONEREAD_SMEM, V.VARIANT_AUTO):
        m, d, lse = (torch.full((w.M,), float("nan"), device="cuda") for _ in range(3))
        y = rwo.softmax_rows_ex(x, m_out=m, d_out=d, lse_out=lse, variant=variant)
        assert rwo.get_status() == rwo.OK and rwo.last_variant() == V.VARIANT_ONEREAD_SMEM
        y_ref, m_ref, d_ref, lse_ref = oracle.softmax_rows(x_host, dtype=odt)
        what = f"packed {N}/{V.VARIANT_NAMES[variant]}"
        check_y(to_host(y), y_ref, dtype, what)
        check_rowsums(to_host(y), dtype, ~np.isfinite(m_ref), what)
        check_state(m.cpu().numpy(), d.cpu().numpy(), lse.cpu().numpy(), m_ref, d_ref, lse_ref, what)
        del y_ref
    ly = rwo.log_softmax_rows(x, variant=V.VARIANT_ONEREAD_SMEM)
    assert rwo.get_status() == rwo.OK
    check_log_values(to_host(ly), oracle.log_softmax_rows(x_host, dtype=odt), dtype, f"packed log {N}")


@pytest.mark.parametrize("dtype,N", [(synth.F32, 20480), (synth.F32, 32768), (synth.BF16, 40000),
                                     (synth.BF16, 61440), (synth.F16, 45064)])
def test_bulk_copy_long_rows_special_values(dtype, N):
    """The bulk-copy configurations for rows above 64 KiB (fp32 in 16 warps, one slot; 16-bit kept
    packed) on special rows: all -inf (y = 0 / -inf), the first half -inf, one huge value, a huge
    negative row, a uniform row; softmax with the state and log softmax against the oracle."""
    M = 160
    rng = np.random.default_rng(N)
    rows = (rng.standard_normal((M, N)) * 3).astype(np.float32)
    big = {synth.F32: 1e30, synth.BF16: 3e38, synth.F16: 65504.0}[dtype]
    rows[0, :] = -np.inf
    rows[1, :N // 2] = -np.inf
    rows[2, N - 7] = big
    rows[3] -= 1e30 if dtype != synth.F16 else 60000.0
    rows[4, :] = 0.5
    x_host = rows if dtype == synth.F32 else synth.f32_to_bf16(rows) if dtype == synth.BF16 else synth.f32_to_f16(rows)
    odt = {synth.F32: oracle.F32, synth.BF16: oracle.BF16, synth.F16: oracle.F16}[dtype]
    x = to_device(x_host, dtype)
    m, d, lse = (torch.full((M,), float("nan"), device="cuda") for _ in range(3))
    y = rwo.softmax_rows_ex(x, m_out=m, d_out=d, lse_out=lse, variant=V.VARIANT_ONEREAD_SMEM)
    assert rwo.get_status() == rwo.OK and rwo.last_variant() == V.VARIANT_ONEREAD_SMEM
    y_ref, m_ref, d_ref, lse_ref = oracle.softmax_rows(x_host, dtype=odt)
    what = f"bulk copy special {N}"
    check_y(to_host(y), y_ref, dtype, what)
    check_rowsums(to_host(y), dtype, ~np.isfinite(m_ref), what)
    check_state(m.cpu().numpy(), d.cpu().numpy(), lse.cpu().numpy(), m_ref, d_ref, lse_ref, what)
    ly = rwo.log_softmax_rows(x, variant=V.VARIANT_ONEREAD_SMEM)
    assert rwo.get_status() == rwo.OK
    check_log_values(to_host(ly), oracle.log_softmax_rows(x_host, dtype=odt), dtype, what + " log")


def test_host_buffers_staged_very_long_rows():
    """Rows of 1 MiB through the staging lanes, whose kernels overlap: AUTO must not take the
    split-row kernel (it needs the whole GPU resident) and the result still matches."""
    w = synth.custom("host-vlong", synth.F32, 20, 1 << 18, seed=13, p1=3.0)
    x_host = synth.generate(w)
    xt = torch.from_numpy(x_host)
    yt = torch.empty_like(xt)
    rwo.softmax_rows_host(xt, yt)
    assert rwo.get_status() == rwo.OK
    assert rwo.last_variant() not in (rwo.VARIANT_SPLITROW, rwo.VARIANT_SPLITROW_STREAM)
    y_ref, *_ = oracle.softmax_rows(x_host)
    check_y(yt.numpy(), y_ref, w.dtype, "host pipeline, 1 MiB rows")


def test_host_buffers_pipeline():
    w = synth.custom("host", synth.F32, 5000, 4096, seed=10, p1=3.0)
    x_host = synth.generate(w)
    xt = torch.from_numpy(x_host).pin_memory()
    yt = torch.empty_like(xt).pin_memory()
    rwo.softmax_rows_host(xt, yt)
    assert rwo.last_variant() == rwo.VARIANT_ONEREAD_REG  # pinned: read and written in place
    y_ref, *_ = oracle.softmax_rows(x_host)
    check_y(yt.numpy(), y_ref, w.dtype, "host pipeline")


def test_variant_choice():
    cases = [  # (workload, rows, variant AUTO must pick)
        ("fp32_64x1024", 64, V.VARIANT_ONEREAD_REG),
        ("fp32_4096x4096", 8, V.VARIANT_ONEREAD_REG),
        ("bf16_logits_16384x32768", 8, V.VARIANT_ONEREAD_SMEM),
        ("bf16_causal_4x32x4096x4096", 8, V.VARIANT_ONEREAD_REG),      # few rows: launch-bound
        ("bf16_causal_4x32x4096x4096", 4096, V.VARIANT_ONEREAD_SMEM),  # many rows: warp per row
    ]
    for name, rows, want in cases:
        w = synth.WORKLOADS[name].with_rows(rows)
        x = to_device(synth.generate(w))
        rwo.softmax_rows(x)
        torch.cuda.synchronize()
        assert rwo.last_variant() == want, (name, rwo.last_variant())
