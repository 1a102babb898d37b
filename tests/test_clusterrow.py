"""The cluster-row two-pass kernel (aligned rows above 64 KiB; clusters of several CTAs from ~260 KiB): every CTA of the
cluster folds its segment of the row, the CTA states are merged over distributed shared memory,
and every CTA normalises its segment.  Against the fp64 oracle; the variant is TWOPASS (forced or
chosen by AUTO for many long rows)."""
import numpy as np
import pytest
import torch

import oracle
import row_wise_online_gb300 as rwo
import synth
from gpu_util import run_softmax, to_device, to_host
from tolerances import check_log_values, check_rowsums, check_state, check_y

pytestmark = pytest.mark.gpu
TDT = {synth.F32: torch.float32, synth.BF16: torch.bfloat16, synth.F16: torch.float16}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from row_wise_online_gb300 import _build

    _build.build()
    torch.cuda.set_device(0)


@pytest.mark.parametrize("dtype,M,N", [
    (synth.F32, 300, 40_000),      # 160 KB rows: clusters of one CTA (AUTO too: no one-read kernel holds them)
    (synth.BF16, 500, 90_000),     # 180 KB rows
    (synth.F16, 257, 40_008),      # 80 KB rows: AUTO takes a one-read kernel, TWOPASS the cluster-row kernel
    (synth.F32, 200, 80_000),      # 320 KB rows: clusters of 2
    (synth.F32, 90, 262_148),      # ~1 MiB rows, the units do not split evenly over the cluster
    (synth.BF16, 120, 1_000_008),  # ~2 MB rows
    (synth.F16, 97, 300_000),
    (synth.F32, 3, 262_144),       # fewer rows than resident clusters
    (synth.F32, 1, 2_000_000),     # a single 8 MB row
])
@pytest.mark.parametrize("variant", [rwo.VARIANT_AUTO, rwo.VARIANT_TWOPASS])
def test_clusterrow_against_oracle(dtype, M, N, variant):
    w = synth.custom("crow", dtype, M, N, seed=N % 997 + M, dist=synth.UNIFORM, p0=-20.0, p1=20.0, late_max=20.0)
    x_host = synth.generate(w)
    x = to_device(x_host, dtype)
    y, m, d, lse = run_softmax(x, variant)
    what = f"cluster rows {M}x{N}/{rwo.VARIANT_NAMES[rwo.last_variant()]}"
    if variant == rwo.VARIANT_TWOPASS:
        assert rwo.last_variant() == rwo.VARIANT_TWOPASS
    y_ref, m_ref, d_ref, lse_ref = oracle.softmax_rows(x_host, dtype=dtype)
    yh = to_host(y)
    check_y(yh, y_ref, dtype, what)
    check_rowsums(yh, dtype, None, what)
    check_state(m.cpu().numpy(), d.cpu().numpy(), lse.cpu().numpy(), m_ref, d_ref, lse_ref, what)


@pytest.mark.parametrize("N,want", [(160_000, rwo.VARIANT_TWOPASS),      # 625 KiB fp32: two passes measured faster
                                    (230_000, rwo.VARIANT_ONEREAD_SMEM)])  # 898 KiB: held on chip
def test_auto_between_512_kib_and_1_mib(N, want):
    w = synth.custom("crow-mid", synth.F32, 300, N, seed=5, p1=3.0)
    x_host = synth.generate(w)
    y = rwo.softmax_rows(to_device(x_host))
    assert rwo.get_status() == rwo.OK and rwo.last_variant() == want
    pick = [0, 151, 299]
    y_ref, *_ = oracle.softmax_rows(x_host[pick])
    check_y(to_host(y)[pick], y_ref, synth.F32, f"auto {N}")


def test_auto_holds_many_long_rows_on_chip():
    """Many 1 MiB rows: AUTO takes a thread-block cluster per row with its segments held on chip
    (reported as ONEREAD_SMEM); forced TWOPASS keeps the cluster-row two passes."""
    w = synth.custom("crow-auto", synth.F32, 300, 1 << 18, seed=3, p1=3.0)
    x_host = synth.generate(w)
    x = to_device(x_host)
    y = rwo.softmax_rows(x)
    assert rwo.get_status() == rwo.OK
    assert rwo.last_variant() == rwo.VARIANT_ONEREAD_SMEM
    pick = [0, 151, 152, 299]
    y_ref, *_ = oracle.softmax_rows(x_host[pick])
    check_y(to_host(y)[pick], y_ref, synth.F32, "cluster rows on chip (sampled rows)")
    check_rowsums(to_host(y), synth.F32, None, "cluster rows on chip")
    rwo.softmax_rows_ex(x, variant=rwo.VARIANT_TWOPASS)
    assert rwo.get_status() == rwo.OK and rwo.last_variant() == rwo.VARIANT_TWOPASS


@pytest.mark.parametrize("dtype,M,N", [
    (synth.F32, 300, 1 << 18),     # 1 MiB rows: clusters of 8, one shared-memory buffer + tensor memory
    (synth.F32, 37, 1 << 17),      # 512 KiB rows, fewer rows than clusters for some
    (synth.BF16, 160, 1 << 18),    # 512 KiB rows
    (synth.F32, 64, 150_000),      # 600 KB rows, ragged segments
    (synth.F16, 41, 80_000),       # 160 KB rows
    (synth.F32, 90, 262_140),      # just below 1 MiB: ragged segments over clusters of 8
])
def test_cluster_rows_held_on_chip_against_oracle(dtype, M, N):
    w = synth.custom("crow-oc", dtype, M, N, seed=N % 991 + M, dist=synth.UNIFORM, p0=-20.0, p1=20.0, late_max=20.0)
    x_host = synth.generate(w)
    x = to_device(x_host, dtype)
    y, m, d, lse = run_softmax(x, rwo.VARIANT_ONEREAD_SMEM)
    assert rwo.last_variant() == rwo.VARIANT_ONEREAD_SMEM
    what = f"cluster rows on chip {M}x{N}"
    y_ref, m_ref, d_ref, lse_ref = oracle.softmax_rows(x_host, dtype=dtype)
    yh = to_host(y)
    check_y(yh, y_ref, dtype, what)
    check_rowsums(yh, dtype, None, what)
    check_state(m.cpu().numpy(), d.cpu().numpy(), lse.cpu().numpy(), m_ref, d_ref, lse_ref, what)


def test_cluster_rows_on_chip_limit():
    """Rows just above 1 MiB do not fit the segments of a cluster of 8 on chip: the forced one-read
    variant reports SOFTMAX_ERR_UNSUPPORTED (AUTO takes the two passes)."""
    x = torch.zeros((4, 262_148), device="cuda")
    with pytest.raises(rwo.SoftmaxError) as ei:
        rwo.softmax_rows_ex(x, variant=rwo.VARIANT_ONEREAD_SMEM)
    assert ei.value.status == rwo.ERR_UNSUPPORTED
    rwo.softmax_rows_ex(x)
    assert rwo.get_status() == rwo.OK


def test_cluster_rows_held_on_chip_special_rows_and_timeout():
    """Masked segments, a fully masked row, one huge value, NaN and +inf rows beside correct rows;
    then a cluster whose rank 0 never hands over its row states: its CTAs' waits run out
    (SOFTMAX_ERR_TIMEOUT), the kernel ends, and the next launch is correct."""
    M, N = 160, 1 << 18
    rows = np.random.default_rng(6).standard_normal((M, N)).astype(np.float32) * 3
    rows[0, : N - 1000] = -np.inf
    rows[1, 1000:] = -np.inf
    rows[2, :] = -np.inf
    rows[3, N // 2] = 1e30
    rows[5, 77] = np.nan
    rows[6, 99] = np.inf
    x = to_device(rows)
    y, m, d, lse = run_softmax(x, rwo.VARIANT_ONEREAD_SMEM)  # status OK
    good = [i for i in range(M) if i not in (5, 6)]
    y_ref, m_ref, d_ref, lse_ref = oracle.softmax_rows(rows[good])
    yh = to_host(y)
    check_y(yh[good], y_ref, synth.F32, "cluster rows on chip special")
    assert np.all(yh[2] == 0.0)
    assert np.isnan(d.cpu().numpy()[5]) and np.isnan(d.cpu().numpy()[6])
    old_limit = rwo.debug_set_wait_limit_ns(20_000_000)  # 20 ms
    old_fault = rwo.debug_set_fault(1)
    try:
        rwo.softmax_rows_ex(x, y, variant=rwo.VARIANT_ONEREAD_SMEM)
        assert rwo.get_status() == rwo.ERR_TIMEOUT
    finally:
        rwo.debug_set_fault(old_fault)
        rwo.debug_set_wait_limit_ns(old_limit)
    rwo.softmax_rows_ex(x, y, variant=rwo.VARIANT_ONEREAD_SMEM)
    assert rwo.get_status() == rwo.OK
    check_y(to_host(y)[good], y_ref, synth.F32, "cluster rows on chip after timeout")


def test_clusterrow_masked_segments_and_special_rows():
    """Segments of whole CTAs that see only -inf merge as the empty state; a fully masked row gives
    y = 0, m = -inf, d = 0; one huge value dominates."""
    M, N = 100, 1 << 18
    rows = np.random.default_rng(4).standard_normal((M, N)).astype(np.float32) * 3
    rows[0, : N - 1000] = -np.inf          # only the last segment has live values
    rows[1, 1000:] = -np.inf               # only the first one
    rows[2, :] = -np.inf                   # fully masked row
    rows[3, N // 2] = 1e30                 # one huge value
    rows[4, ::2] = -np.inf                 # every other element masked
    x = to_device(rows)
    y, m, d, lse = run_softmax(x, rwo.VARIANT_TWOPASS)
    y_ref, m_ref, d_ref, lse_ref = oracle.softmax_rows(rows)
    yh = to_host(y)
    check_y(yh, y_ref, synth.F32, "cluster rows special")
    check_rowsums(yh, synth.F32, ~np.isfinite(m_ref), "cluster rows special")
    assert np.all(yh[2] == 0.0)
    check_state(m.cpu().numpy(), d.cpu().numpy(), lse.cpu().numpy(), m_ref, d_ref, lse_ref, "cluster rows special")


def test_clusterrow_in_place():
    w = synth.custom("crow-ip", synth.BF16, 80, 1 << 19, seed=8, p1=2.0)
    x_host = synth.generate(w)
    x = to_device(x_host)
    rwo.softmax_rows_ex(x, x, variant=rwo.VARIANT_TWOPASS)
    assert rwo.get_status() == rwo.OK
    y_ref, *_ = oracle.softmax_rows(x_host)
    check_y(to_host(x), y_ref, synth.BF16, "cluster rows in place")


@pytest.mark.parametrize("log", [False, True])
def test_clusterrow_strided_scaled(log):
    """Column blocks of a wider matrix, a scale, softmax and log-softmax output."""
    dtype, M, N, wx, off, wy, scale = synth.BF16, 150, 200_000, 200_064, 32, 200_008, 0.3
    scale = float(np.float32(scale))
    full = synth.generate(synth.custom("crow-str", dtype, M, wx, seed=17, p1=3.0))
    block = np.ascontiguousarray(full[:, off:off + N])
    xf = to_device(full, dtype)
    yf = torch.full((M, wy), 7.0, dtype=TDT[dtype], device="cuda")
    m, d, lse = (torch.full((M,), float("nan"), device="cuda") for _ in range(3))
    rwo.softmax_rows_strided(xf[:, off:off + N], yf[:, :N], m, d, lse, scale=scale, log=log)
    assert rwo.get_status() == rwo.OK
    assert rwo.last_variant() == rwo.VARIANT_TWOPASS
    yh = to_host(yf[:, :N].contiguous())
    what = f"cluster rows strided log={log}"
    if log:
        check_log_values(yh, oracle.log_softmax_rows(block, dtype=dtype, scale=scale), dtype, what)
    else:
        y_ref, *_ = oracle.softmax_rows(block, dtype=dtype, scale=scale)
        check_y(yh, y_ref, dtype, what)
    _, m_ref, d_ref, lse_ref = oracle.softmax_rows(block, dtype=dtype, scale=scale, want_y=False)
    check_state(m.cpu().numpy(), d.cpu().numpy(), lse.cpu().numpy(), m_ref, d_ref, lse_ref, what)
    assert torch.all(yf[:, N:] == 7.0)


def test_log_softmax_long_rows():
    w = synth.custom("crow-log", synth.F32, 100, 300_000, seed=23, p1=4.0)
    x_host = synth.generate(w)
    x = to_device(x_host)
    y = rwo.log_softmax_rows(x)
    assert rwo.get_status() == rwo.OK and rwo.last_variant() == rwo.VARIANT_TWOPASS
    check_log_values(to_host(y), oracle.log_softmax_rows(x_host), synth.F32, "cluster rows log")
