"""Split-row path: rows spread over every CTA, cluster (DSMEM) merge, bounded cross-cluster exchange.

The failure test makes the exchange wait run out on purpose from the host side (a test hook
keeps one cluster from publishing its state): the kernel must record SOFTMAX_ERR_TIMEOUT in the
status word and terminate, and the next launch must work normally.  Nothing faults or hangs.
"""
import numpy as np
import pytest
import torch

import oracle
import row_wise_online_gb300 as rwo
import synth
from gpu_util import run_softmax, to_device, to_host
from tolerances import check_rowsums, check_state, check_y

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from row_wise_online_gb300 import _build

    _build.build()
    torch.cuda.set_device(0)


SPLIT_VARIANTS = [rwo.VARIANT_SPLITROW, rwo.VARIANT_SPLITROW_STREAM]


@pytest.mark.parametrize("variant", SPLIT_VARIANTS)
@pytest.mark.parametrize("dtype,M,N", [
    (synth.F32, 3, 1 << 21), (synth.F32, 5, 1_500_000), (synth.BF16, 2, 1 << 22), (synth.BF16, 7, 3_000_008),
    (synth.F32, 1, 4_000_000), (synth.F32, 9, 4_194_304), (synth.BF16, 17, 777_784), (synth.F32, 2, 160_000),
])
def test_splitrow_against_oracle(dtype, M, N, variant):
    """Both split-row kernels, element by element: the segment held on chip (SPLITROW; rows of
    ~1.5 - 16 MiB give 2 - 8 row buffers, ragged segments and a partial last piece) and the
    streaming form."""
    w = synth.custom("split", dtype, M, N, seed=N % 1000, dist=synth.UNIFORM, p0=-20.0, p1=20.0, late_max=20.0)
    x_host = synth.generate(w)
    x = to_device(x_host)
    y, m, d, lse = run_softmax(x, variant)
    assert rwo.last_variant() == variant
    y_ref, m_ref, d_ref, lse_ref = oracle.softmax_rows(x_host)
    yh = to_host(y)
    check_y(yh, y_ref, dtype, f"split {M}x{N}")
    check_rowsums(yh, dtype, None, "split")
    check_state(m.cpu().numpy(), d.cpu().numpy(), lse.cpu().numpy(), m_ref, d_ref, lse_ref, "split")


@pytest.mark.parametrize("N", [1 << 21, 1 << 22])
@pytest.mark.parametrize("variant", SPLIT_VARIANTS)
def test_splitrow_masked_segments_and_special_rows(variant, N):
    """Whole CTA segments and clusters that see only -inf must merge as the empty state (8 MiB rows
    keep four row buffers in shared memory; 16 MiB rows park folded segments in tensor memory)."""
    rows = np.random.default_rng(0).standard_normal((4, N)).astype(np.float32) * 3
    rows[0, : N - 1000] = -np.inf          # only the tail survives: most CTAs hold empty states
    rows[1, 1000:] = -np.inf               # only the head survives
    rows[2, :] = -np.inf                   # fully masked row
    rows[3, N // 2] = 1e30                 # one huge value
    x = to_device(rows)
    y, m, d, lse = run_softmax(x, variant)
    y_ref, m_ref, d_ref, lse_ref = oracle.softmax_rows(rows)
    yh = to_host(y)
    check_y(yh, y_ref, synth.F32, "split special")
    check_rowsums(yh, synth.F32, ~np.isfinite(m_ref), "split special")
    check_state(m.cpu().numpy(), d.cpu().numpy(), lse.cpu().numpy(), m_ref, d_ref, lse_ref, "split special")
    assert not np.isnan(yh).any()


@pytest.mark.parametrize("variant", SPLIT_VARIANTS)
def test_splitrow_in_place(variant):
    w = synth.custom("split-ip", synth.BF16, 3, 1 << 22, seed=5, p1=2.0)
    x_host = synth.generate(w)
    x = to_device(x_host)
    rwo.softmax_rows_ex(x, x, variant=variant)
    assert rwo.get_status() == rwo.OK
    y_ref, *_ = oracle.softmax_rows(x_host)
    check_y(to_host(x), y_ref, synth.BF16, "split in place")


def test_auto_takes_splitrow_for_few_long_rows():
    w = synth.WORKLOADS["fp32_longrow_32x4194304"].with_rows(4)
    x = to_device(synth.generate(w))
    rwo.softmax_rows(x)
    torch.cuda.synchronize()
    assert rwo.last_variant() == rwo.VARIANT_SPLITROW  # 16 MiB rows: segments held on chip


@pytest.mark.parametrize("M,N", [(76, 1 << 18), (8, 1 << 19), (64, 1 << 20)])
def test_auto_avoids_the_split_row_where_rows_are_many_and_shorter(M, N):
    """Rows of 1 - 4 MiB at these counts run faster with a cluster per row (segments held on chip
    where they fit, else the two passes) than split over the GPU (each row's exchange would cost
    more than the clusters' parallel rows)."""
    x_host = np.random.default_rng(M).standard_normal((M, N)).astype(np.float32)
    x = to_device(x_host)
    y = rwo.softmax_rows(x)
    assert rwo.get_status() == rwo.OK
    assert rwo.last_variant() in (rwo.VARIANT_ONEREAD_SMEM, rwo.VARIANT_TWOPASS)
    y_ref, *_ = oracle.softmax_rows(x_host[[0, M - 1]])
    check_y(to_host(y)[[0, M - 1]], y_ref, synth.F32, f"auto {M}x{N}")


def test_auto_takes_splitrow_for_many_rows_of_8mib():
    """Rows of 8 MiB and more go to the split kernel at any row count (here 100 rows, more than
    half the SMs); 4 MiB rows at the same count stay with the two-pass kernel.  Sampled rows
    against the oracle, every row's sum."""
    M, N = 100, 1 << 21
    w = synth.custom("split-many", synth.F32, M, N, seed=41, p1=3.0)
    x_host = synth.generate(w)
    x = to_device(x_host)
    y, m, d, lse = run_softmax(x, rwo.VARIANT_AUTO)
    assert rwo.last_variant() in (rwo.VARIANT_SPLITROW, rwo.VARIANT_SPLITROW_STREAM)
    yh = to_host(y)
    check_rowsums(yh, synth.F32, None, "split 100 x 8 MiB")
    pick = [0, 37, 76, 77, 99]
    y_ref, m_ref, d_ref, lse_ref = oracle.softmax_rows(x_host[pick])
    check_y(yh[pick], y_ref, synth.F32, "split 100 x 8 MiB (sampled rows)")
    check_state(m.cpu().numpy()[pick], d.cpu().numpy()[pick], lse.cpu().numpy()[pick], m_ref, d_ref, lse_ref,
                "split 100 x 8 MiB (sampled rows)")
    del x, y
    x = to_device(x_host[:, : N // 2].copy())
    rwo.softmax_rows(x)
    torch.cuda.synchronize()
    assert rwo.last_variant() == rwo.VARIANT_TWOPASS


@pytest.mark.parametrize("M,N", [(3, 1 << 21), (5, 1 << 22)])
@pytest.mark.parametrize("variant", SPLIT_VARIANTS)
def test_exchange_wait_runs_out_and_reports_timeout(variant, M, N):
    w = synth.custom("fault", synth.F32, M, N, seed=1, p1=2.0)
    x_host = synth.generate(w)
    x = to_device(x_host)
    y = torch.empty_like(x)
    assert rwo.get_status() == rwo.OK
    old_limit = rwo.debug_set_wait_limit_ns(20_000_000)  # 20 ms
    old_fault = rwo.debug_set_fault(1)
    try:
        rwo.softmax_rows_ex(x, y, variant=variant)
        assert rwo.last_variant() == variant
        assert rwo.get_status() == rwo.ERR_TIMEOUT
    finally:
        rwo.debug_set_fault(old_fault)
        rwo.debug_set_wait_limit_ns(old_limit)
    # the context is intact and the next launch is correct
    assert rwo.get_status() == rwo.OK
    rwo.softmax_rows_ex(x, y, variant=variant)
    assert rwo.get_status() == rwo.OK
    y_ref, *_ = oracle.softmax_rows(x_host)
    check_y(to_host(y), y_ref, synth.F32, "after timeout")


def test_rows_larger_than_l2():
    """A single 32 Mi-element fp32 row (128 MiB, larger than L2): too long to hold on chip, so the
    streaming split kernel takes it (its second pass then reads HBM again); AUTO picks it too."""
    N = 1 << 25
    w = synth.custom("split-huge", synth.F32, 1, N, seed=77, dist=synth.UNIFORM, p0=-20.0, p1=20.0, late_max=20.0)
    x_host = synth.generate(w)
    x = to_device(x_host)
    y, m, d, lse = run_softmax(x, rwo.VARIANT_SPLITROW)
    assert rwo.last_variant() == rwo.VARIANT_SPLITROW_STREAM  # too long to hold on chip
    y_ref, m_ref, d_ref, lse_ref = oracle.softmax_rows(x_host)
    yh = to_host(y)
    check_y(yh, y_ref, synth.F32, "split 1 x 32Mi")
    check_rowsums(yh, synth.F32, None, "split 1 x 32Mi")
    check_state(m.cpu().numpy(), d.cpu().numpy(), lse.cpu().numpy(), m_ref, d_ref, lse_ref, "split 1 x 32Mi")
    del y_ref
    rwo.softmax_rows(x)
    torch.cuda.synchronize()
    assert rwo.last_variant() == rwo.VARIANT_SPLITROW_STREAM


@pytest.mark.parametrize("N", [1 << 21, 1 << 22])
@pytest.mark.parametrize("variant", SPLIT_VARIANTS)
def test_splitrow_nan_and_inf_rows_stay_in_their_row(variant, N):
    """A row holding a NaN or +inf has a NaN state (e^(inf - inf)); it must be published and merged
    like any other state, so only that row's outputs are NaN, the other rows are correct and the
    exchange does not wait out its limit (no SOFTMAX_ERR_TIMEOUT)."""
    rows = np.random.default_rng(3).standard_normal((4, N)).astype(np.float32) * 3
    rows[1, N // 3] = np.nan
    rows[2, 2 * N // 3] = np.inf
    x = to_device(rows)
    assert rwo.get_status() == rwo.OK
    y, m, d, lse = run_softmax(x, variant)  # asserts status OK
    yh = to_host(y)
    good = [0, 3]
    y_ref, m_ref, d_ref, lse_ref = oracle.softmax_rows(rows[good])
    check_y(yh[good], y_ref, synth.F32, "split rows beside NaN / inf rows")
    check_state(m.cpu().numpy()[good], d.cpu().numpy()[good], lse.cpu().numpy()[good], m_ref, d_ref, lse_ref,
                "split rows beside NaN / inf rows")
    dh = d.cpu().numpy()
    assert np.isnan(dh[1]) and np.isnan(dh[2])
    assert np.isnan(yh[1]).any() and np.isnan(yh[2]).any()


def test_splitrow_replayed_from_a_cuda_graph():
    """Captured in a CUDA graph, each on-chip split-row call becomes a pool allocation, a memset and
    a free around the kernel: launches replayed back to back, with rows of another length in
    between, all match the oracle on every replay."""
    ws = [synth.custom("split-graph", synth.F32, 6, 1 << 22, seed=60 + i, dist=synth.UNIFORM, p0=-20.0, p1=20.0,
                       late_max=20.0) for i in range(2)]
    hosts = [synth.generate(w) for w in ws]
    xs = [to_device(h) for h in hosts]
    ys = [torch.empty_like(x) for x in xs]
    short = to_device(synth.generate(synth.custom("split-graph-short", synth.F32, 3, 1 << 21, seed=62)))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):  # one eager call first (the kernel's attributes are set outside the capture)
        rwo.softmax_rows_ex(xs[0], ys[0], variant=rwo.VARIANT_SPLITROW, stream=s)
        assert rwo.last_variant() == rwo.VARIANT_SPLITROW
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for i in (0, 1, 0):
            rwo.softmax_rows_ex(xs[i], ys[i], variant=rwo.VARIANT_SPLITROW, stream=s)
            rwo.softmax_rows_ex(short, variant=rwo.VARIANT_SPLITROW, stream=s)
    for _ in range(3):
        for y in ys:
            y.fill_(float("nan"))
        g.replay()
        assert rwo.get_status(s) == rwo.OK
        for h, y in zip(hosts, ys):
            y_ref, *_ = oracle.softmax_rows(h)
            check_y(to_host(y), y_ref, synth.F32, "split row replayed from a graph")
