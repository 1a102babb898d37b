"""GPU edge cases ("Softmax 数值稳定性与 IO-Aware Attention" §9.2: huge positive and negative
inputs, all-equal rows, one-element rows, unaligned lengths and tails, mask boundaries),
unaligned base pointers, and guard regions around every output to catch stray writes."""
import numpy as np
import pytest
import torch

import oracle
import row_wise_online_gb300 as rwo
import synth
from gpu_util import run_softmax, to_device, to_host
from tolerances import check_rowsums, check_state, check_y

pytestmark = pytest.mark.gpu

V = rwo
ALL_VARIANTS = [V.VARIANT_AUTO, V.VARIANT_ONEREAD_REG, V.VARIANT_ONEREAD_SMEM, V.VARIANT_TWOPASS]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from row_wise_online_gb300 import _build

    _build.build()
    torch.cuda.set_device(0)


def _check_case(x_host, dtype, variant, what):
    x = to_device(x_host)
    try:
        y, m, d, lse = run_softmax(x, variant)
    except rwo.SoftmaxError as e:
        assert variant != V.VARIANT_AUTO and e.status in (rwo.ERR_UNSUPPORTED, rwo.ERR_MISALIGNED), (what, e)
        return None
    y_ref, m_ref, d_ref, lse_ref = oracle.softmax_rows(x_host)
    yh = to_host(y)
    check_y(yh, y_ref, dtype, what)
    check_rowsums(yh, dtype, ~np.isfinite(m_ref), what)
    check_state(m.cpu().numpy(), d.cpu().numpy(), lse.cpu().numpy(), m_ref, d_ref, lse_ref, what)
    return yh


@pytest.mark.parametrize("dtype", [synth.F32, synth.BF16])
@pytest.mark.parametrize("N", [1, 2, 3, 7, 8, 31, 33, 127, 129, 1023, 4097, 8191])
@pytest.mark.parametrize("variant", ALL_VARIANTS)
def test_row_lengths(dtype, N, variant):
    w = synth.custom("len", dtype, 37, N, seed=N, p1=2.5)
    _check_case(synth.generate(w), dtype, variant, f"N={N}/{V.VARIANT_NAMES[variant]}")


@pytest.mark.parametrize("dtype", [synth.F32, synth.BF16])
@pytest.mark.parametrize("N", [64, 1000, 4096, 40000])
def test_unaligned_base_pointer(dtype, N):
    """x and y start 4 (fp32) or 2 (bf16) bytes past a 16-byte boundary: AUTO takes the scalar path."""
    M = 19
    w = synth.custom("mis", dtype, M, N, seed=3, p1=3.0)
    x_host = synth.generate(w)
    tdt = torch.float32 if dtype == synth.F32 else torch.bfloat16
    xbuf = torch.empty(M * N + 8, dtype=tdt, device="cuda")
    ybuf = torch.zeros(M * N + 8, dtype=tdt, device="cuda")
    x = xbuf[1:1 + M * N].view(M, N)
    y = ybuf[1:1 + M * N].view(M, N)
    x.copy_(to_device(x_host))
    assert x.data_ptr() % 16 != 0
    rwo.softmax_rows(x, y)
    y_ref, *_ = oracle.softmax_rows(x_host)
    check_y(to_host(y), y_ref, dtype, f"unaligned N={N}")
    assert torch.all(ybuf[0] == 0) and torch.all(ybuf[1 + M * N:] == 0)
    for variant in (V.VARIANT_ONEREAD_SMEM,):
        with pytest.raises(rwo.SoftmaxError) as ei:
            rwo.softmax_rows_ex(x, y, variant=variant)
        assert ei.value.status == rwo.ERR_MISALIGNED


def _special_rows(dtype, N):
    rng = np.random.default_rng(N)
    rows = []
    rows.append(np.full(N, 0.75))                       # all equal
    r = rng.standard_normal(N); r[N // 3] = 1e30; rows.append(r)          # one huge value
    r = rng.standard_normal(N); r[-1] = 3.0e38 / 2; rows.append(r)       # fp32 max / 2
    rows.append(np.full(N, -1e30))                      # huge negative, all equal
    rows.append(-1e4 + rng.uniform(-3, 3, N))           # huge negative offset
    r = np.full(N, -np.inf); r[N // 2] = -2.0; rows.append(r)            # all -inf but one
    rows.append(np.full(N, -np.inf))                    # fully masked row
    for lo, hi in ((0, 128), (N // 2 - 64, N // 2 + 64), (N - 128, N)):  # masked 128-wide chunks
        r = rng.standard_normal(N) * 3
        r[max(lo, 0):min(hi, N)] = -np.inf
        rows.append(r)
    r = rng.standard_normal(N) * 3; r[1::2] = -np.inf; rows.append(r)     # alternating mask
    r = rng.standard_normal(N); r[N // 4] = 80.0; r[3 * N // 4] = -80.0; rows.append(r)
    x = np.stack(rows).astype(np.float32)
    return x if dtype == synth.F32 else synth.f32_to_bf16(x)


@pytest.mark.parametrize("dtype", [synth.F32, synth.BF16])
@pytest.mark.parametrize("N", [256, 1024, 4096, 32768, 65536])
@pytest.mark.parametrize("variant", ALL_VARIANTS)
def test_special_values(dtype, N, variant):
    x_host = _special_rows(dtype, N)
    yh = _check_case(x_host, dtype, variant, f"special N={N}/{V.VARIANT_NAMES[variant]}")
    if yh is not None:
        assert not np.isnan(yh.astype(np.float64) if dtype == synth.F32 else synth.bf16_to_f32(yh)).any()


def test_canary_regions_untouched():
    """Outputs written exactly in bounds: y, m, d, lse sit inside larger buffers filled with a sentinel."""
    for dtype, N in ((synth.F32, 4096), (synth.BF16, 32768), (synth.F32, 1000), (synth.BF16, 4104)):
        M = 53
        w = synth.custom("can", dtype, M, N, seed=4, p1=2.0)
        x = to_device(synth.generate(w))
        tdt = x.dtype
        pad = 4096
        ybuf = torch.full((M * N + 2 * pad,), 7.0, dtype=tdt, device="cuda")
        y = ybuf[pad:pad + M * N].view(M, N)
        sbufs = [torch.full((M + 2 * pad,), 7.0, dtype=torch.float32, device="cuda") for _ in range(3)]
        m, d, lse = (b[pad:pad + M] for b in sbufs)
        for variant in ALL_VARIANTS:
            try:
                rwo.softmax_rows_ex(x, y, m, d, lse, variant=variant)
            except rwo.SoftmaxError as e:
                assert e.status == rwo.ERR_UNSUPPORTED
                continue
            assert rwo.get_status() == rwo.OK
            assert torch.all(ybuf[:pad] == 7.0) and torch.all(ybuf[pad + M * N:] == 7.0), (dtype, N, variant)
            for b in sbufs:
                assert torch.all(b[:pad] == 7.0) and torch.all(b[pad + M:] == 7.0)


def test_zero_rows_is_noop():
    x = torch.empty((0, 128), device="cuda")
    y = rwo.softmax_rows(x)
    assert y.shape == (0, 128)


def test_rows_exceeding_32bit_element_index():
    """M * N >= 2^31 elements: every offset is 64-bit (the last rows are checked)."""
    M, N = 524288 + 8, 4096
    w = synth.custom("big", synth.BF16, M, N, seed=12, p1=1.0)
    x_host = synth.generate(w, row0=M - 16, nrows=16)
    x = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    x[M - 16:] = to_device(x_host)
    y = rwo.softmax_rows(x)
    y_ref, *_ = oracle.softmax_rows(x_host)
    check_y(to_host(y[M - 16:]), y_ref, synth.BF16, "64-bit offsets")
    assert torch.allclose(y[0].float(), torch.full((N,), 1.0 / N, device="cuda"))
