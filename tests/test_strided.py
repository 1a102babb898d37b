"""softmax_rows_strided: row pitches (column blocks of wider matrices), a scale folded into the
exponent, and softmax / log-softmax output, against the fp64 oracle of softmax(scale * x)."""
import numpy as np
import pytest
import torch

import oracle
import row_wise_online_gb300 as rwo
import synth
from gpu_util import to_device, to_host
from tolerances import check_log_values, check_rowsums, check_state, check_y

pytestmark = pytest.mark.gpu
V = rwo
TDT = {synth.F32: torch.float32, synth.BF16: torch.bfloat16, synth.F16: torch.float16}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from row_wise_online_gb300 import _build

    _build.build()
    torch.cuda.set_device(0)


CASES = [
    # dtype, M, N, full width of x, column offset, full width of y, scale
    (synth.F32, 300, 1000, 1024, 8, 1000, 1.0 / np.sqrt(128.0)),      # aligned pitch and offset
    (synth.F32, 200, 1000, 1003, 3, 1001, 0.125),                      # unaligned: scalar paths
    (synth.BF16, 257, 4096, 8192, 4096, 4104, 3.0),                    # right half of a wider matrix
    (synth.BF16, 64, 32768, 33000, 104, 32768, 0.5),                   # long rows: bulk-copy kernel
    (synth.F16, 500, 2048, 2056, 8, 2048, 1.0 / np.sqrt(64.0)),
    (synth.F32, 40, 20000, 20004, 4, 20000, 2.0),                      # beyond the register kernel
    # 16-bit rows on the bulk-copy kernel with x kept packed (12, 40 and 78 KiB rows)
    (synth.BF16, 120, 6144, 6200, 8, 6144, 0.7),
    (synth.F16, 100, 20000, 20008, 8, 20000, 1.7),
    (synth.BF16, 80, 40000, 40016, 16, 40008, 0.3),
]


@pytest.mark.parametrize("dtype,M,N,wx,off,wy,scale", CASES)
@pytest.mark.parametrize("log", [False, True])
@pytest.mark.parametrize("variant", [V.VARIANT_AUTO, V.VARIANT_ONEREAD_REG, V.VARIANT_ONEREAD_SMEM, V.VARIANT_TWOPASS])
def test_strided_scaled_against_oracle(dtype, M, N, wx, off, wy, scale, log, variant):
    scale = float(np.float32(scale))
    w = synth.custom("strided", dtype, M, wx, seed=600 + N, p1=3.0)
    full = synth.generate(w)
    block = np.ascontiguousarray(full[:, off:off + N])
    xf = to_device(full, dtype)
    x = xf[:, off:off + N]
    yf = torch.full((M, wy), 7.0, dtype=TDT[dtype], device="cuda")
    y = yf[:, :N]
    m, d, lse = (torch.full((M,), float("nan"), device="cuda") for _ in range(3))
    try:
        rwo.softmax_rows_strided(x, y, m, d, lse, scale=scale, log=log, variant=variant)
    except rwo.SoftmaxError as e:
        assert variant != V.VARIANT_AUTO and e.status in (rwo.ERR_UNSUPPORTED, rwo.ERR_MISALIGNED)
        return
    assert rwo.get_status() == rwo.OK
    what = f"strided {M}x{N} ld {wx}/{wy} off {off} scale {scale} log {log}/{V.VARIANT_NAMES[rwo.last_variant()]}"
    yh = to_host(y.contiguous())
    if log:
        check_log_values(yh, oracle.log_softmax_rows(block, dtype=dtype, scale=scale), dtype, what)
    else:
        y_ref, *_ = oracle.softmax_rows(block, dtype=dtype, scale=scale)
        check_y(yh, y_ref, dtype, what)
        check_rowsums(yh, dtype, None, what)
    _, m_ref, d_ref, lse_ref = oracle.softmax_rows(block, dtype=dtype, scale=scale, want_y=False)
    check_state(m.cpu().numpy(), d.cpu().numpy(), lse.cpu().numpy(), m_ref, d_ref, lse_ref, what)
    # the padding columns of y are untouched
    if wy > N:
        assert torch.all(yf[:, N:] == 7.0)
    # the input is untouched
    assert torch.equal(xf, to_device(full, dtype))


@pytest.mark.parametrize("variant,N", [(V.VARIANT_ONEREAD_REG, 4096), (V.VARIANT_ONEREAD_SMEM, 32768),
                                       (V.VARIANT_TWOPASS, 4096)])
def test_scale_one_contiguous_equals_softmax_rows_ex(variant, N):
    """With scale 1 and contiguous rows the call runs the same kernel as softmax_rows_ex (rows over
    16 KiB for ONEREAD_SMEM, where softmax_rows_ex also takes the CTA bulk-copy kernel): bitwise equal."""
    w = synth.custom("s1", synth.BF16, 333, N, seed=61, p1=3.0)
    x = to_device(synth.generate(w))
    a = rwo.softmax_rows_strided(x, variant=variant)
    b = rwo.softmax_rows_ex(x, variant=variant)
    assert rwo.get_status() == rwo.OK
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    la = rwo.softmax_rows_strided(x, log=True, variant=variant)
    lb = rwo.log_softmax_rows(x, variant=variant)
    assert torch.equal(la.view(torch.int16), lb.view(torch.int16))


def test_strided_in_place_and_errors():
    w = synth.custom("ip", synth.F32, 100, 1024, seed=62, p1=3.0)
    full = synth.generate(w)
    xf = to_device(full)
    x = xf[:, :1000]
    rwo.softmax_rows_strided(x, x, scale=0.25)  # in place, same pitch
    assert rwo.get_status() == rwo.OK
    y_ref, *_ = oracle.softmax_rows(np.ascontiguousarray(full[:, :1000]), scale=0.25)
    check_y(to_host(x.contiguous()), y_ref, synth.F32, "in place strided")
    assert torch.equal(xf[:, 1000:], to_device(full)[:, 1000:])
    for bad in (0.0, -1.0, float("inf"), float("nan")):
        with pytest.raises(rwo.SoftmaxError) as ei:
            rwo.softmax_rows_strided(xf, scale=bad)
        assert ei.value.status == rwo.ERR_INVALID_ARG
    with pytest.raises(rwo.SoftmaxError) as ei:
        rwo.softmax_rows_strided(xf, variant=V.VARIANT_SPLITROW)
    assert ei.value.status == rwo.ERR_UNSUPPORTED
