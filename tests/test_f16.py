"""fp16 (IEEE binary16) input and output through every kernel, against the fp64 oracle.

The oracle widens fp16 exactly; outputs are compared within one fp16 ulp of the reference
(subnormal spacing below 2^-14), row sums within 1e-3, m bit-exact.
"""
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
F16 = synth.F16


@pytest.fixture(scope="module", autouse=True)
def _built():
    from row_wise_online_gb300 import _build

    _build.build()
    torch.cuda.set_device(0)


def _run(x, variant):
    M = x.numel() // x.shape[-1]
    m, d, lse = (torch.full((M,), float("nan"), device="cuda") for _ in range(3))
    y = rwo.softmax_rows_ex(x, m_out=m, d_out=d, lse_out=lse, variant=variant)
    assert rwo.get_status() == rwo.OK
    return y, m, d, lse


@pytest.mark.parametrize("M,N", [(64, 1024), (1000, 1000), (700, 4104), (300, 32768), (33, 40000), (5000, 2048),
                                 (77, 24584)])
@pytest.mark.parametrize("variant", [V.VARIANT_AUTO, V.VARIANT_ONEREAD_REG, V.VARIANT_ONEREAD_SMEM, V.VARIANT_TWOPASS])
def test_f16_softmax_against_oracle(M, N, variant):
    w = synth.custom("f16", F16, M, N, seed=500 + N, p1=3.0)
    x_host = synth.generate(w)
    x = to_device(x_host, F16)
    try:
        y, m, d, lse = _run(x, variant)
    except rwo.SoftmaxError as e:
        assert variant != V.VARIANT_AUTO and e.status == rwo.ERR_UNSUPPORTED
        return
    assert y.dtype == torch.float16
    what = f"f16 {M}x{N}/{V.VARIANT_NAMES[rwo.last_variant()]}"
    y_ref, m_ref, d_ref, lse_ref = oracle.softmax_rows(x_host, dtype=oracle.F16)
    yh = to_host(y)
    check_y(yh, y_ref, F16, what)
    check_rowsums(yh, F16, None, what)
    check_state(m.cpu().numpy(), d.cpu().numpy(), lse.cpu().numpy(), m_ref, d_ref, lse_ref, what)


def test_f16_special_values():
    """Largest finite fp16 (65504), subnormal inputs, -inf entries, a fully masked row, a uniform row."""
    N = 4096
    rng = np.random.default_rng(6)
    rows = (rng.standard_normal((6, N)) * 3).astype(np.float32)
    rows[0, 17] = 65504.0
    rows[1] = rng.standard_normal(N).astype(np.float32) * 1e-6   # subnormal fp16 inputs
    rows[2, 100:] = -np.inf
    rows[3, :] = -np.inf
    rows[4, :] = 0.5
    rows[5] -= 60000.0
    x_host = synth.f32_to_f16(rows)
    for variant in (V.VARIANT_AUTO, V.VARIANT_ONEREAD_REG, V.VARIANT_ONEREAD_SMEM, V.VARIANT_TWOPASS):
        y, m, d, lse = _run(to_device(x_host, F16), variant)
        what = f"f16 special/{V.VARIANT_NAMES[rwo.last_variant()]}"
        y_ref, m_ref, d_ref, lse_ref = oracle.softmax_rows(x_host, dtype=oracle.F16)
        yh = to_host(y)
        check_y(yh, y_ref, F16, what)
        check_rowsums(yh, F16, ~np.isfinite(m_ref), what)
        check_state(m.cpu().numpy(), d.cpu().numpy(), lse.cpu().numpy(), m_ref, d_ref, lse_ref, what)


def test_f16_split_row():
    w = synth.custom("f16-split", F16, 3, 1 << 21, seed=31, dist=synth.UNIFORM, p0=-8.0, p1=8.0)
    x_host = synth.generate(w)
    y, m, d, lse = _run(to_device(x_host, F16), V.VARIANT_SPLITROW)
    assert rwo.last_variant() == V.VARIANT_SPLITROW
    y_ref, m_ref, d_ref, lse_ref = oracle.softmax_rows(x_host, dtype=oracle.F16)
    check_y(to_host(y), y_ref, F16, "f16 split")
    check_state(m.cpu().numpy(), d.cpu().numpy(), lse.cpu().numpy(), m_ref, d_ref, lse_ref, "f16 split")


def test_f16_log_softmax_and_cross_entropy():
    w = synth.custom("f16-log", F16, 400, 4104, seed=32, p1=4.0)
    x_host = synth.generate(w)
    x = to_device(x_host, F16)
    for variant in (V.VARIANT_AUTO, V.VARIANT_ONEREAD_SMEM, V.VARIANT_TWOPASS):
        y = rwo.log_softmax_rows(x, variant=variant)
        assert rwo.get_status() == rwo.OK
        check_log_values(to_host(y), oracle.log_softmax_rows(x_host, dtype=oracle.F16), F16, "f16 log")
    labels = np.random.default_rng(3).integers(0, w.N, w.M)
    loss = rwo.cross_entropy_rows(x, torch.from_numpy(labels).cuda())
    assert rwo.get_status() == rwo.OK
    check_log_values(loss.cpu().numpy(), oracle.cross_entropy_rows(x_host, labels, dtype=oracle.F16), synth.F32,
                     "f16 ce")


def test_f16_causal():
    M, N, Q = 512, 4096, 256
    w = synth.custom("f16-causal", F16, M, N, seed=33, p1=2.0)
    x_host = synth.generate(w)
    lengths = np.clip(np.arange(M) % Q + 1, 0, N)
    masked = np.arange(N)[None, :] >= lengths[:, None]
    ref_in = np.where(masked, np.uint16(0xFC00), x_host).astype(np.uint16)   # -inf
    gpu_in = np.where(masked, np.uint16(0x7E00), x_host).astype(np.uint16)   # NaN: must never be read
    y = rwo.softmax_rows_causal(to_device(gpu_in, F16), Q)
    assert rwo.get_status() == rwo.OK and rwo.last_variant() == V.VARIANT_ONEREAD_SMEM
    y_ref, *_ = oracle.softmax_rows(ref_in, dtype=oracle.F16)
    check_y(to_host(y), y_ref, F16, "f16 causal")
