"""softmax_rows_causal: rows masked by position, masked entries never read.

The oracle sees the masked entries as -inf (the definition); the GPU input holds NaN there, so
any read of a masked entry would show up in the result.  Row lengths follow
L_r = clamp(r % q_period + 1 + key_offset, 0, N).
"""
import numpy as np
import pytest
import torch

import oracle
import row_wise_online_gb300 as rwo
import synth
from gpu_util import to_device, to_host
from tolerances import check_rowsums, check_state, check_y

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from row_wise_online_gb300 import _build

    _build.build()
    torch.cuda.set_device(0)


def _lengths(M, N, q_period, key_offset, row0=0):
    r = np.arange(row0, row0 + M, dtype=np.int64)
    return np.clip(r % q_period + 1 + key_offset, 0, N)


def _masked_inputs(x_host, lengths, dtype):
    """(oracle input with -inf beyond L_r, GPU input with NaN beyond L_r)."""
    cols = np.arange(x_host.shape[1])[None, :]
    masked = cols >= lengths[:, None]
    if dtype == synth.F32:
        ref = np.where(masked, np.float32(-np.inf), x_host).astype(np.float32)
        gpu = np.where(masked, np.float32(np.nan), x_host).astype(np.float32)
    else:
        ref = np.where(masked, np.uint16(0xFF80), x_host).astype(np.uint16)
        gpu = np.where(masked, np.uint16(0x7FC0), x_host).astype(np.uint16)
    return ref, gpu


CASES = [
    # dtype, M, N, q_period, key_offset, base offset (elements)
    (synth.BF16, 600, 4096, 256, 0, 0),       # warp-per-row path, fully masked vectors and chunks
    (synth.F32, 777, 1000, 300, 0, 0),        # ragged tails inside a vector
    (synth.F32, 500, 4096, 4096, -7, 0),      # negative offset: the first rows have L = 0
    (synth.BF16, 300, 2056, 100, 1500, 0),    # offset: long live prefixes
    (synth.F32, 64, 20000, 64, 9000, 0),      # rows > 16 KiB: two-pass over the live prefix
    (synth.BF16, 90, 40000, 45, 30000, 0),
    (synth.F32, 123, 1001, 50, 3, 1),         # unaligned base: scalar two-pass
    (synth.BF16, 77, 4097, 40, 4000, 1),
    (synth.F32, 10, 64, 3, 100, 0),           # offset beyond N: nothing masked
]


@pytest.mark.parametrize("dtype,M,N,q_period,key_offset,shift", CASES)
def test_causal_against_oracle(dtype, M, N, q_period, key_offset, shift):
    w = synth.custom("causal", dtype, M, N, seed=N + q_period, p1=3.0)
    x_host = synth.generate(w)
    lengths = _lengths(M, N, q_period, key_offset)
    ref_in, gpu_in = _masked_inputs(x_host, lengths, dtype)
    tdt = torch.float32 if dtype == synth.F32 else torch.bfloat16
    xbuf = torch.empty(M * N + 8, dtype=tdt, device="cuda")
    ybuf = torch.full((M * N + 8,), 7.0, dtype=tdt, device="cuda")
    x = xbuf[shift:shift + M * N].view(M, N)
    y = ybuf[shift:shift + M * N].view(M, N)
    x.copy_(to_device(gpu_in))
    m, d, lse = (torch.full((M,), float("nan"), device="cuda") for _ in range(3))
    rwo.softmax_rows_causal(x, q_period, key_offset, y, m, d, lse)
    assert rwo.get_status() == rwo.OK
    y_ref, m_ref, d_ref, lse_ref = oracle.softmax_rows(ref_in)
    what = f"causal {M}x{N} Q={q_period} off={key_offset} variant={rwo.VARIANT_NAMES[rwo.last_variant()]}"
    yh = to_host(y)
    check_y(yh, y_ref, dtype, what)
    check_rowsums(yh, dtype, lengths == 0, what)
    check_state(m.cpu().numpy(), d.cpu().numpy(), lse.cpu().numpy(), m_ref, d_ref, lse_ref, what)
    # nothing written outside y
    assert torch.all(ybuf[:shift] == 7.0) and torch.all(ybuf[shift + M * N:] == 7.0)


def test_causal_attention_workload_full_size():
    """The bf16 causal workload (4 x 32 x 4096 queries over 4096 keys): masked keys hold NaN on the
    GPU; sampled rows against the oracle, every row for the row sum and the exact max."""
    w = synth.WORKLOADS["bf16_causal_4x32x4096x4096"]
    x = to_device(synth.generate(w))
    q = torch.arange(w.M, device="cuda") % 4096
    masked = torch.arange(w.N, device="cuda")[None, :] > q[:, None]
    assert torch.all(torch.isneginf(x[masked].float()))
    x_ref_amax = x.amax(dim=1).float()
    x.masked_fill_(masked, float("nan"))
    del masked
    m = torch.empty(w.M, device="cuda")
    y = rwo.softmax_rows_causal(x, 4096, 0, m_out=m)
    assert rwo.get_status() == rwo.OK and rwo.last_variant() == rwo.VARIANT_ONEREAD_SMEM
    assert torch.equal(m, x_ref_amax)
    sums = torch.sum(y, dim=1, dtype=torch.float64)
    assert float((sums - 1).abs().max()) <= 4e-3
    rows = np.unique(np.concatenate([np.random.default_rng(5).integers(0, w.M, 40),
                                     [0, 1, 127, 128, 4095, 4096, w.M - 1]]))
    x_rows = synth.generate_rows(w, rows)
    y_ref, *_ = oracle.softmax_rows(x_rows)
    idx = torch.from_numpy(rows).cuda()
    check_y(to_host(y.index_select(0, idx)), y_ref, w.dtype, "causal workload")


def test_causal_invalid_period():
    x = torch.zeros((4, 64), device="cuda")
    with pytest.raises(rwo.SoftmaxError) as ei:
        rwo.softmax_rows_causal(x, 0)
    assert ei.value.status == rwo.ERR_INVALID_ARG
