"""log_softmax_rows and cross_entropy_rows against the fp64 oracle ("从原始Softmax到在线Softmax",
section "softmax实际代码实现": log_probs = logits - max - log(sum_exp), loss = -log_probs[label]).

Every kernel that writes log softmax (register, CTA bulk-copy, two-pass) is compared element by
element on small and ragged shapes; the bf16 logits workload (16384 x 32768) runs at full size in
the benchmark's launch configuration, sampled rows against the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import row_wise_online_gb300 as rwo
import synth
from gpu_util import to_device, to_host
from tolerances import check_log_values, check_state

pytestmark = pytest.mark.gpu
V = rwo


@pytest.fixture(scope="module", autouse=True)
def _built():
    from row_wise_online_gb300 import _build

    _build.build()
    torch.cuda.set_device(0)


def _run_log(x, variant):
    M = x.numel() // x.shape[-1]
    m, d, lse = (torch.full((M,), float("nan"), device="cuda") for _ in range(3))
    y = rwo.log_softmax_rows(x, m_out=m, d_out=d, lse_out=lse, variant=variant)
    assert rwo.get_status() == rwo.OK
    return y, m, d, lse


SHAPES = [
    (synth.F32, 64, 1024), (synth.F32, 1000, 1000), (synth.F32, 300, 4100), (synth.F32, 65, 20000),
    (synth.BF16, 1000, 1000), (synth.BF16, 517, 4104), (synth.BF16, 70, 32768), (synth.BF16, 33, 40000),
    (synth.F32, 400, 20480), (synth.F32, 400, 32764),  # fp32 rows of 80 and ~128 KiB: one row slot a CTA
    (synth.BF16, 400, 50264),                           # 98 KiB of bf16: x kept packed
    (synth.F32, 300, 40000), (synth.BF16, 200, 100000), (synth.F32, 260, 200000),  # a cluster per row
]


@pytest.mark.parametrize("dtype,M,N", SHAPES)
@pytest.mark.parametrize("variant", [V.VARIANT_AUTO, V.VARIANT_ONEREAD_REG, V.VARIANT_ONEREAD_SMEM,
                                     V.VARIANT_TWOPASS])
def test_log_softmax_against_oracle(dtype, M, N, variant):
    w = synth.custom("logsm", dtype, M, N, seed=300 + N, p1=4.0)
    x_host = synth.generate(w)
    x = to_device(x_host)
    try:
        y, m, d, lse = _run_log(x, variant)
    except rwo.SoftmaxError as e:
        assert variant != V.VARIANT_AUTO and e.status == rwo.ERR_UNSUPPORTED
        return
    what = f"log {M}x{N}/{V.VARIANT_NAMES[rwo.last_variant()]}"
    ly_ref = oracle.log_softmax_rows(x_host)
    check_log_values(to_host(y), ly_ref, dtype, what)
    _, m_ref, d_ref, lse_ref = oracle.softmax_rows(x_host, want_y=False)
    check_state(m.cpu().numpy(), d.cpu().numpy(), lse.cpu().numpy(), m_ref, d_ref, lse_ref, what)


@pytest.mark.parametrize("variant", [V.VARIANT_AUTO, V.VARIANT_ONEREAD_REG, V.VARIANT_ONEREAD_SMEM,
                                     V.VARIANT_TWOPASS])
def test_log_softmax_masked_and_extreme_rows(variant):
    N = 2048
    rng = np.random.default_rng(3)
    rows = (rng.standard_normal((6, N)) * 3).astype(np.float32)
    rows[0, 100:] = -np.inf     # masked tail
    rows[1, :] = -np.inf        # fully masked: log 0 everywhere
    rows[2, 7] = 1e30           # one huge value
    rows[3] -= 1e30             # huge negative row (shift invariance)
    rows[4, ::2] = -np.inf
    rows[5, :] = 0.25           # uniform: -ln N
    x = to_device(rows)
    y, m, d, lse = _run_log(x, variant)
    what = f"log special/{V.VARIANT_NAMES[rwo.last_variant()]}"
    ly_ref = oracle.log_softmax_rows(rows)
    check_log_values(to_host(y), ly_ref, synth.F32, what)
    _, m_ref, d_ref, lse_ref = oracle.softmax_rows(rows, want_y=False)
    check_state(m.cpu().numpy(), d.cpu().numpy(), lse.cpu().numpy(), m_ref, d_ref, lse_ref, what)


@pytest.mark.parametrize("variant", [V.VARIANT_AUTO, V.VARIANT_ONEREAD_SMEM])
def test_log_softmax_cluster_rows_special_values(variant):
    """Rows of 160 KB held on chip by a thread-block cluster, log output: an all -inf row (-inf
    everywhere), a row whose first quarter is -inf (a CTA's whole segment empty), one huge value,
    a huge negative row."""
    M, N = 200, 40000
    rng = np.random.default_rng(9)
    rows = (rng.standard_normal((M, N)) * 3).astype(np.float32)
    rows[0, :] = -np.inf
    rows[1, :N // 4] = -np.inf
    rows[2, N - 1] = 1e30
    rows[3] -= 1e30
    x = to_device(rows)
    y, m, d, lse = _run_log(x, variant)
    assert rwo.last_variant() == V.VARIANT_ONEREAD_SMEM
    what = f"log cluster special/{V.VARIANT_NAMES[variant]}"
    check_log_values(to_host(y), oracle.log_softmax_rows(rows), synth.F32, what)
    _, m_ref, d_ref, lse_ref = oracle.softmax_rows(rows, want_y=False)
    check_state(m.cpu().numpy(), d.cpu().numpy(), lse.cpu().numpy(), m_ref, d_ref, lse_ref, what)


def test_log_softmax_unaligned_base():
    w = synth.custom("log-unaligned", synth.BF16, 123, 1001, seed=21, p1=3.0)
    x_host = synth.generate(w)
    buf = torch.empty(w.M * w.N + 8, dtype=torch.bfloat16, device="cuda")
    out = torch.full((w.M * w.N + 8,), 5.0, dtype=torch.bfloat16, device="cuda")
    x = buf[1:1 + w.M * w.N].view(w.M, w.N)
    y = out[1:1 + w.M * w.N].view(w.M, w.N)
    x.copy_(to_device(x_host))
    rwo.log_softmax_rows(x, y)
    assert rwo.get_status() == rwo.OK
    check_log_values(to_host(y), oracle.log_softmax_rows(x_host), synth.BF16, "log unaligned")
    assert torch.all(out[:1] == 5.0) and torch.all(out[1 + w.M * w.N:] == 5.0)


def test_log_softmax_splitrow_is_unsupported():
    x = torch.zeros((2, 1 << 20), device="cuda")
    with pytest.raises(rwo.SoftmaxError) as ei:
        rwo.log_softmax_rows(x, variant=V.VARIANT_SPLITROW)
    assert ei.value.status == rwo.ERR_UNSUPPORTED


def test_log_softmax_logits_workload_full_size():
    """bf16 16384 x 32768 logits, AUTO (the CTA bulk-copy kernel): sampled rows against the oracle,
    every row for m (exact) and for logsumexp(y) = 0."""
    w = synth.WORKLOADS["bf16_logits_16384x32768"]
    x = to_device(synth.generate(w))
    m = torch.empty(w.M, device="cuda")
    y = rwo.log_softmax_rows(x, m_out=m)
    assert rwo.get_status() == rwo.OK and rwo.last_variant() == V.VARIANT_ONEREAD_SMEM
    assert torch.equal(m, x.amax(dim=1).float())
    # sum_j exp(log y_j) = 1 for every row, up to each value's bf16 rounding (half an ulp) plus the
    # kernel's own 1e-5 * max(1, |log y_j|): exp of the error bounds each term's relative error.
    v = y.double()
    a = v.abs()
    ulp = torch.where(a > 0, torch.exp2(torch.floor(torch.log2(torch.where(a > 0, a, 1.0))) - 7), 0.0)
    h = ulp / 2 + 1e-5 * torch.clamp(a, min=1.0)
    ev = torch.exp(v)
    dev = (ev.sum(dim=1) - 1).abs()
    bound = (ev * torch.expm1(h)).sum(dim=1) + 1e-6
    assert bool(torch.all(dev <= bound)), float((dev / bound).max())
    del v, a, ulp, h, ev
    rows = np.unique(np.concatenate([np.random.default_rng(8).integers(0, w.M, 24), [0, 100, 16300, w.M - 1]]))
    ly_ref = oracle.log_softmax_rows(synth.generate_rows(w, rows))
    idx = torch.from_numpy(rows).cuda()
    check_log_values(to_host(y.index_select(0, idx)), ly_ref, w.dtype, "log logits workload")


# ---------------------------------------------------------------------------------------------
# cross entropy
# ---------------------------------------------------------------------------------------------


@pytest.mark.parametrize("dtype,M,N,shift", [
    (synth.F32, 64, 1024, 0), (synth.F32, 500, 1001, 1), (synth.BF16, 300, 32768, 0), (synth.BF16, 77, 50000, 1),
    (synth.F32, 5, 1, 0), (synth.F32, 400, 24576, 0),
])
def test_cross_entropy_against_oracle(dtype, M, N, shift):
    w = synth.custom("ce", dtype, M, N, seed=40 + N, p1=4.0)
    x_host = synth.generate(w)
    rng = np.random.default_rng(N)
    labels = rng.integers(0, N, M)
    labels[::7] = -1  # ignored rows
    tdt = torch.float32 if dtype == synth.F32 else torch.bfloat16
    buf = torch.empty(M * N + 8, dtype=tdt, device="cuda")
    x = buf[shift:shift + M * N].view(M, N)
    x.copy_(to_device(x_host))
    lab = torch.from_numpy(labels).cuda()
    lse = torch.full((M,), float("nan"), device="cuda")
    loss = rwo.cross_entropy_rows(x, lab, lse_out=lse)
    assert rwo.get_status() == rwo.OK
    what = f"ce {M}x{N}"
    check_log_values(loss.cpu().numpy(), oracle.cross_entropy_rows(x_host, labels), synth.F32, what)
    _, m_ref, d_ref, lse_ref = oracle.softmax_rows(x_host, want_y=False)
    check_state(None, None, lse.cpu().numpy(), m_ref, d_ref, lse_ref, what)


def test_cross_entropy_logits_workload_full_size():
    w = synth.WORKLOADS["bf16_logits_16384x32768"]
    x_host = synth.generate(w)
    labels = np.random.default_rng(12).integers(0, w.N, w.M)
    loss = rwo.cross_entropy_rows(to_device(x_host), torch.from_numpy(labels).cuda())
    assert rwo.get_status() == rwo.OK
    check_log_values(loss.cpu().numpy(), oracle.cross_entropy_rows(x_host, labels), synth.F32, "ce logits")


def test_cross_entropy_masked_rows_and_bad_label():
    rows = np.array([[1.0, -np.inf, 2.0, 0.5], [-np.inf] * 4, [3.0, 1.0, -np.inf, 0.0], [0.0, 1.0, 2.0, 3.0]],
                    np.float32)
    x = to_device(rows)
    labels = np.array([1, 0, 0, 3])  # masked labelled entry: +inf; all -inf row: NaN
    loss = rwo.cross_entropy_rows(x, torch.from_numpy(labels).cuda())
    assert rwo.get_status() == rwo.OK
    check_log_values(loss.cpu().numpy(), oracle.cross_entropy_rows(rows, labels), synth.F32, "ce masked")
    # a label >= N: NaN for that row, the others unaffected, the status word reports it once
    bad = np.array([0, 1, 4, 3])
    loss = rwo.cross_entropy_rows(x, torch.from_numpy(bad).cuda())
    assert rwo.get_status() == rwo.ERR_INVALID_ARG
    assert rwo.get_status() == rwo.OK
    check_log_values(loss.cpu().numpy(), oracle.cross_entropy_rows(rows, bad), synth.F32, "ce bad label")


@pytest.mark.parametrize("dtype,N", [(synth.F32, 8196), (synth.F32, 40000), (synth.BF16, 50264),
                                     (synth.BF16, 151936), (synth.F16, 100000)])
def test_cross_entropy_rows_streamed_in_chunks(dtype, N):
    """Rows longer than 32 KiB reach the state-only kernel in 32 KiB chunks.  Labels on both sides
    of every chunk boundary, on the first and last entries, ignored (-1); rows whose maximum sits
    in the last chunk (every chunk's state rescaled at the merge), whose first chunk is all -inf,
    whose only finite entry is the last one, and one that is all -inf (loss NaN); against the
    fp64 oracle, with the LSE."""
    M = 300
    w = synth.custom("ce-chunks", dtype, M, N, seed=N % 83, p1=4.0)
    x_host = synth.generate(w)
    per_chunk = 32768 // (4 if dtype == synth.F32 else 2)
    f32 = synth.bf16_to_f32 if dtype == synth.BF16 else synth.f16_to_f32 if dtype == synth.F16 else None
    rows = x_host.astype(np.float32) if f32 is None else f32(x_host)
    rows[0, N - 3] = 40.0           # the maximum in the last chunk
    rows[1, :per_chunk] = -np.inf   # the first chunk empty
    rows[2, :N - 1] = -np.inf       # only the last entry finite
    rows[3, :] = -np.inf            # all -inf: NaN
    if dtype == synth.F32:
        x_host = rows
    else:
        x_host = synth.f32_to_bf16(rows) if dtype == synth.BF16 else synth.f32_to_f16(rows)
    rng = np.random.default_rng(N)
    labels = rng.integers(0, N, M)
    edges = [0, N - 1] + [c * per_chunk + o for c in range(1, (N - 1) // per_chunk + 1) for o in (-1, 0)]
    labels[4:4 + len(edges)] = edges
    labels[::11] = -1
    labels[1] = per_chunk // 2       # an -inf labelled entry: +inf loss
    x = to_device(x_host, dtype) if dtype == synth.F16 else to_device(x_host)
    lse = torch.full((M,), float("nan"), device="cuda")
    loss = rwo.cross_entropy_rows(x, torch.from_numpy(labels).cuda(), lse_out=lse)
    assert rwo.get_status() == rwo.OK
    assert rwo.last_variant() == V.VARIANT_ONEREAD_SMEM
    what = f"ce chunks {N}"
    odt = {synth.F32: oracle.F32, synth.BF16: oracle.BF16, synth.F16: oracle.F16}[dtype]
    check_log_values(loss.cpu().numpy(), oracle.cross_entropy_rows(x_host, labels, dtype=odt), synth.F32, what)
    _, m_ref, d_ref, lse_ref = oracle.softmax_rows(x_host, dtype=odt, want_y=False)
    check_state(None, None, lse.cpu().numpy(), m_ref, d_ref, lse_ref, what)


@pytest.mark.parametrize("dtype", [synth.F32, synth.BF16])
def test_cross_entropy_large_magnitude_rows(dtype):
    """Row maxima on both sides of 2^20 (the shifted-exponent fast path and its fallback), huge
    values and huge negative rows: loss and LSE against the oracle."""
    N = 4096
    rng = np.random.default_rng(17)
    base = rng.standard_normal((8, N)) * 2
    rows = base.copy()
    rows[0] += 1000.0
    rows[1] += 2.0 ** 20 * 0.99
    rows[2] += 2.0 ** 20 * 1.01
    rows[3] -= 2.0 ** 21
    rows[4, 123] = 1e30
    rows[5] -= 1e30
    rows[6] *= 40.0
    rows[7] += 3.0e5
    rows = rows.astype(np.float32)
    if dtype == synth.BF16:
        rows_in = synth.f32_to_bf16(rows)
    else:
        rows_in = rows
    labels = np.array([5, 9, 4000, 17, 123, 0, 2047, 4095])
    lse = torch.empty(8, device="cuda")
    loss = rwo.cross_entropy_rows(to_device(rows_in), torch.from_numpy(labels).cuda(), lse_out=lse)
    assert rwo.get_status() == rwo.OK
    check_log_values(loss.cpu().numpy(), oracle.cross_entropy_rows(rows_in, labels), synth.F32, "ce large")
    _, m_ref, d_ref, lse_ref = oracle.softmax_rows(rows_in, want_y=False)
    check_state(None, None, lse.cpu().numpy(), m_ref, d_ref, lse_ref, "ce large")
    m, d, l2 = rwo.softmax_row_state(to_device(rows_in))
    check_state(m.cpu().numpy(), d.cpu().numpy(), l2.cpu().numpy(), m_ref, d_ref, lse_ref, "state large")
