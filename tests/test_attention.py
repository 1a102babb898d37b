"""attention_forward (the FlashAttention forward tile on tcgen05) against the fp64 oracle.

Tolerance, derived from the arithmetic: scores and the row state are fp32 (bf16 and fp16 products
are exact in fp32); P is rounded to the element type before the P V product (relative 2^-9 per
weight for bf16, 2^-11 for fp16) while l sums the unrounded weights, so |O - O_ref| <= 2^-9 (2^-11)
max_j |v_j| plus the output's own rounding; the test allows 2^-8 (bf16) or 2^-10 (fp16) max|v| + one
ulp of O_ref in the element type.  LSE within 1e-4 max(1, |LSE|).
"""
import numpy as np
import pytest
import torch

import oracle
import row_wise_online_gb300 as rwo
import synth
from gpu_util import to_device, to_host
from tolerances import bf16_ulp, f16_ulp

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from row_wise_online_gb300 import _build

    _build.build()
    torch.cuda.set_device(0)


def _qkv(BH, Sq, Sk, d, seed, q_sd=1.0, dtype=synth.BF16):
    gen = lambda M, N, s, sd: synth.generate(synth.custom("attn", dtype, M, N, seed=s, p1=sd))
    q = gen(BH * Sq, d, seed, q_sd).reshape(BH, Sq, d)
    k = gen(BH * Sk, d, seed + 1, 1.0).reshape(BH, Sk, d)
    v = gen(BH * Sk, d, seed + 2, 1.0).reshape(BH, Sk, d)
    return q, k, v


def _check(o_gpu, lse_gpu, q, k, v, rows, causal, scale, what, dtype=synth.BF16):
    o_ref, lse_ref = oracle.attention_rows(q, k, v, rows, dtype=dtype, scale=scale, causal=causal)
    widen = synth.f16_to_f32 if dtype == synth.F16 else synth.bf16_to_f32
    vmax = np.abs(widen(v).astype(np.float64)).max(axis=(1, 2))
    idx = np.asarray(rows)
    og = widen(o_gpu[idx[:, 0], idx[:, 1]]).astype(np.float64)
    if dtype == synth.F16:
        bound = (2.0 ** -10) * vmax[idx[:, 0]][:, None] + f16_ulp(o_ref)
    else:
        bound = (2.0 ** -8) * vmax[idx[:, 0]][:, None] + bf16_ulp(o_ref)
    err = np.abs(og - o_ref)
    bad = ~(err <= bound)
    assert not bad.any(), f"{what}: {bad.sum()} outputs off; worst {err.max()} at {np.unravel_index(np.argmax(err), err.shape)}"
    lg = lse_gpu[idx[:, 0], idx[:, 1]].astype(np.float64)
    fin = np.isfinite(lse_ref)
    assert np.all(np.isneginf(lg[~fin]))
    assert np.all(np.abs(lg[fin] - lse_ref[fin]) <= 1e-4 * np.maximum(1.0, np.abs(lse_ref[fin]))), f"{what}: LSE"


@pytest.mark.parametrize("BH,Sq,Sk", [(1, 128, 128), (2, 300, 300), (3, 1, 1), (2, 128, 1000), (2, 513, 513),
                                     (2, 1000, 77), (1, 77, 1000), (2, 256, 384)])
@pytest.mark.parametrize("causal", [False, True])
def test_attention_against_oracle(BH, Sq, Sk, causal):
    d = 128
    q, k, v = _qkv(BH, Sq, Sk, d, seed=Sq * 7 + Sk)
    lse = torch.full((BH, Sq), float("nan"), device="cuda")
    o = rwo.attention_forward(to_device(q), to_device(k), to_device(v), lse_out=lse, causal=causal)
    assert rwo.get_status() == rwo.OK
    rows = [(h, i) for h in range(BH) for i in range(Sq)]
    _check(to_host(o), lse.cpu().numpy(), q, k, v, rows, causal, 1.0 / np.sqrt(d), f"attn {BH}x{Sq}x{Sk} causal={causal}")


@pytest.mark.parametrize("BH,Sq,Sk", [(2, 300, 300), (1, 77, 1000), (2, 256, 384), (2, 1000, 77)])
@pytest.mark.parametrize("causal", [False, True])
def test_attention_f16_against_oracle(BH, Sq, Sk, causal):
    d = 128
    q, k, v = _qkv(BH, Sq, Sk, d, seed=Sq * 5 + Sk, dtype=synth.F16)
    lse = torch.full((BH, Sq), float("nan"), device="cuda")
    qd, kd, vd = (to_device(t, synth.F16) for t in (q, k, v))
    o = rwo.attention_forward(qd, kd, vd, lse_out=lse, causal=causal)
    assert o.dtype == torch.float16
    rows = [(h, i) for h in range(BH) for i in range(Sq)]
    _check(to_host(o), lse.cpu().numpy(), q, k, v, rows, causal, 1.0 / np.sqrt(d),
           f"attn fp16 {BH}x{Sq}x{Sk} causal={causal}", dtype=synth.F16)


@pytest.mark.parametrize("dtype", [synth.BF16, synth.F16])
@pytest.mark.parametrize("BH,Sq,Sk", [(2, 300, 300), (1, 77, 1000), (2, 256, 384), (2, 1000, 77), (3, 1, 1)])
@pytest.mark.parametrize("causal", [False, True])
def test_attention_d64_against_oracle(dtype, BH, Sq, Sk, causal):
    d = 64
    q, k, v = _qkv(BH, Sq, Sk, d, seed=Sq * 3 + Sk + d, dtype=dtype)
    lse = torch.full((BH, Sq), float("nan"), device="cuda")
    qd, kd, vd = (to_device(t, dtype) for t in (q, k, v))
    o = rwo.attention_forward(qd, kd, vd, lse_out=lse, causal=causal)
    assert rwo.get_status() == rwo.OK
    rows = [(h, i) for h in range(BH) for i in range(Sq)]
    _check(to_host(o), lse.cpu().numpy(), q, k, v, rows, causal, 1.0 / np.sqrt(d),
           f"attn d=64 {BH}x{Sq}x{Sk} causal={causal}", dtype=dtype)


def test_attention_large_scores_and_scale():
    """Scores spread over hundreds (sharp rows) with a non-default scale."""
    BH, S, d = 2, 384, 128
    q, k, v = _qkv(BH, S, S, d, seed=91, q_sd=8.0)
    lse = torch.empty((BH, S), device="cuda")
    o = rwo.attention_forward(to_device(q), to_device(k), to_device(v), lse_out=lse, scale=0.3, causal=True)
    assert rwo.get_status() == rwo.OK
    _check(to_host(o), lse.cpu().numpy(), q, k, v, [(h, i) for h in range(BH) for i in range(S)], True, 0.3, "sharp")


def test_attention_default_scale_is_one_over_sqrt_d():
    """scale 0 (the binding's default) is the library's 1/sqrt(d): bitwise the explicit value."""
    for d in (64, 128):
        q, k, v = _qkv(1, 200, 300, d, seed=95)
        qd, kd, vd = to_device(q), to_device(k), to_device(v)
        la, lb = torch.empty((1, 200), device="cuda"), torch.empty((1, 200), device="cuda")
        oa = rwo.attention_forward(qd, kd, vd, lse_out=la)
        ob = rwo.attention_forward(qd, kd, vd, lse_out=lb, scale=float(np.float32(1.0 / np.sqrt(d))))
        assert rwo.get_status() == rwo.OK
        assert torch.equal(oa, ob) and torch.equal(la, lb)
        _check(to_host(oa), la.cpu().numpy(), q, k, v, [(0, i) for i in range(0, 200, 7)], False, 1.0 / np.sqrt(d),
               f"default scale d={d}")


@pytest.mark.parametrize("BH,S", [(70, 384), (3, 33000)])
def test_attention_causal_cta_order(BH, S):
    """Causal CTAs run in head groups of ~128 CTAs: a partial last group (70 heads of 2 pairs:
    groups of 64) and one head per group (129 pairs of 256 rows); sampled rows against the oracle,
    every row's LSE finite and every head's first and last rows included."""
    d = 128
    q, k, v = _qkv(BH, S, S, d, seed=BH * 3 + S)
    lse = torch.full((BH, S), float("nan"), device="cuda")
    o = rwo.attention_forward(to_device(q), to_device(k), to_device(v), lse_out=lse, causal=True)
    assert rwo.get_status() == rwo.OK
    lse_h = lse.cpu().numpy()
    assert np.all(np.isfinite(lse_h)), "every row sees at least its own key"
    rng = np.random.default_rng(BH + S)
    rows = sorted({(h, i) for h in range(BH) for i in (0, S - 1)} |
                  {(int(h), int(i)) for h, i in zip(rng.integers(0, BH, 96), rng.integers(0, S, 96))})
    _check(to_host(o), lse_h, q, k, v, rows, True, 1.0 / np.sqrt(d), f"causal order {BH}x{S}")


def test_attention_causal_workload_full_size():
    """4 x 32 heads, 4096 queries and keys, d = 128, causal: sampled rows against the oracle."""
    BH, S, d = 128, 4096, 128
    q, k, v = _qkv(BH, S, S, d, seed=5)
    lse = torch.empty((BH, S), device="cuda")
    o = rwo.attention_forward(to_device(q), to_device(k), to_device(v), lse_out=lse, causal=True)
    assert rwo.get_status() == rwo.OK
    rng = np.random.default_rng(3)
    rows = [(int(h), int(i)) for h, i in zip(rng.integers(0, BH, 48), rng.integers(0, S, 48))]
    rows += [(0, 0), (0, 127), (0, 128), (77, 4095), (127, 4095), (127, 2048)]
    _check(to_host(o), lse.cpu().numpy(), q, k, v, rows, True, 1.0 / np.sqrt(d), "causal 128x4096")


def test_attention_wait_runs_out_and_reports_timeout():
    """A V tile that is never copied: every wait on it runs out (bounded), the kernel terminates
    with SOFTMAX_ERR_TIMEOUT, and the next launch is correct."""
    BH, S, d = 1, 256, 128
    q, k, v = _qkv(BH, S, S, d, seed=3)
    qd, kd, vd = to_device(q), to_device(k), to_device(v)
    assert rwo.get_status() == rwo.OK
    old_limit = rwo.debug_set_wait_limit_ns(5_000_000)  # 5 ms
    old_fault = rwo.debug_set_fault(2)
    try:
        rwo.attention_forward(qd, kd, vd)
        assert rwo.get_status() == rwo.ERR_TIMEOUT
    finally:
        rwo.debug_set_fault(old_fault)
        rwo.debug_set_wait_limit_ns(old_limit)
    assert rwo.get_status() == rwo.OK
    lse = torch.empty((BH, S), device="cuda")
    o = rwo.attention_forward(qd, kd, vd, lse_out=lse)
    assert rwo.get_status() == rwo.OK
    _check(to_host(o), lse.cpu().numpy(), q, k, v, [(0, i) for i in range(S)], False, 1.0 / np.sqrt(d), "after timeout")


def test_attention_unsupported_and_errors():
    q = torch.zeros((1, 16, 96), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(rwo.SoftmaxError) as ei:
        rwo.attention_forward(q, q, q)  # d = 96
    assert ei.value.status == rwo.ERR_UNSUPPORTED
    q = torch.zeros((1, 16, 128), dtype=torch.float32, device="cuda")
    with pytest.raises(rwo.SoftmaxError) as ei:
        rwo.attention_forward(q, q, q)  # fp32
    assert ei.value.status == rwo.ERR_UNSUPPORTED
    q = torch.zeros((1, 16, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(rwo.SoftmaxError) as ei:
        rwo.attention_forward(q, q, q, scale=-1.0)
    assert ei.value.status == rwo.ERR_INVALID_ARG
