"""softmax_row_state and merge_states on the GPU: the per-row state against the oracle, and the
chunk test of "Softmax 数值稳定性与 IO-Aware Attention" §4.1 -- cut rows into random chunks,
compute each chunk's state, merge them repeatedly; the result is the whole row's state."""
import math

import numpy as np
import pytest
import torch

import oracle
import row_wise_online_gb300 as rwo
import synth
from gpu_util import to_device
from tolerances import check_state

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from row_wise_online_gb300 import _build

    _build.build()
    torch.cuda.set_device(0)


@pytest.mark.parametrize("dtype,M,N", [(synth.F32, 64, 1024), (synth.F32, 300, 4100), (synth.BF16, 100, 32768),
                                       (synth.BF16, 9, 7), (synth.F32, 4, 1 << 20),
                                       # rows streamed in 32 KiB chunks: a 16-byte last chunk, ragged
                                       # chunks, many rows per CTA
                                       (synth.F32, 150, 8196), (synth.BF16, 700, 50264), (synth.F32, 500, 30000)])
def test_row_state_against_oracle(dtype, M, N):
    w = synth.custom("state", dtype, M, N, seed=N % 97, p1=4.0)
    x_host = synth.generate(w)
    m, d, lse = rwo.softmax_row_state(to_device(x_host))
    torch.cuda.synchronize()
    _, m_ref, d_ref, lse_ref = oracle.softmax_rows(x_host, want_y=False)
    check_state(m.cpu().numpy(), d.cpu().numpy(), lse.cpu().numpy(), m_ref, d_ref, lse_ref, "row_state")


def _empty(M):
    return (torch.full((M,), -math.inf, device="cuda"), torch.zeros(M, device="cuda"))


def test_random_chunks_merge_to_whole_row():
    rng = np.random.default_rng(3)
    for trial in range(12):
        M = int(rng.integers(1, 200))
        N = int(rng.integers(1, 20000))
        dtype = synth.F32 if trial % 2 == 0 else synth.BF16
        w = synth.custom("chunks", dtype, M, N, seed=trial, p1=float(rng.choice([1.0, 5.0, 20.0])))
        x_host = synth.generate(w)
        if trial % 3 == 0 and N > 4:  # a chunk that is entirely -inf
            lo = N // 4
            inf_bits = np.float32(-np.inf) if dtype == synth.F32 else synth.f32_to_bf16(np.float32([-np.inf]))[0]
            x_host[:, lo:lo + N // 4] = inf_bits
        x = to_device(x_host)
        ncuts = int(rng.integers(0, 8))
        cuts = sorted(set(int(c) for c in rng.integers(1, N, ncuts))) if N > 1 else []
        bounds = [0] + cuts + [N]
        m_acc, d_acc = _empty(M)
        order = list(range(len(bounds) - 1))
        rng.shuffle(order)  # merge order is free: the merge is associative and commutative
        for i in order:
            a, b = bounds[i], bounds[i + 1]
            m_c, d_c, _ = rwo.softmax_row_state(x[:, a:b].contiguous())
            rwo.merge_states(m_acc, d_acc, m_c, d_c, m_acc, d_acc)  # in place
        lse = torch.empty(M, device="cuda")
        rwo.merge_states(m_acc, d_acc, *_empty(M), m_acc, d_acc, lse)  # identity merge, with LSE
        torch.cuda.synchronize()
        _, m_ref, d_ref, lse_ref = oracle.softmax_rows(x_host, want_y=False)
        check_state(m_acc.cpu().numpy(), d_acc.cpu().numpy(), lse.cpu().numpy(), m_ref, d_ref, lse_ref,
                    f"chunks trial {trial}")


def test_merge_states_empty_operands_against_oracle_merge():
    vals = [(-math.inf, 0.0), (2.0, 1.6065), (3.0, 1.0821), (-1e30, 5.0), (1e30, 1.0), (0.0, 7.0)]
    pairs = [(a, b) for a in vals for b in vals]
    ma = torch.tensor([p[0][0] for p in pairs], dtype=torch.float32, device="cuda")
    da = torch.tensor([p[0][1] for p in pairs], dtype=torch.float32, device="cuda")
    mb = torch.tensor([p[1][0] for p in pairs], dtype=torch.float32, device="cuda")
    db = torch.tensor([p[1][1] for p in pairs], dtype=torch.float32, device="cuda")
    lse = torch.empty_like(ma)
    m, d, _ = rwo.merge_states(ma, da, mb, db, lse_out=lse)
    torch.cuda.synchronize()
    m, d, lse = m.cpu().numpy(), d.cpu().numpy(), lse.cpu().numpy()
    for i, (a, b) in enumerate(pairs):
        a32 = (float(np.float32(a[0])), float(np.float32(a[1])))
        b32 = (float(np.float32(b[0])), float(np.float32(b[1])))
        rm, rd = oracle.merge_state(a32, b32)
        assert m[i] == np.float32(rm), (a, b)
        assert abs(d[i] - rd) <= 1e-6 * rd, (a, b, d[i], rd)
        if rm == -math.inf:
            assert d[i] == 0.0 and lse[i] == -np.inf
        else:
            assert abs(lse[i] - (rm + math.log(rd))) <= 1e-5 * max(1.0, abs(rm + math.log(rd)))
