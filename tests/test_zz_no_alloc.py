"""The allocation-free split-row entry point, called through the C ABI.

softmax_rows_splitrow_noalloc serves callers that cannot let a library allocate device memory
(a memory budget fixed in advance, a framework allocator that owns the device, a host thread
that must not block on an allocation).  It keeps its exchange scratch in a fixed device array
shared by every call, so two calls in a row must each give the same result as the regular
split-row call, which takes its scratch from the memory pool per call.  This file is collected
last.
"""
import ctypes

import numpy as np
import pytest
import torch

import row_wise_online_gb300 as rwo
import synth
from gpu_util import to_device, to_host
from tolerances import check_state, check_y

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from row_wise_online_gb300 import _build

    _build.build()
    torch.cuda.set_device(0)


def _call_noalloc(x, y, m, d, lse):
    lib = rwo.capi()
    M, N = x.shape
    dtype = rwo.F32 if x.dtype == torch.float32 else rwo.BF16
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    return lib.softmax_rows_splitrow_noalloc(p(x), p(y), p(m), p(d), p(lse), M, N, dtype, stream)


@pytest.mark.parametrize("dtype,M,N,seed", [(synth.F32, 3, 1 << 21, 31), (synth.BF16, 5, 1 << 22, 32)])
def test_no_alloc_matches_regular_split_row_on_two_calls(dtype, M, N, seed):
    for call in range(2):  # the second call reuses the scratch the first one left behind
        w = synth.custom("noalloc", dtype, M, N, seed=seed + call, dist=synth.UNIFORM, p0=-20.0, p1=20.0,
                         late_max=20.0)
        x = to_device(synth.generate(w))
        y = torch.empty_like(x)
        m, d, lse = (torch.full((M,), float("nan"), device="cuda") for _ in range(3))
        assert _call_noalloc(x, y, m, d, lse) == rwo.OK
        assert rwo.get_status() == rwo.OK
        m_ref, d_ref, lse_ref = (torch.empty(M, device="cuda") for _ in range(3))
        y_ref = rwo.softmax_rows_ex(x, m_out=m_ref, d_out=d_ref, lse_out=lse_ref, variant=rwo.VARIANT_SPLITROW)
        assert rwo.get_status() == rwo.OK
        # same kernel and states: compare with the regular call within the parity tolerance
        yr = to_host(y_ref)
        ref = (synth.bf16_to_f32(yr) if dtype == synth.BF16 else yr).astype(np.float64)
        check_y(to_host(y), ref, dtype, f"no-alloc call {call}")
        check_state(m.cpu().numpy(), d.cpu().numpy(), lse.cpu().numpy(), m_ref.cpu().numpy().astype(np.float64),
                    d_ref.cpu().numpy().astype(np.float64), lse_ref.cpu().numpy().astype(np.float64),
                    f"no-alloc call {call}")


def test_no_alloc_rejects_shapes_beyond_its_scratch():
    x = torch.zeros((4096, 1 << 18), device="cuda")  # 4096 rows x 19 clusters > 40960 slots
    y = torch.empty_like(x)
    m = d = lse = torch.empty(4096, device="cuda")
    assert _call_noalloc(x, y, m, d, lse) == rwo.ERR_UNSUPPORTED
    assert rwo.get_status() == rwo.OK
