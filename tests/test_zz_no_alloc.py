"""The allocation-free split-row entry point, called through the C ABI.

softmax_rows_splitrow_noalloc serves callers that cannot let a library allocate device memory
(a memory budget fixed in advance, a framework allocator that owns the device, a host thread
that must not block on an allocation).  It keeps its exchange scratch in a fixed device array
shared by every call.  Two calls in a row must each give the fp64 oracle's result (within the
parity tolerances) and the regular split-row call's result, and neither may take memory from
the CUDA memory pool or torch's allocator.  This file is collected last.
"""
import ctypes
import glob
import os

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


def _call_noalloc(x, y, m, d, lse):
    lib = rwo.capi()
    M, N = x.shape
    dtype = rwo.F32 if x.dtype == torch.float32 else rwo.BF16
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    return lib.softmax_rows_splitrow_noalloc(p(x), p(y), p(m), p(d), p(lse), M, N, dtype, stream)


class _PoolProbe:
    """High-water mark of the device's current stream-ordered memory pool (the pool cudaMallocAsync
    draws from), read through the CUDA runtime; None where no runtime library can be loaded."""

    USED_MEM_HIGH = 8  # cudaMemPoolAttrUsedMemHigh

    def __init__(self):
        self.rt = None
        cands = ["libcudart.so.13", "/usr/local/cuda/lib64/libcudart.so.13"]
        cands += glob.glob(os.path.join(os.path.dirname(torch.__file__), "..", "nvidia", "cu13", "lib", "libcudart.so*"))
        for c in cands:
            try:
                self.rt = ctypes.CDLL(c)
                break
            except OSError:
                continue
        if self.rt is None:
            return
        self.pool = ctypes.c_void_p()
        if self.rt.cudaDeviceGetMemPool(ctypes.byref(self.pool), ctypes.c_int(torch.cuda.current_device())) != 0:
            self.rt = None

    def reset(self):
        zero = ctypes.c_uint64(0)
        assert self.rt.cudaMemPoolSetAttribute(self.pool, self.USED_MEM_HIGH, ctypes.byref(zero)) == 0

    def high(self) -> int:
        v = ctypes.c_uint64(0)
        assert self.rt.cudaMemPoolGetAttribute(self.pool, self.USED_MEM_HIGH, ctypes.byref(v)) == 0
        return int(v.value)


@pytest.mark.parametrize("dtype,M,N,seed", [(synth.F32, 3, 1 << 21, 31), (synth.BF16, 5, 1 << 22, 32),
                                            (synth.F32, 4, 1 << 25, 33)])
def test_no_alloc_matches_oracle_and_regular_split_row_on_two_calls(dtype, M, N, seed):
    """The last case (128 MiB rows) runs the streaming kernel, the others the on-chip one."""
    probe = _PoolProbe()
    for call in range(2):  # the second call reuses the scratch the first one left behind
        w = synth.custom("noalloc", dtype, M, N, seed=seed + call, dist=synth.UNIFORM, p0=-20.0, p1=20.0,
                         late_max=20.0)
        x_host = synth.generate(w)
        x = to_device(x_host)
        y = torch.empty_like(x)
        m, d, lse = (torch.full((M,), float("nan"), device="cuda") for _ in range(3))
        torch.cuda.synchronize()
        torch.cuda.reset_peak_memory_stats()
        before = torch.cuda.memory_allocated()
        if probe.rt is not None:
            probe.reset()
        assert _call_noalloc(x, y, m, d, lse) == rwo.OK
        assert rwo.get_status() == rwo.OK
        # (the peak, not the current figure: a garbage collection may free unrelated tensors meanwhile)
        assert torch.cuda.max_memory_allocated() <= before, "torch's allocator was used"
        if probe.rt is not None:
            assert probe.high() == 0, "the stream-ordered memory pool was used"
        yh = to_host(y)
        what = f"no-alloc {M}x{N} call {call}"
        # against the fp64 oracle
        y_ref, m_ref, d_ref, lse_ref = oracle.softmax_rows(x_host)
        check_y(yh, y_ref, dtype, what)
        check_rowsums(yh, dtype, None, what)
        check_state(m.cpu().numpy(), d.cpu().numpy(), lse.cpu().numpy(), m_ref, d_ref, lse_ref, what)
        del y_ref
        # against the regular split-row call (same kernel choice, scratch from the memory pool)
        m_r, d_r, lse_r = (torch.empty(M, device="cuda") for _ in range(3))
        y_r = rwo.softmax_rows_ex(x, m_out=m_r, d_out=d_r, lse_out=lse_r, variant=rwo.VARIANT_SPLITROW)
        assert rwo.get_status() == rwo.OK
        if probe.rt is not None:
            assert probe.high() > 0, "the pool probe does not see the regular call's scratch"
        yr = to_host(y_r)
        ref = (synth.bf16_to_f32(yr) if dtype == synth.BF16 else yr).astype(np.float64)
        check_y(yh, ref, dtype, what + " vs the regular call")
        check_state(m.cpu().numpy(), d.cpu().numpy(), lse.cpu().numpy(), m_r.cpu().numpy().astype(np.float64),
                    d_r.cpu().numpy().astype(np.float64), lse_r.cpu().numpy().astype(np.float64),
                    what + " vs the regular call")


def test_no_alloc_rejects_shapes_beyond_its_scratch():
    x = torch.zeros((4096, 1 << 18), device="cuda")  # 4096 rows x 19 clusters > 40960 slots
    y = torch.empty_like(x)
    m = d = lse = torch.empty(4096, device="cuda")
    assert _call_noalloc(x, y, m, d, lse) == rwo.ERR_UNSUPPORTED
    assert rwo.get_status() == rwo.OK
