"""Failure detection on the GPU without a fault: every wait of the TMA and tensor-core
kernels on a copy or an MMA gives up after a time limit, records SPOPS_DEV_MBAR_TIMEOUT in
the device error word and lets its kernel return. The self-test call makes one such wait run
out (a barrier nothing arrives on, nothing in flight, a limit of a few milliseconds); the
test checks, through the C ABI, that the kernel came back, that the error word holds the
timeout code, that reading it clears it, and that a normal call afterwards still works."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import assert_close, to_gpu

pytestmark = pytest.mark.gpu

SPOPS_DEV_MBAR_TIMEOUT = 1


@pytest.fixture(scope="module")
def lib():
    from unstructured_sparse_linear_gb300 import _lib, build
    build.build()
    return _lib.load()


def _device_error(lib, stream) -> int:
    code = ctypes.c_int32(-1)
    assert lib.spops_get_device_error(stream, ctypes.byref(code)) == 0, lib.spops_last_error()
    return code.value


def test_bounded_wait_gives_up_and_the_context_stays_usable(lib):
    import unstructured_sparse_linear_gb300 as sp
    torch.cuda.set_device(0)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert _device_error(lib, stream) == 0  # nothing recorded before
    waited = torch.zeros(1, dtype=torch.int64, device="cuda")
    limit_ns = 5_000_000  # 5 ms
    for _ in range(2):  # twice: the word is cleared by the read in between
        assert lib.spops_selftest_wait_timeout(limit_ns, ctypes.c_void_p(waited.data_ptr()), stream) == 0
        assert _device_error(lib, stream) == SPOPS_DEV_MBAR_TIMEOUT
        w = int(waited.item())
        assert limit_ns <= w < 2_000_000_000, w  # it waited its limit, then returned
        assert _device_error(lib, stream) == 0   # read-and-clear
    # a following normal call still runs and is correct
    w = wl.generate(wl.spec("rosa", m=600, n=600, N=64, kd=64))
    g = to_gpu(w)
    C = sp.spmm(g["val"], g["ro"], g["row_idx"], g["col"], g["B"], w.m)
    torch.cuda.synchronize()
    assert_close(C, oracle.spmm(w.row_offsets.numpy(), w.col_idx.numpy(), w.values, w.B), w.dtype, "spmm after")
    assert _device_error(lib, stream) == 0
    assert np.isfinite(C.float().cpu().numpy()).all()


def test_bounded_wait_rejects_limits_out_of_range(lib):
    assert lib.spops_selftest_wait_timeout(10, None, None) == 1
    assert lib.spops_selftest_wait_timeout(5_000_000_000, None, None) == 1
    assert lib.spops_selftest_wait_timeout(5_000_000, ctypes.c_void_p(0x10004), None) == 1  # misaligned
