"""spops_sort_rows_static: the row permutation for callers that cannot allocate device
memory where they need it (a plugin whose host application owns all device memory, or a
loop that must not call cudaMalloc because it can synchronize the device). Its scratch is
a static device array inside the library. The test calls it through the C ABI, twice in a
row on different masks, and checks each result against spops_sort_rows (which takes a
workspace); index outputs must match bit for bit. This file is collected last."""
import ctypes

import numpy as np
import pytest
import torch

import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from unstructured_sparse_linear_gb300 import _lib, build
    build.build()
    return _lib.load()


def _static_sort(lib, ro: torch.Tensor, nnz: int, index_dtype) -> torch.Tensor:
    m = ro.numel() - 1
    out = torch.full((m,), -1, dtype=index_dtype, device=ro.device)
    it = 0 if index_dtype == torch.int16 else 1
    st = lib.spops_sort_rows_static(ctypes.c_void_p(ro.data_ptr()), m, nnz, ctypes.c_void_p(out.data_ptr()), it,
                                    ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, lib.spops_last_error()
    return out


def test_static_scratch_sort_matches_workspace_sort_twice_in_a_row(lib):
    import unstructured_sparse_linear_gb300 as sp
    torch.cuda.set_device(0)
    cases = [
        (wl.clustered_mask(1, 4096, 4096, 0.01), torch.int16),              # RoSA-adapter mask
        (wl.zipf_band_mask(3, 20000, 20000, max_len=3000, band=2000), torch.int32),  # wide keys, many ties
    ]
    for (ro_np, col_np), idx in cases:
        ro = torch.from_numpy(ro_np).cuda()
        nnz = int(col_np.size)
        got = _static_sort(lib, ro, nnz, idx)
        want = sp.sort_rows(ro, nnz=nnz, index_dtype=idx)
        torch.cuda.synchronize()
        assert torch.equal(got, want)
        assert np.array_equal(np.sort(got.cpu().numpy().astype(np.int64)), np.arange(ro.numel() - 1))


def test_static_scratch_rejects_more_rows_than_it_holds(lib):
    cap = lib.spops_sort_rows_static_max_rows()
    assert cap == 131072
    # the size check runs before any device work, so no buffers are needed
    assert lib.spops_sort_rows_static(ctypes.c_void_p(16), cap + 1, 10, ctypes.c_void_p(16), 1, None) == 2
    assert b"static scratch" in lib.spops_last_error()
