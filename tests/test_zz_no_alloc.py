"""spops_sort_rows_static: the row permutation for callers that cannot allocate device
memory where they need it (a plugin whose host application owns all device memory, or a
loop that must not call cudaMalloc because it can synchronize the device). Its scratch is
a static device array inside the library. The test calls it through the C ABI, twice in a
row on different masks large enough to use that array, and checks each result against
spops_sort_rows (which takes a workspace); index outputs must match bit for bit. This file
is collected last."""
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
    """Both masks have more than 16384 rows, so both calls take the multi-CTA radix sort,
    whose passes run through the static array (the single-CTA sort of smaller masks keeps
    its keys in shared memory): an int16 RoSA-like clustered mask of 30000 rows, then an
    int32 Zipf-banded mask of 20000 rows, queued back to back on one stream before either
    result is read, so the second call reuses the array the first one left behind."""
    import unstructured_sparse_linear_gb300 as sp
    torch.cuda.set_device(0)
    cases = [
        (wl.clustered_mask(1, 30000, 30000, 0.0005), torch.int16),                    # int16 scatter
        (wl.zipf_band_mask(3, 20000, 20000, max_len=3000, band=2000), torch.int32),   # wide keys, many ties
    ]
    got, want = [], []
    for (ro_np, col_np), idx in cases:
        ro = torch.from_numpy(ro_np).cuda()
        assert ro.numel() - 1 > 16384
        nnz = int(col_np.size)
        got.append(_static_sort(lib, ro, nnz, idx))
    for (ro_np, col_np), idx in cases:
        want.append(sp.sort_rows(torch.from_numpy(ro_np).cuda(), nnz=int(col_np.size), index_dtype=idx))
    torch.cuda.synchronize()
    for g, w_, ((ro_np, _), _) in zip(got, want, cases):
        assert torch.equal(g, w_)
        assert np.array_equal(np.sort(g.cpu().numpy().astype(np.int64)), np.arange(ro_np.size - 1))


def test_static_scratch_rejects_more_rows_than_it_holds(lib):
    cap = lib.spops_sort_rows_static_max_rows()
    assert cap == 131072
    # the size check runs before any device work, so no buffers are needed
    assert lib.spops_sort_rows_static(ctypes.c_void_p(16), cap + 1, 10, ctypes.c_void_p(16), 1, None) == 2
    assert b"static scratch" in lib.spops_last_error()
