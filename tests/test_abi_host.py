"""Host-side checks of the C ABI that need no GPU: the library loads, exports every call
include/spops_gb300.h declares, and rejects bad arguments before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "spops_gb300.h")


@pytest.fixture(scope="module")
def lib():
    from unstructured_sparse_linear_gb300 import _lib, build
    build.build()
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"SPOPS_API\s+[\w\s\*]+?\b(spops_\w+)\s*\(", text)


def test_header_declares_the_pages_operators():
    names = declared_functions()
    for op in ("spops_spmm", "spops_sddmm", "spops_csr_add", "spops_sort_rows", "spops_row_bins"):
        assert op in names


def test_every_declared_symbol_is_exported(lib):
    from unstructured_sparse_linear_gb300 import _lib
    names = declared_functions()
    assert names, "no declarations parsed"
    for n in names:
        assert hasattr(lib, n), n
        assert n in _lib.SIGNATURES, f"binding lacks a signature for {n}"
    assert set(_lib.SIGNATURES) == set(names)


def test_status_strings_and_version(lib):
    assert lib.spops_status_string(0) == b"SPOPS_OK"
    assert lib.spops_status_string(3) == b"SPOPS_ERR_WORKSPACE"
    assert lib.spops_status_string(99) == b"SPOPS_UNKNOWN_STATUS"
    assert b"sm_103a" in lib.spops_version()


def test_workspace_sizes_are_positive_and_monotone(lib):
    assert lib.spops_sort_rows_workspace_size(1000) >= 4 * 1000 * 4
    assert lib.spops_sort_rows_workspace_size(100000) > lib.spops_sort_rows_workspace_size(1000)
    assert lib.spops_spmm_workspace_size(4096, 4096, 2048, 167772, 1, 0) >= 16
    assert lib.spops_sddmm_workspace_size(4096, 4096, 2048, 167772, 1, 0, 1) >= 16
    assert lib.spops_plan_size(4096, 4096, 167772) >= 1024
    assert lib.spops_check_csr_workspace_size(64) >= 8


P = ctypes.c_void_p
FAKE = P(0x10000)  # never dereferenced: every call below fails validation first


def test_bad_arguments_rejected_on_host(lib):
    W = 1 << 30  # a workspace size large enough for every call below
    # dtype / itype / backend / path out of range
    assert lib.spops_spmm(FAKE, FAKE, FAKE, FAKE, 0, 7, 4, 4, 4, FAKE, 4, FAKE, 0, None, FAKE, W, None) == 1
    assert lib.spops_spmm(FAKE, FAKE, FAKE, FAKE, 5, 0, 4, 4, 4, FAKE, 4, FAKE, 0, None, FAKE, W, None) == 1
    assert lib.spops_spmm(FAKE, FAKE, FAKE, FAKE, 0, 0, 4, 4, 4, P(0x20000), 4, P(0x40000), 9, None, FAKE, W,
                          None) == 1
    assert lib.spops_sddmm(FAKE, FAKE, FAKE, 0, 0, 4, 4, 4, 4, FAKE, FAKE, FAKE, 9, None, FAKE, W, None) == 1
    # negative sizes
    assert lib.spops_csr_add(FAKE, FAKE, None, FAKE, 0, 0, -1, 4, 4, FAKE, FAKE, None) == 1
    # int16 cannot index 40000 rows
    assert lib.spops_spmm(FAKE, FAKE, FAKE, FAKE, 0, 0, 40000, 4, 4, FAKE, 4, FAKE, 0, None, FAKE, W, None) == 2
    assert b"int16" in lib.spops_last_error()
    # NULL row_offsets / misaligned values
    assert lib.spops_csr_add(FAKE, None, None, FAKE, 0, 0, 4, 4, 4, FAKE, FAKE, None) == 1
    assert lib.spops_csr_add(P(0x10001), FAKE, None, FAKE, 0, 0, 4, 4, 4, FAKE, FAKE, None) == 1
    # partial overlap of B and C in csr_add
    assert lib.spops_csr_add(FAKE, FAKE, None, FAKE, 0, 0, 4, 4, 4, P(0x20000), P(0x20004), None) == 1
    # SpMM output overlapping B
    assert lib.spops_spmm(FAKE, FAKE, FAKE, FAKE, 0, 0, 4, 4, 4, P(0x20000), 4, P(0x20010), 0, None, FAKE, W,
                          None) == 1
    # a plan that is not 1024-byte aligned
    assert lib.spops_spmm(FAKE, FAKE, FAKE, FAKE, 0, 0, 4, 4, 4, P(0x20000), 4, P(0x40000), 0, P(0x30010), FAKE, W,
                          None) == 1
    # workspace too small / missing; plan buffer too small
    assert lib.spops_spmm(FAKE, FAKE, FAKE, FAKE, 0, 0, 4, 4, 4, P(0x20000), 4, P(0x40000), 0, None, None, 0,
                          None) == 3
    assert lib.spops_sort_rows(FAKE, 10, 5, FAKE, 0, FAKE, 8, None) == 3
    assert lib.spops_plan_build(FAKE, FAKE, FAKE, 0, 10, 10, 5, P(0x40000), 64, None) == 3
    assert lib.spops_row_bins(FAKE, 10, 0, FAKE, None) == 1
    # the plan's row order: misaligned plan or output; no panels beyond 65536 columns
    assert lib.spops_plan_row_order(P(0x30010), 10, 10, 5, FAKE, None) == 1
    assert lib.spops_plan_row_order(P(0x40000), 10, 10, 5, P(0x10002), None) == 1
    assert lib.spops_plan_row_order(P(0x40000), 10, 70000, 5, FAKE, None) == 2
    assert lib.spops_get_device_error(None, None) == 1
    # the wait self-test: limits outside [1 us, 1 s], misaligned output
    assert lib.spops_selftest_wait_timeout(999, None, None) == 1
    assert lib.spops_selftest_wait_timeout(1_000_000_001, None, None) == 1
    assert lib.spops_selftest_wait_timeout(5_000_000, P(0x10004), None) == 1


def test_plan_size_grows_with_the_mask(lib):
    small = lib.spops_plan_size(4096, 4096, 167772)
    assert small > 0
    assert lib.spops_plan_size(8192, 4096, 167772) > small          # more panels
    assert lib.spops_plan_size(4096, 200000, 167772) < small        # no panels beyond 65536 columns
    assert lib.spops_spmm_workspace_size(4096, 4096, 2048, 167772, 1, 0) > small   # plan + images
    assert lib.spops_sddmm_workspace_size(4096, 4096, 2048, 167772, 1, 0, 1) >= small


def test_empty_problems_are_no_ops(lib):
    # m * n == 0 returns before any device work
    assert lib.spops_spmm(None, FAKE, None, None, 0, 0, 0, 4, 0, FAKE, 4, None, 0, None, None, 0, None) == 0
    assert lib.spops_csr_add(None, FAKE, None, None, 0, 0, 5, 0, 0, None, None, None) == 0
    assert lib.spops_sort_rows(FAKE, 0, 0, None, 0, None, 0, None) == 0


def test_widened_operators_reject_bad_arguments_on_host(lib):
    W = 1 << 30
    d = ctypes.c_double
    # csr_transpose: values without values_t; int16 for 40000 columns; workspace too small
    assert lib.spops_csr_transpose(FAKE, FAKE, FAKE, 0, 0, 4, 4, 4, FAKE, P(0x50000), None, None, FAKE, W, None) == 1
    assert lib.spops_csr_transpose(FAKE, FAKE, None, 0, 0, 4, 40000, 4, FAKE, P(0x50000), None, None, FAKE, W,
                                   None) == 2
    assert lib.spops_csr_transpose(FAKE, FAKE, None, 0, 0, 4, 4, 4, FAKE, P(0x50000), None, None, FAKE, 8, None) == 3
    # an output overlapping an input
    assert lib.spops_csr_transpose(FAKE, P(0x50000), None, 0, 0, 4, 4, 4, FAKE, P(0x50002), None, None, FAKE, W,
                                   None) == 1
    assert lib.spops_csr_transpose_workspace_size(1000) >= 4 * 1000 * 4
    # permute_values: bad dtype, negative nnz, output over the input
    assert lib.spops_csr_permute_values(FAKE, FAKE, 9, 4, P(0x60000), None) == 1
    assert lib.spops_csr_permute_values(FAKE, FAKE, 0, -1, P(0x60000), None) == 1
    assert lib.spops_csr_permute_values(P(0x60000), FAKE, 0, 4, P(0x60004), None) == 1
    # masked Adam: step 0, beta 1, negative lr, aliased state, grad dtype out of range
    adam = lambda *a: lib.spops_masked_adam(*a)  # noqa: E731
    args = (P(0x100000), P(0x200000), P(0x300000), P(0x400000), 0, 64)
    assert adam(*args, 0, d(1e-3), d(0.9), d(0.999), d(1e-8), 0, None) == 1
    assert adam(*args, 1, d(1e-3), d(1.0), d(0.999), d(1e-8), 0, None) == 1
    assert adam(*args, 1, d(-1.0), d(0.9), d(0.999), d(1e-8), 0, None) == 1
    assert adam(P(0x100000), P(0x100000), P(0x300000), P(0x400000), 0, 64, 1, d(1e-3), d(0.9), d(0.999), d(1e-8), 0,
                None) == 1
    assert adam(P(0x100000), P(0x200000), P(0x300000), P(0x400000), 7, 64, 1, d(1e-3), d(0.9), d(0.999), d(1e-8), 0,
                None) == 1
    assert adam(None, None, None, None, 0, 0, 1, d(1e-3), d(0.9), d(0.999), d(1e-8), 0, None) == 0  # nothing to do
    # masked Adam on a dense parameter: int16 indices for 40000 columns
    assert lib.spops_masked_adam_csr(P(0x100000), P(0x200000), P(0x300000), P(0x400000), 0, FAKE, FAKE, 0, 4, 40000,
                                     4, 1, d(1e-3), d(0.9), d(0.999), d(1e-8), 0, None) == 2
