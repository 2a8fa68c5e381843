"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the same seeded
inputs. Every case compares every element, the five full-size configurations included: by the
stated relative Frobenius tolerance and by the element-wise bound of fp32 accumulation."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import (TOL, abs_of, as_f64, assert_bits_equal, assert_close, assert_elementwise, index_dtype,
                     spmm_terms, to_gpu)

pytestmark = pytest.mark.gpu

sp = pytest.importorskip("unstructured_sparse_linear_gb300")

# Scaled-down versions of the five workloads: several tiles and ragged tails everywhere.
SMALL = {
    "tiny": wl.spec("tiny"),
    "rosa_s": wl.spec("rosa", m=1000, n=1000, N=200, kd=200),
    "llama_s": wl.spec("llama_mlp", m=1100, n=512, N=520, kd=264),
    "zipf_s": wl.spec("zipf", m=4000, n=4000, N=36, mask_kw=(("max_len", 600), ("band", 700))),
    "butterfly_s": wl.spec("butterfly", m=1024, n=256, N=256, kd=136, mask_kw=(("block", 32),)),
    "rosa_i32": wl.spec("rosa", m=700, n=900, N=64, kd=72, mask_kw=(("row_frac", 0.3), ("col_frac", 0.3))),
    # fully dense 150 x 150 cluster: two dense panels (128 + 22 rows), ragged N and kd
    "rosa_dense": wl.spec("rosa", m=1500, n=1500, density=0.02, N=264, kd=136),
    # bf16, int32 indices, long K (split-K over 16 chunks of 64)
    "rosa_dense_i32": wl.spec("rosa", m=1500, n=1300, density=0.02, dtype="bf16", N=64, kd=1000),
    # 200 x 1500 cluster half full: |U| = 1500 panels, SpMM on tensor cores, SDDMM general
    "rosa_wide": wl.spec("rosa", m=2000, n=3000, density=0.025, N=136, kd=72,
                         mask_kw=(("row_frac", 0.1), ("col_frac", 0.5))),
    # the 384 -> 1536 pixelfly layer (48 x 48 blocks, not a multiple of the 64-wide K chunk),
    # fewer tokens
    "fly_s": wl.spec("fly_small_1", N=200, kd=136),
}
INT32_CASES = ("rosa_i32", "rosa_dense_i32")


@pytest.fixture(scope="module")
def small_cases():
    return {k: wl.generate(s) for k, s in SMALL.items()}


def run_all_ops(w, g, backend="structure_aware"):
    """backend "structure_aware" also lets SpMM take its dense-panel path; "general" runs
    both on the general row kernels."""
    out = {}
    if w.B is not None:
        path = "auto" if backend == "structure_aware" else "general"
        out["spmm"] = sp.spmm(g["val"], g["ro"], g["row_idx"], g["col"], g["B"], w.m, path=path)
    if w.A is not None:
        out["sddmm"] = sp.sddmm(g["ro"], g["row_idx"], g["col"], g["A"], g["BT"], backend=backend)
    if w.W is not None:
        out["csr_add"] = sp.csr_add(g["val"], g["ro"], g["row_idx"], g["col"], g["W"])
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("backend", ["structure_aware", "general"])
def test_small_all_elements(small_cases, name, backend):
    w = small_cases[name]
    idx = torch.int32 if name in INT32_CASES else None
    g = to_gpu(w, idx_dtype=idx)
    out = run_all_ops(w, g, backend)
    ro, col = w.row_offsets.numpy(), w.col_idx.numpy()
    if "spmm" in out:
        want = oracle.spmm(ro, col, w.values, w.B)
        assert_close(out["spmm"], want, w.dtype, f"{name} spmm")
        assert_elementwise(out["spmm"], want, oracle.spmm(ro, col, abs_of(w.values), abs_of(w.B)), spmm_terms(ro),
                           w.dtype, f"{name} spmm")
    if "sddmm" in out:
        want = oracle.sddmm(ro, col, w.A, w.BT)
        assert_close(out["sddmm"], want, w.dtype, f"{name} sddmm {backend}")
        assert_elementwise(out["sddmm"], want, oracle.sddmm(ro, col, abs_of(w.A), abs_of(w.BT)), w.A.shape[1],
                           w.dtype, f"{name} sddmm {backend}")
    if "csr_add" in out:
        assert_bits_equal(out["csr_add"], oracle.csr_add(ro, col, w.values, w.W), w.dtype, f"{name} csr_add")


@pytest.mark.parametrize("name", ["tiny", "rosa_s", "llama_s", "butterfly_s", "rosa_dense"])
def test_integer_valued_inputs_are_exact(name):
    """Small-integer inputs make every product and partial sum exact in fp32, so the GPU
    must equal the oracle bit for bit whatever its summation order."""
    s = SMALL[name]
    if s.kd:
        s = dataclasses.replace(s, kd=min(s.kd, 64))
    w = wl.generate(s, integer_valued=True)
    g = to_gpu(w)
    ro, col = w.row_offsets.numpy(), w.col_idx.numpy()
    for backend in ("structure_aware", "general"):
        out = run_all_ops(w, g, backend)
        if "spmm" in out:
            assert_bits_equal(out["spmm"], oracle.spmm(ro, col, w.values, w.B), w.dtype, f"{name} spmm")
        if "sddmm" in out:
            assert_bits_equal(out["sddmm"], oracle.sddmm(ro, col, w.A, w.BT), w.dtype, f"{name} sddmm {backend}")


def test_row_idx_any_permutation_gives_same_result(small_cases):
    """No row of this case reaches a long-row bin, so every row is summed in the same order
    whatever its position, and the results must be bitwise identical."""
    w = small_cases["llama_s"]
    assert np.diff(w.row_offsets.numpy()).max() < min(sp.SDDMM_LONG_ROW, sp.SPMM_LONG_ROW)
    g = to_gpu(w)
    ref = run_all_ops(w, g)
    perm = wl.random_permutation(5, w.m)
    g2 = to_gpu(w, row_idx=perm)
    out = run_all_ops(w, g2)
    for k in ref:
        assert torch.equal(ref[k].view(torch.int16), out[k].view(torch.int16)), k


@pytest.mark.parametrize("name", ["rosa_s", "rosa_dense", "rosa_wide"])
def test_row_idx_swaps_across_the_bins(small_cases, name):
    """A row order that is sorted except for swaps across the bin boundaries: the longest row
    goes to the last position (past the count of non-empty rows, where empty rows are
    expected) and an empty row to the first, and a non-empty row of a dense panel trades
    places with an empty row of a later panel. Every row must still be computed (or zeroed)
    exactly once, on the panel or the general path."""
    w = small_cases[name]
    ro = w.row_offsets.numpy()
    order = oracle.sort_rows(ro).copy()
    lens = np.diff(ro)[order]
    empty = np.flatnonzero(lens == 0)
    assert empty.size >= 2 and lens[0] > 0
    order[[0, -1]] = order[[-1, 0]]
    j = int(empty[empty > 256][0]) if (empty > 256).any() else int(empty[-2])
    order[[5, j]] = order[[j, 5]]
    g = to_gpu(w, row_idx=torch.from_numpy(order))
    out = run_all_ops(w, g)
    assert_close(out["spmm"], oracle.spmm(ro, w.col_idx.numpy(), w.values, w.B), w.dtype, f"{name} spmm")
    assert_close(out["sddmm"], oracle.sddmm(ro, w.col_idx.numpy(), w.A, w.BT), w.dtype, f"{name} sddmm")


def test_repeated_calls_are_bitwise_deterministic(small_cases):
    w = small_cases["rosa_s"]
    g = to_gpu(w)
    a = run_all_ops(w, g)
    b = run_all_ops(w, g)
    for k in a:
        assert torch.equal(a[k].view(torch.int16), b[k].view(torch.int16)), k


def test_release_streams_then_calls_recreate_them(small_cases):
    """The side streams (the library's persistent host-side resources) can be released at
    any point between calls; the next calls create them again and give identical results."""
    w = small_cases["rosa_dense"]
    g = to_gpu(w)
    a = run_all_ops(w, g)
    sp.release_streams()
    sp.release_streams()  # nothing left to release: still fine
    b = run_all_ops(w, g)
    for k in a:
        assert torch.equal(a[k].view(torch.int16), b[k].view(torch.int16)), k


# ------------------------------------------------------------------ row scheduler


@pytest.mark.parametrize("name", list(SMALL))
def test_sort_rows_and_bins_bit_exact(small_cases, name):
    w = small_cases[name]
    ro = w.row_offsets.numpy()
    dev_ro = w.row_offsets.cuda()
    for itd in ([torch.int16, torch.int32] if w.m <= 32768 else [torch.int32]):
        got = sp.sort_rows(dev_ro, index_dtype=itd).cpu().numpy().astype(np.int64)
        assert np.array_equal(got, oracle.sort_rows(ro))
    for t in (1, 64, 256):
        assert np.array_equal(sp.row_bins(dev_ro, t).cpu().numpy(), oracle.row_bins(ro, t))


def test_sort_rows_many_ties_and_wide_keys():
    rng = np.random.default_rng(3)
    m = 70000
    lens = rng.integers(0, 3, size=m)
    lens[rng.choice(m, 20, replace=False)] = rng.integers(1000, 300000, size=20)  # keys over 3 radix digits
    ro = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    got = sp.sort_rows(torch.from_numpy(ro).cuda(), index_dtype=torch.int32).cpu().numpy()
    assert np.array_equal(got, oracle.sort_rows(ro))


@pytest.mark.parametrize("m", [1, 2, 31, 100, 1024, 1025])
def test_sort_rows_small_masks(m):
    """Up to 1024 rows the sort ranks each row's (nnz descending, row id) key against all the
    others; 1025 takes the one-CTA radix sort. Ties and empty rows included."""
    rng = np.random.default_rng(m + 7)
    lens = rng.integers(0, 40, size=m)
    lens[rng.random(m) < 0.3] = 5  # runs of ties
    lens[rng.random(m) < 0.1] = 0
    ro = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    for itd in (torch.int16, torch.int32):
        got = sp.sort_rows(torch.from_numpy(ro).cuda(), index_dtype=itd).cpu().numpy().astype(np.int64)
        assert np.array_equal(got, oracle.sort_rows(ro))


@pytest.mark.parametrize("m", [16384, 16385])
def test_sort_rows_many_distinct_lengths(m):
    """Row lengths spread over 0..5999 (up to 32 distinct radix digits in a warp): the one-CTA
    sort at m = 16384 takes two passes (9 + 4 bits), the grid-wide sort at m = 16385 three of 8
    bits; both must give the oracle's order (nnz descending, ties by ascending row id)."""
    rng = np.random.default_rng(m)
    lens = rng.integers(0, 6000, size=m)
    ties = rng.random(m) < 0.2  # a fifth of the rows share three lengths: long runs of ties
    lens[ties] = rng.integers(0, 3, size=int(ties.sum()))
    ro = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    for itd in ([torch.int16, torch.int32] if m <= 32768 else [torch.int32]):
        got = sp.sort_rows(torch.from_numpy(ro).cuda(), index_dtype=itd).cpu().numpy().astype(np.int64)
        assert np.array_equal(got, oracle.sort_rows(ro))


# ------------------------------------------------------------------ edge cases


def _csr(m, n, rows, cols, dtype, seed=0):
    ro, col = wl.csr_from_coords(np.asarray(rows), np.asarray(cols), m)
    vals = wl.normal(seed, 1, (col.size,), 1.0, dtype)
    return ro, col, vals


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_empty_matrix(dtype):
    m, n, N = 37, 29, 24
    ro = np.zeros(m + 1, dtype=np.int32)
    col = np.zeros(0, dtype=np.int32)
    tdt = wl.DTYPES[dtype]
    B = torch.randn(n, N).to(tdt).cuda()
    W = torch.randn(m, n).to(tdt).cuda()
    dro, dcol = torch.from_numpy(ro).cuda(), torch.from_numpy(col).to(torch.int16).cuda()
    ridx = torch.arange(m, dtype=torch.int16).cuda()
    vals = torch.zeros(0, dtype=tdt).cuda()
    C = sp.spmm(vals, dro, ridx, dcol, B, m)
    assert torch.count_nonzero(C) == 0
    assert torch.equal(sp.csr_add(vals, dro, ridx, dcol, W), W)
    A = torch.randn(m, 16).to(tdt).cuda()
    BT = torch.randn(n, 16).to(tdt).cuda()
    assert sp.sddmm(dro, ridx, dcol, A, BT).numel() == 0


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("N", [1, 7, 8, 33, 264])
def test_ragged_and_unaligned_widths(dtype, N):
    rng = np.random.default_rng(N)
    m, n = 301, 257
    mask = rng.random((m, n)) < 0.05
    mask[5] = False
    mask[7, :] = True  # one dense row (257 entries: a long row for SpMM)
    ro, col, vals = _csr(m, n, *np.nonzero(mask), dtype)
    tdt = wl.DTYPES[dtype]
    B = wl.normal(9, 2, (n, N), 1.0, dtype)
    A = wl.normal(9, 3, (m, N), 1.0, dtype)
    BT = wl.normal(9, 4, (n, N), 1.0, dtype)
    W = wl.normal(9, 5, (m, n), 1.0, dtype)
    dro = torch.from_numpy(ro).cuda()
    dcol = torch.from_numpy(col).to(torch.int16).cuda()
    ridx = torch.from_numpy(oracle.sort_rows(ro)).to(torch.int16).cuda()
    dv = vals.cuda()
    C = sp.spmm(dv, dro, ridx, dcol, B.cuda(), m)
    assert_close(C, oracle.spmm(ro, col, vals, B), dtype, "spmm")
    for be in ("structure_aware", "general"):
        o = sp.sddmm(dro, ridx, dcol, A.cuda(), BT.cuda(), backend=be)
        assert_close(o, oracle.sddmm(ro, col, A, BT), dtype, f"sddmm {be}")
    assert_bits_equal(sp.csr_add(dv, dro, ridx, dcol, W.cuda()), oracle.csr_add(ro, col, vals, W), dtype, "csr_add")


@pytest.mark.parametrize("m", [400, 800, 1500, 24000, 50000])
def test_sddmm_row_teams_and_alternating_deal(m):
    """The general SDDMM deals short rows in bands whose direction alternates, to teams of 8,
    4 or 2 warp groups where rows are fewer than groups (these m give each size on a 152-SM
    part, then one group per row), the members of a team splitting each row's entries; long
    rows go a CTA each, also in alternating bands (over 500 of them at m = 50000: two bands).
    Heavy-tailed lengths, empty rows, small-integer operands: every dot product is exact, so
    the result must equal the oracle bit for bit, whatever team computed an entry."""
    rng = np.random.default_rng(m)
    n, kd = 2048, 256
    lens = np.minimum(rng.zipf(1.6, size=m), 63)
    lens[rng.random(m) < 0.1] = 0
    longs = rng.choice(m, size=max(8, m // 90), replace=False)
    lens[longs] = rng.integers(64, 700, size=longs.size)
    rows = np.repeat(np.arange(m), lens)
    start = rng.integers(0, n, size=m)
    cols = (np.repeat(start, lens) + (np.arange(rows.size) - np.repeat(np.cumsum(lens) - lens, lens)) * 31) % n
    ro, col = wl.csr_from_coords(rows, cols, m)
    assert np.array_equal(np.diff(ro), lens)
    A = wl.integers(m, 3, (m, kd), -2, 2, "f32")
    BT = wl.integers(m, 4, (n, kd), -2, 2, "f32")
    dro, dcol = torch.from_numpy(ro).cuda(), torch.from_numpy(col).cuda()
    ridx = torch.from_numpy(oracle.sort_rows(ro)).to(torch.int32).cuda()
    want = oracle.sddmm(ro, col, A, BT)
    for be in ("general", "structure_aware"):
        got = sp.sddmm(dro, ridx, dcol, A.cuda(), BT.cuda(), backend=be)
        assert_bits_equal(got, want, "f32", f"sddmm {be} m={m}")


def test_unaligned_pointers_take_the_plain_path():
    """Operands that start 2 bytes into an allocation (not 16-byte aligned)."""
    m, n, N = 64, 80, 40
    rng = np.random.default_rng(1)
    ro, col, vals = _csr(m, n, *np.nonzero(rng.random((m, n)) < 0.1), "f16")
    B = wl.normal(1, 2, (n, N), 1.0, "f16")
    W = wl.normal(1, 3, (m, n), 1.0, "f16")
    Bbuf = torch.empty(n * N + 1, dtype=torch.float16, device="cuda")
    Bbuf[1:] = B.cuda().view(-1)
    Bu = Bbuf[1:].view(n, N)
    Wbuf = torch.empty(m * n + 1, dtype=torch.float16, device="cuda")
    Wbuf[1:] = W.cuda().view(-1)
    Wu = Wbuf[1:].view(m, n)
    Cbuf = torch.empty(m * N + 1, dtype=torch.float16, device="cuda")
    dro, dcol = torch.from_numpy(ro).cuda(), torch.from_numpy(col).to(torch.int16).cuda()
    ridx = torch.from_numpy(oracle.sort_rows(ro)).to(torch.int16).cuda()
    C = sp.spmm(vals.cuda(), dro, ridx, dcol, Bu, m, out=Cbuf[1:].view(m, N))
    assert_close(C, oracle.spmm(ro, col, vals, B), "f16", "spmm unaligned")
    assert_bits_equal(sp.csr_add(vals.cuda(), dro, ridx, dcol, Wu), oracle.csr_add(ro, col, vals, W), "f16",
                      "csr_add unaligned")


@pytest.mark.parametrize("m,n,density,dtype,itype", [(64, 20000, 0.3, "f32", "int16"),
                                                      (64, 20000, 1.0, "f32", "int32"),
                                                      (3, 300000, 0.05, "bf16", "int32"),
                                                      (40, 9000, 0.6, "f16", "int16")])
def test_csr_add_wide_rows(m, n, density, dtype, itype):
    """Rows wider than a 16 KB tile: each tile finds its first and last entry in the edge
    rows by searching the sorted columns. Rows of every width from empty to full."""
    rng = np.random.default_rng(m + n)
    mask = rng.random((m, n)) < density
    mask[1] = False
    mask[2 % m, :] = True
    mask[0, : n // 3] = False
    ro, col, vals = _csr(m, n, *np.nonzero(mask), dtype, seed=4)
    W = wl.normal(4, 2, (m, n), 1.0, dtype)
    idt = torch.int16 if itype == "int16" else torch.int32
    dro, dcol = torch.from_numpy(ro).cuda(), torch.from_numpy(col).to(idt).cuda()
    ridx = torch.from_numpy(oracle.sort_rows(ro)).to(idt).cuda()
    got = sp.csr_add(vals.cuda(), dro, ridx, dcol, W.cuda())
    assert_bits_equal(got, oracle.csr_add(ro, col, vals, W), dtype, f"csr_add {m}x{n}")


def test_csr_add_in_place():
    w = wl.generate(SMALL["llama_s"])
    g = to_gpu(w)
    want = oracle.csr_add(w.row_offsets.numpy(), w.col_idx.numpy(), w.values, w.W)
    Wd = g["W"].clone()
    out = sp.csr_add(g["val"], g["ro"], g["row_idx"], g["col"], Wd, out=Wd)
    assert out.data_ptr() == Wd.data_ptr()
    assert_bits_equal(Wd, want, "bf16", "csr_add in place")


def test_single_long_row_and_int16_edge_columns():
    m, n, N = 3, 32768, 16
    cols = np.concatenate([np.arange(0, 32768, 8), [32767]])
    cols = np.unique(cols)
    rows = np.zeros_like(cols)
    rows = np.concatenate([rows, [2]])
    cols = np.concatenate([cols, [32767]])
    ro, col, vals = _csr(m, n, rows, cols, "f32")
    B = wl.normal(2, 2, (n, N), 1.0, "f32")
    A = wl.normal(2, 3, (m, N), 1.0, "f32")
    BT = wl.normal(2, 4, (n, N), 1.0, "f32")
    dro = torch.from_numpy(ro).cuda()
    dcol = torch.from_numpy(col.astype(np.int16)).cuda()
    ridx = torch.from_numpy(oracle.sort_rows(ro)).to(torch.int16).cuda()
    C = sp.spmm(vals.cuda(), dro, ridx, dcol, B.cuda(), m)
    assert_close(C, oracle.spmm(ro, col, vals, B), "f32", "spmm long row")
    for be in ("structure_aware", "general"):
        assert_close(sp.sddmm(dro, ridx, dcol, A.cuda(), BT.cuda(), backend=be), oracle.sddmm(ro, col, A, BT),
                     "f32", f"sddmm long row {be}")


def test_check_csr_accepts_valid_and_flags_invalid():
    w = wl.generate(SMALL["rosa_s"])
    g = to_gpu(w)
    sp.check_csr(g["ro"], g["col"], g["row_idx"], w.n)
    bad_col = g["col"].clone()
    bad_col[10] = w.n + 3  # out of range: the check reads it, never indexes with it
    with pytest.raises(sp.SpopsError):
        sp.check_csr(g["ro"], bad_col, g["row_idx"], w.n)
    dup = g["row_idx"].clone()
    dup[1] = dup[0]
    with pytest.raises(sp.SpopsError):
        sp.check_csr(g["ro"], g["col"], dup, w.n)
    sp.check_csr(g["ro"], g["col"], g["row_idx"], w.n)  # the error word was cleared


# ------------------------------------------------------------------ full-size workloads


@pytest.mark.slow
@pytest.mark.parametrize("name", wl.CONFIG_ORDER)
def test_full_size_every_element(name):
    """Each of the five configurations at full size, every output element: SpMM on the
    tensor-core path and on the general path, SDDMM on both backends, each against the
    oracle by the stated relative Frobenius tolerance and by the element-wise bound of fp32
    accumulation (the oracle run on |values| and |operands| gives sum |a b| per element);
    csr_add and sort_rows bit for bit."""
    w = wl.generate(name)
    g = to_gpu(w)
    ro, col = w.row_offsets.numpy(), w.col_idx.numpy()
    assert np.array_equal(sp.sort_rows(g["ro"], index_dtype=g["row_idx"].dtype).cpu().numpy().astype(np.int64),
                          oracle.sort_rows(ro))
    if w.B is not None:
        want = oracle.spmm(ro, col, w.values, w.B)
        absdot = oracle.spmm(ro, col, abs_of(w.values), abs_of(w.B))
        terms = spmm_terms(ro)
        for path in ("auto", "general"):
            C = sp.spmm(g["val"], g["ro"], g["row_idx"], g["col"], g["B"], w.m, path=path)
            torch.cuda.synchronize()
            assert_close(C, want, w.dtype, f"{name} spmm {path}")
            assert_elementwise(C, want, absdot, terms, w.dtype, f"{name} spmm {path}")
            del C
        del want, absdot
    if w.A is not None:
        want = oracle.sddmm(ro, col, w.A, w.BT)
        absdot = oracle.sddmm(ro, col, abs_of(w.A), abs_of(w.BT))
        for backend in ("structure_aware", "general"):
            out = sp.sddmm(g["ro"], g["row_idx"], g["col"], g["A"], g["BT"], backend=backend)
            torch.cuda.synchronize()
            assert_close(out, want, w.dtype, f"{name} sddmm {backend}")
            assert_elementwise(out, want, absdot, w.A.shape[1], w.dtype, f"{name} sddmm {backend}")
        del want, absdot
    if w.W is not None:
        D = sp.csr_add(g["val"], g["ro"], g["row_idx"], g["col"], g["W"])
        torch.cuda.synchronize()
        assert_bits_equal(D, oracle.csr_add(ro, col, w.values, w.W), w.dtype, f"{name} csr_add")


@pytest.mark.parametrize("case", ["butterfly", "clustered"])
def test_spmm_many_units_pipeline_exact(case):
    """More units (dense panels x column tiles) than four per SM, so SpMM takes the
    warp-specialized tensor-core pipeline: a butterfly mask (64 dense panels whose U lists
    are runs of 64 consecutive columns, loaded as tiles) and a clustered mask (random U
    columns, gathered row by row); 17 or 9 column tiles, the last one 8 columns wide.
    Small-integer inputs make every sum exact, so the result must equal the general row
    kernel and the oracle bit for bit on every element."""
    if case == "butterfly":
        s = wl.spec("butterfly", N=2056, kd=64)
    else:
        s = wl.spec("rosa", m=16384, n=4096, N=1032, kd=64)
    w = wl.generate(s, integer_valued=True)
    g = to_gpu(w)
    plan = sp.plan_build(g["ro"], g["row_idx"], g["col"], w.n)
    st = plan.stats()
    assert st["spmm_panels"] == st["panels"] == 64 if case == "butterfly" else st["spmm_panels"] >= 10
    C = sp.spmm(g["val"], g["ro"], g["row_idx"], g["col"], g["B"], w.m, plan=plan)
    ref = sp.spmm(g["val"], g["ro"], g["row_idx"], g["col"], g["B"], w.m, path="general")
    torch.cuda.synchronize()
    assert torch.equal(C.view(torch.int16), ref.view(torch.int16))
    ro, col = w.row_offsets.numpy(), w.col_idx.numpy()
    assert_bits_equal(C, oracle.spmm(ro, col, w.values, w.B), w.dtype, f"{case} many-units spmm")


def test_spmm_direct_values_gate_on_permuted_butterfly():
    """Every row of the butterfly mask has the same length, and after the plan's row order its
    panels are full, so the SpMM pipeline reads their A chunks straight from the CSR values,
    but only when a panel's rows are two runs of 64 consecutive rows. Shuffling the rows in
    blocks of 32 keeps runs long enough for the row order, so the panels stay full and dense,
    but breaks the 64-row runs: the images are built as usual. Exact small-integer sums on
    both masks, every element against the general kernel and the oracle."""
    s = wl.spec("butterfly", N=2056, kd=64)
    w = wl.generate(s, integer_valued=True)
    ro, col = w.row_offsets.numpy(), w.col_idx.numpy()
    rng = np.random.default_rng(11)
    blocks = rng.permutation(w.m // 32)
    perm = blocks[np.arange(w.m) // 32] * 32 + np.arange(w.m) % 32  # old row i becomes row perm[i]
    rows = np.repeat(np.arange(w.m), np.diff(ro))
    ro2, col2 = wl.csr_from_coords(perm[rows], col, w.m)
    order = np.lexsort((col, perm[rows]))
    vals2 = w.values[torch.from_numpy(order)]
    for r_o, c_o, v_o, what in ((ro, col, w.values, "butterfly"), (ro2, col2, vals2, "permuted butterfly")):
        dro = torch.from_numpy(np.asarray(r_o, dtype=np.int32)).cuda()
        dcol = torch.from_numpy(np.asarray(c_o)).to(torch.int16).cuda()
        ridx = torch.from_numpy(oracle.sort_rows(r_o)).to(torch.int16).cuda()
        plan = sp.plan_build(dro, ridx, dcol, w.n)
        assert plan.stats()["spmm_panels"] == 64, what
        C = sp.spmm(v_o.cuda(), dro, ridx, dcol, w.B.cuda(), w.m, plan=plan)
        ref = sp.spmm(v_o.cuda(), dro, ridx, dcol, w.B.cuda(), w.m, path="general")
        torch.cuda.synchronize()
        assert torch.equal(C.view(torch.int16), ref.view(torch.int16)), what
        assert_bits_equal(C, oracle.spmm(r_o, c_o, v_o, w.B), w.dtype, what)


def test_spmm_direct_values_with_a_partial_last_chunk():
    """Rows of 200 entries (a multiple of 8, not of 64) in 64-row groups that share one run of
    200 consecutive columns: the SpMM pipeline reads the A chunks straight from the values, the
    last chunk's box reaching past the 200 columns (filled with zeros), and gathers the last
    chunk's 8 B rows (the first three are 64-row tiles). Exact small-integer sums."""
    m, n, L, N = 8192, 2048, 200, 2056
    rng = np.random.default_rng(13)
    g = np.arange(m) // 64
    starts = (g % 8) * 240
    rows = np.repeat(np.arange(m), L)
    cols = (starts[:, None] + np.arange(L)[None, :]).ravel()
    ro, col = wl.csr_from_coords(rows, cols, m)
    vals = torch.from_numpy(rng.integers(-3, 4, size=col.size).astype(np.float32)).to(torch.bfloat16)
    B = torch.from_numpy(rng.integers(-3, 4, size=(n, N)).astype(np.float32)).to(torch.bfloat16)
    dro = torch.from_numpy(ro).cuda()
    dcol = torch.from_numpy(col).to(torch.int16).cuda()
    ridx = torch.from_numpy(oracle.sort_rows(ro)).to(torch.int16).cuda()
    plan = sp.plan_build(dro, ridx, dcol, n)
    assert plan.stats()["spmm_panels"] == 64
    C = sp.spmm(vals.cuda(), dro, ridx, dcol, B.cuda(), m, plan=plan)
    ref = sp.spmm(vals.cuda(), dro, ridx, dcol, B.cuda(), m, path="general")
    torch.cuda.synchronize()
    assert torch.equal(C.view(torch.int16), ref.view(torch.int16))
    assert_bits_equal(C, oracle.spmm(ro, col, vals, B), "bf16", "direct values, partial chunk")


@pytest.mark.parametrize("L", [100, 200])
def test_direct_panels_derive_their_positions(L):
    """Rows of L entries in 64-row groups that share one run of L consecutive columns: every
    panel is direct (each row holds all of U in order), so the plan skips their per-entry U
    positions and tile tables and the kernels derive them from the row id and |U|. L = 100 is
    not a multiple of 8, so SpMM densifies these panels (identity positions) instead of loading
    the values by boxes; SDDMM's last tile is partial in both cases (100 and 72 columns).
    Exact small-integer sums, bit for bit against the oracle and the general path."""
    m, n, N, kd = 8192, 2048, 264, 136
    rng = np.random.default_rng(L)
    g = np.arange(m) // 64
    starts = (g % 8) * 240
    rows = np.repeat(np.arange(m), L)
    cols = (starts[:, None] + np.arange(L)[None, :]).ravel()
    ro, col = wl.csr_from_coords(rows, cols, m)
    vals = wl.integers(L, 1, (col.size,), -3, 3, "bf16")
    B = wl.integers(L, 2, (n, N), -3, 3, "bf16")
    A = wl.integers(L, 3, (m, kd), -2, 2, "bf16")
    BT = wl.integers(L, 4, (n, kd), -2, 2, "bf16")
    dro = torch.from_numpy(ro).cuda()
    dcol = torch.from_numpy(col).to(torch.int16).cuda()
    ridx = torch.from_numpy(oracle.sort_rows(ro)).to(torch.int16).cuda()
    plan = sp.plan_build(dro, ridx, dcol, n)
    st = plan.stats()
    assert st["spmm_panels"] == 64 and st["dense_panels"] == 64
    C = sp.spmm(vals.cuda(), dro, ridx, dcol, B.cuda(), m, plan=plan)
    assert_bits_equal(C, oracle.spmm(ro, col, vals, B), "bf16", f"spmm direct L={L}")
    out = sp.sddmm(dro, ridx, dcol, A.cuda(), BT.cuda(), plan=plan)
    ref = sp.sddmm(dro, ridx, dcol, A.cuda(), BT.cuda(), backend="general")
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert_bits_equal(out, oracle.sddmm(ro, col, A, BT), "bf16", f"sddmm direct L={L}")


def _mixed_panels(seed=5):
    """A 16384 x 4096 mask whose panels alternate between the SpMM pipeline's kinds, in
    row_idx order (rows by nnz): 400 of 1200 pool columns (|U| = 1200, gathered, streamed
    image), 64-row block-rows of four 64-column blocks (|U| = 256, tiles, resident image),
    180 of 600 (|U| = 600, gathered, streamed) and 150 of 200 (|U| = 200, gathered, resident)."""
    rng = np.random.default_rng(seed)
    n = 4096
    rows, cols = [], []
    for br in range(64):  # rows 0 .. 4095: block-rows
        cs = np.concatenate([np.arange(b * 64, b * 64 + 64) for b in ((br % 16) * 4 + np.arange(4))])
        rows.append(np.repeat(np.arange(br * 64, br * 64 + 64), cs.size))
        cols.append(np.tile(cs, 64))
    for base, per, pool_n in ((4096, 400, 1200), (8192, 180, 600), (12288, 150, 200)):
        pool = rng.choice(n, pool_n, replace=False)
        pick = np.argsort(rng.random((4096, pool_n)), axis=1)[:, :per]
        rows.append(np.repeat(np.arange(base, base + 4096), per))
        cols.append(pool[pick].ravel())
    ro, col = wl.csr_from_coords(np.concatenate(rows), np.concatenate(cols), 16384)
    vals = torch.from_numpy(rng.integers(-3, 4, size=col.size).astype(np.float32)).to(torch.bfloat16)
    B = torch.from_numpy(rng.integers(-3, 4, size=(n, 2056)).astype(np.float32)).to(torch.bfloat16)
    return ro, col, vals, B


def test_spmm_mixed_panels_pipeline_exact():
    """The warp-specialized SpMM pipeline across panel changes between resident images
    (|U| <= 256, loaded once per run of units) and streamed ones, on tile and gather paths:
    exact small-integer sums, so every element equals the general kernel and the oracle."""
    ro, col, vals, B = _mixed_panels()
    m = len(ro) - 1
    dro = torch.from_numpy(ro).cuda()
    dcol = torch.from_numpy(col).to(torch.int16).cuda()
    ridx = torch.from_numpy(oracle.sort_rows(ro)).to(torch.int16).cuda()
    plan = sp.plan_build(dro, ridx, dcol, B.shape[0])
    st = plan.stats()
    assert st["spmm_panels"] == st["panels"] == 128, st
    C = sp.spmm(vals.cuda(), dro, ridx, dcol, B.cuda(), m, plan=plan)
    ref = sp.spmm(vals.cuda(), dro, ridx, dcol, B.cuda(), m, path="general")
    torch.cuda.synchronize()
    assert torch.equal(C.view(torch.int16), ref.view(torch.int16))
    assert_bits_equal(C, oracle.spmm(ro, col, vals, B), "bf16", "mixed panels spmm")


@pytest.mark.parametrize("case", ["butterfly", "clustered"])
def test_sddmm_many_tiles_pipeline_exact(case):
    """At least two SDDMM tiles per SM are possible, so the structure-aware SDDMM runs its
    tiles without a K split, eight warps per CTA: a butterfly mask (192 tiles) and a
    clustered mask with random rows and columns (52 tiles); kd = 136 leaves a partial last
    K chunk. Small-integer inputs make every dot product exact, so every entry must equal
    the general kernel and the oracle bit for bit."""
    if case == "butterfly":
        s = wl.spec("butterfly", N=64, kd=136)
    else:
        s = wl.spec("rosa", m=16384, n=4096, N=64, kd=136)
    w = wl.generate(s, integer_valued=True)
    g = to_gpu(w)
    plan = sp.plan_build(g["ro"], g["row_idx"], g["col"], w.n)
    assert plan.stats()["sddmm_tiles"] >= 40
    got = sp.sddmm(g["ro"], g["row_idx"], g["col"], g["A"], g["BT"], plan=plan)
    ref = sp.sddmm(g["ro"], g["row_idx"], g["col"], g["A"], g["BT"], backend="general")
    torch.cuda.synchronize()
    assert torch.equal(got.view(torch.int16), ref.view(torch.int16))
    ro, col = w.row_offsets.numpy(), w.col_idx.numpy()
    assert_bits_equal(got, oracle.sddmm(ro, col, w.A, w.BT), w.dtype, f"{case} many-tiles sddmm")


# ------------------------------------------------------------------ mask plan


def _mix_col(c):
    """The plan's hash of one column index (32-bit arithmetic)."""
    h = (np.asarray(c, dtype=np.uint64) * np.uint64(0x9E3779B1)) & np.uint64(0xFFFFFFFF)
    h ^= h >> np.uint64(15)
    h = (h * np.uint64(0x85EBCA77)) & np.uint64(0xFFFFFFFF)
    h ^= h >> np.uint64(13)
    return h


def plan_order(ro, col, row_idx, n):
    """The plan's row order restated on the host: for masks of at most 16384 rows (with column
    panels, n <= 65536), row_idx stably sorted by (nnz descending, counts of 65535 and more
    tied, then a 16-bit signature of the row's first, middle and last column); left as
    row_idx unless two runs of at least 32 positions (maximal stretches of non-empty rows
    with one key, in row_idx order) have the same key."""
    m = len(ro) - 1
    order = np.asarray(row_idx, dtype=np.int64)
    if m > 16384 or n > 65536:
        return order
    lens = np.diff(ro).astype(np.int64)
    ne = lens > 0
    a = np.asarray(ro[:-1], dtype=np.int64)
    c0 = np.where(ne, col[np.minimum(a, len(col) - 1)], 0).astype(np.uint64)
    c1 = np.where(ne, col[np.minimum(a + lens // 2, len(col) - 1)], 0).astype(np.uint64)
    c2 = np.where(ne, col[np.maximum(a + lens - 1, 0)], 0).astype(np.uint64)
    h = (_mix_col(c0) + _mix_col(c1 ^ np.uint64(0x55555555)) + _mix_col(c2 ^ np.uint64(0xAAAAAAAA))) & np.uint64(0xFFFFFFFF)
    sig = np.where(ne, (h >> np.uint64(16)) ^ (h & np.uint64(0xFFFF)), np.uint64(0))
    key = (0xFFFF - np.minimum(lens, 0xFFFF)).astype(np.uint64) << np.uint64(16) | sig
    kp, lp = key[order], lens[order]
    long_keys = []
    p = 0
    while p < m:
        e = p + 1
        while e < m and kp[e] == kp[p]:
            e += 1
        if lp[p] > 0 and e - p >= 32:
            long_keys.append(int(kp[p]))
        p = e
    if len(set(long_keys)) == len(long_keys):
        return order
    return order[np.argsort(kp, kind="stable")]


def expected_plan(ro, col, row_idx, n):
    """The panel rule restated on the host: 128 consecutive positions of the plan's row order per panel;
    filled when it has at least 16 non-empty rows and entries * 4 >= rows * |U|; SDDMM tiles
    when also |U| <= 1024 (in groups of up to four tiles), a SpMM image when |U| <= 4096
    (images all fit the budget here)."""
    m = len(ro) - 1
    dense = entries = tiles = spmm = groups = 0
    P = (m + 127) // 128
    for p in range(P):
        rows = row_idx[p * 128:(p + 1) * 128]
        cols = [col[ro[i]:ro[i + 1]] for i in rows]
        nnz_p = sum(len(c) for c in cols)
        ne = sum(1 for c in cols if len(c))
        U = len(np.unique(np.concatenate(cols))) if nnz_p else 0
        filled = nnz_p > 0 and ne >= 16 and nnz_p * 4 >= ne * U
        if filled and U <= 1024:
            dense += 1
            entries += nnz_p
            tiles += (U + 127) // 128
            groups += ((U + 127) // 128 + 3) // 4
        if filled and U <= 4096:
            spmm += 1
    lens = np.diff(ro)
    bins = lambda t: [0, int((lens >= t).sum()), int((lens >= 1).sum()), m]  # noqa: E731
    return {"dense_panels": dense, "dense_entries": entries, "sddmm_tiles": tiles, "spmm_panels": spmm, "panels": P,
            "sddmm_groups": groups,
            "bins_spmm": bins(sp.SPMM_LONG_ROW), "bins_sddmm": bins(sp.SDDMM_LONG_ROW)}


@pytest.mark.parametrize("name", ["rosa_s", "llama_s", "butterfly_s", "rosa_dense", "rosa_dense_i32", "rosa_wide",
                                  "fly_s"])
def test_plan_matches_rule(small_cases, name):
    w = small_cases[name]
    g = to_gpu(w, idx_dtype=torch.int32 if name in INT32_CASES else None)
    got = sp.plan_build(g["ro"], g["row_idx"], g["col"], w.n).stats()
    ro, col = w.row_offsets.numpy(), w.col_idx.numpy()
    row_idx = oracle.sort_rows(ro)
    order = plan_order(ro, col, row_idx, w.n)
    # block masks repeat their rows' patterns and get the order; these random masks keep row_idx
    assert (not np.array_equal(order, row_idx)) == (name in ("butterfly_s", "fly_s")), name
    want = expected_plan(ro, col, order, w.n)
    for k, v in want.items():
        assert got[k] == v, (k, got[k], v)
    if name == "rosa_wide":  # the SpMM-only panels: |U| between 1024 and 4096
        assert got["spmm_panels"] >= 1 and got["dense_panels"] == 0
    elif name != "llama_s":
        assert got["dense_panels"] >= 1  # these cases exercise the tensor-core path


def _pattern_rows(m, n, runs, nnz=16, seed=0):
    """A CSR mask of m rows with nnz entries each: rows in each (start, length) of `runs` hold
    one shared column pattern, every other row its own random pattern."""
    rng = np.random.default_rng(seed)
    shared = np.sort(rng.choice(n, nnz, replace=False))
    rows, cols = [], []
    for i in range(m):
        c = shared if any(s <= i < s + L for s, L in runs) else np.sort(rng.choice(n, nnz, replace=False))
        rows += [i] * nnz
        cols += list(c)
    return _csr(m, n, rows, cols, "bf16", seed)


ORDER_CASES = {
    # two runs of 32 rows, each straddling a 64-position window boundary: ordered
    "straddle": dict(m=512, n=1024, runs=[(48, 32), (300, 32)]),
    # the second run one row short of a long run: row_idx kept
    "short_run": dict(m=512, n=1024, runs=[(48, 32), (300, 31)]),
    # one long run only (a clustered mask's full rows): row_idx kept
    "one_run": dict(m=512, n=1024, runs=[(100, 200)]),
    # more than 1024 runs (the positions' radix sort instead of the runs' bitonic sort)
    "many_runs": dict(m=3000, n=1024, runs=[(48, 32), (2000, 40)]),
}


@pytest.mark.parametrize("name", list(ORDER_CASES) + ["butterfly_s", "fly_s", "rosa_s", "llama_s", "rosa_dense_i32",
                                                      "butterfly", "fly_small_1", "fly_large_1", "rosa", "llama_mlp"])
def test_plan_row_order_matches_rule(small_cases, name):
    """The plan's row order, position by position, against the rule restated on the host."""
    if name in ORDER_CASES:
        c = ORDER_CASES[name]
        ro, col, _ = _pattern_rows(c["m"], c["n"], c["runs"])
        n, idt = c["n"], torch.int16
    else:
        w = small_cases[name] if name in small_cases else wl.generate(wl.spec(name, N=8, kd=8))
        ro, col, n = w.row_offsets.numpy(), w.col_idx.numpy(), w.n
        idt = torch.int32 if name in INT32_CASES else torch.int16
    row_idx = oracle.sort_rows(ro)
    dro = torch.from_numpy(np.asarray(ro, dtype=np.int32)).cuda()
    dcol = torch.from_numpy(np.asarray(col)).to(idt).cuda()
    ridx = torch.from_numpy(row_idx).to(idt).cuda()
    got = sp.plan_build(dro, ridx, dcol, n).row_order().cpu().numpy()
    want = plan_order(ro, col, row_idx, n)
    assert np.array_equal(got, want), name
    ordered = not np.array_equal(want, row_idx)
    assert ordered == (name in ("straddle", "many_runs", "butterfly_s", "fly_s", "butterfly", "fly_small_1",
                                "fly_large_1")), name


@pytest.mark.parametrize("name", ["rosa_dense", "butterfly_s", "llama_s"])
def test_prebuilt_plan_gives_identical_results(small_cases, name):
    w = small_cases[name]
    g = to_gpu(w)
    plan = sp.plan_build(g["ro"], g["row_idx"], g["col"], w.n)
    a = sp.spmm(g["val"], g["ro"], g["row_idx"], g["col"], g["B"], w.m)
    b = sp.spmm(g["val"], g["ro"], g["row_idx"], g["col"], g["B"], w.m, plan=plan)
    c = sp.sddmm(g["ro"], g["row_idx"], g["col"], g["A"], g["BT"])
    d = sp.sddmm(g["ro"], g["row_idx"], g["col"], g["A"], g["BT"], plan=plan)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert torch.equal(c.view(torch.int16), d.view(torch.int16))
    with pytest.raises(ValueError):
        sp.spmm(g["val"], g["ro"], g["row_idx"], g["col"], g["B"][:-1].contiguous(), w.m, plan=plan)


def test_padding_rows_never_leak_into_results(small_cases):
    """Rows of B, A and BT that the mask never references are filled with NaN. The dense
    panels pad their tiles (rows past a panel's |U|, positions past m); those pads must not
    reach any output, so every result stays finite and matches the oracle."""
    w = small_cases["rosa_dense"]
    ro, col = w.row_offsets.numpy(), w.col_idx.numpy()
    used_cols = np.unique(col)
    unused_col = int(np.setdiff1d(np.arange(w.n), used_cols)[0])
    empty_row = int(np.nonzero(np.diff(ro) == 0)[0][0])
    B, A, BT = w.B.clone(), w.A.clone(), w.BT.clone()
    B[unused_col] = float("nan")
    BT[unused_col] = float("nan")
    A[empty_row] = float("nan")
    g = to_gpu(w)
    C = sp.spmm(g["val"], g["ro"], g["row_idx"], g["col"], B.cuda(), w.m)
    out = sp.sddmm(g["ro"], g["row_idx"], g["col"], A.cuda(), BT.cuda())
    torch.cuda.synchronize()
    assert sp.plan_build(g["ro"], g["row_idx"], g["col"], w.n).stats()["dense_panels"] >= 1
    assert_close(C, oracle.spmm(ro, col, w.values, B), w.dtype, "spmm with poisoned unused rows")
    assert_close(out, oracle.sddmm(ro, col, A, BT), w.dtype, "sddmm with poisoned unused rows")
