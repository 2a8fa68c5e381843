"""Pins for the fp64 oracle: each check ties it to something other than itself --
worked structures printed on the pages, brute force on tiny inputs, closed forms,
special cases that reduce to numpy/torch routines, and invariants of the definitions.
CPU only."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as wl


def rand_csr(rng, m, n, density, empty_rows=()):
    mask = rng.random((m, n)) < density
    for r in empty_rows:
        mask[r] = False
    rows, cols = np.nonzero(mask)
    ro, col = wl.csr_from_coords(rows, cols, m)
    return ro, col


def densify(ro, col, val, m, n):
    D = np.zeros((m, n))
    for i in range(m):
        for k in range(ro[i], ro[i + 1]):
            D[i, col[k]] = val[k]
    return D


# ------------------------------------------------------------------ worked structures


def test_golden_ust_coo_structure(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "ust_coo_4x8.json")))
    m, n = g["shape"]
    ro, col = wl.csr_from_coords(np.array(g["row"]), np.array(g["col"]), m)
    d = g["derived_by_hand"]
    assert ro.tolist() == d["row_offsets"]
    assert col.tolist() == d["col_idx"]
    assert np.diff(ro).tolist() == d["row_lengths"]
    assert oracle.sort_rows(ro).tolist() == d["row_idx"]
    # A @ I8 is A itself, made dense
    val = np.array(g["val"], dtype=np.float64)
    C = oracle.spmm(ro, col, val, np.eye(n))
    assert C.tolist() == d["dense"]
    # B = 0: csr_add gives dense(A); row_offsets[m] = nnz
    assert oracle.csr_add(ro, col, val, np.zeros((m, n))).tolist() == d["dense"]
    assert ro[-1] == len(g["val"])


def test_golden_tsgu_sparse_gradient(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "tsgu_coo_2x3.json")))
    idx = np.array(g["indices"])
    vals = np.array(g["values"])
    m, n = g["A_shape"]
    ro, col = wl.csr_from_coords(idx[0], idx[1], m)
    d = g["derived_by_hand"]
    assert ro.tolist() == d["row_offsets"] and col.tolist() == d["col_idx"]
    assert oracle.sort_rows(ro).tolist() == d["row_idx"]
    assert densify(ro, col, vals, m, n).tolist() == d["dense"]
    # the sparse gradient of sum(A @ B) by autograd on a dense copy, read at A's entries
    B = torch.from_numpy(np.random.default_rng(5).standard_normal((n, g["B_cols"])))
    Ad = torch.tensor(d["dense"], dtype=torch.float64, requires_grad=True)
    (Ad @ B).sum().backward()
    want = Ad.grad.numpy()[idx[0], idx[1]]
    got = oracle.sddmm(ro, col, np.ones((m, g["B_cols"])), B.numpy())
    np.testing.assert_allclose(got, want, rtol=1e-15, atol=0)
    # closed form: the row sums of B at each entry's column
    np.testing.assert_allclose(got, B.numpy().sum(1)[col], rtol=1e-15)


# ------------------------------------------------------------------ brute force


@pytest.mark.parametrize("seed", range(4))
def test_spmm_brute_force(seed):
    rng = np.random.default_rng(100 + seed)
    m, k, n = rng.integers(1, 40, size=3)
    ro, col = rand_csr(rng, m, k, 0.3, empty_rows=[0] if m > 2 else [])
    val = rng.integers(-4, 5, size=col.size).astype(np.float64)
    B = rng.integers(-3, 4, size=(k, n)).astype(np.float64)
    D = densify(ro, col, val, m, k)
    assert np.array_equal(oracle.spmm(ro, col, val, B), D @ B)  # integers: exact
    valf = rng.standard_normal(col.size)
    Bf = rng.standard_normal((k, n))
    np.testing.assert_allclose(oracle.spmm(ro, col, valf, Bf), densify(ro, col, valf, m, k) @ Bf, rtol=1e-12,
                               atol=1e-12)
    rows = rng.permutation(m)[: max(1, m // 2)]
    np.testing.assert_allclose(oracle.spmm(ro, col, valf, Bf, rows=rows), (densify(ro, col, valf, m, k) @ Bf)[rows],
                               rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("seed", range(4))
def test_sddmm_brute_force(seed):
    rng = np.random.default_rng(200 + seed)
    m, n, kd = rng.integers(1, 40, size=3)
    ro, col = rand_csr(rng, m, n, 0.3)
    A = rng.standard_normal((m, kd))
    BT = rng.standard_normal((n, kd))
    full = A @ BT.T
    rows_of = np.repeat(np.arange(m), np.diff(ro))
    np.testing.assert_allclose(oracle.sddmm(ro, col, A, BT), full[rows_of, col], rtol=1e-12, atol=1e-12)
    Ai = rng.integers(-3, 4, size=(m, kd)).astype(np.float64)
    Bi = rng.integers(-3, 4, size=(n, kd)).astype(np.float64)
    assert np.array_equal(oracle.sddmm(ro, col, Ai, Bi), (Ai @ Bi.T)[rows_of, col])
    sel = rng.permutation(m)[: max(1, m // 3)]
    want = np.concatenate([full[i, col[ro[i]:ro[i + 1]]] for i in sel])
    np.testing.assert_allclose(oracle.sddmm(ro, col, A, BT, rows=sel), want, rtol=1e-12, atol=1e-12)


def test_sddmm_full_mask_is_matmul():
    rng = np.random.default_rng(3)
    m, n, kd = 17, 23, 9
    ro, col = wl.csr_from_coords(*np.nonzero(np.ones((m, n))), m)
    A = rng.standard_normal((m, kd))
    BT = rng.standard_normal((n, kd))
    np.testing.assert_allclose(oracle.sddmm(ro, col, A, BT).reshape(m, n), A @ BT.T, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("seed", range(3))
def test_csr_add_brute_force(seed):
    rng = np.random.default_rng(300 + seed)
    m, n = rng.integers(1, 50, size=2)
    ro, col = rand_csr(rng, m, n, 0.2)
    val = rng.standard_normal(col.size)
    B = rng.standard_normal((m, n))
    assert np.array_equal(oracle.csr_add(ro, col, val, B), B + densify(ro, col, val, m, n))
    rows = np.arange(m)[::2]
    assert np.array_equal(oracle.csr_add(ro, col, val, B, rows=rows), (B + densify(ro, col, val, m, n))[rows])


# ------------------------------------------------------------------ special cases


def test_identity_spmm_returns_B():
    n = 37
    ro, col = wl.csr_from_coords(np.arange(n), np.arange(n), n)
    B = np.random.default_rng(1).standard_normal((n, 5))
    assert np.array_equal(oracle.spmm(ro, col, np.ones(n), B), B)


def test_empty_matrix():
    m, n = 6, 9
    ro = np.zeros(m + 1, dtype=np.int32)
    col = np.zeros(0, dtype=np.int32)
    B = np.random.default_rng(2).standard_normal((n, 4))
    assert np.array_equal(oracle.spmm(ro, col, np.zeros(0), B), np.zeros((m, 4)))
    W = np.random.default_rng(2).standard_normal((m, n))
    assert np.array_equal(oracle.csr_add(ro, col, np.zeros(0), W), W)
    assert oracle.sddmm(ro, col, np.ones((m, 3)), np.ones((n, 3))).size == 0
    assert oracle.sort_rows(ro).tolist() == list(range(m))
    assert oracle.row_bins(ro, 4).tolist() == [0, 0, 0, m]


def test_adjoint_identity_links_spmm_and_sddmm():
    """sum_k S_k * SDDMM(mask, A, BT)_k == <A, S @ BT>_F for any values S on the mask.
    A transposed operand, a wrong column index or a dropped term in either function
    breaks it."""
    rng = np.random.default_rng(11)
    m, n, kd = 31, 27, 13
    ro, col = rand_csr(rng, m, n, 0.25)
    S = rng.standard_normal(col.size)
    A = rng.standard_normal((m, kd))
    BT = rng.standard_normal((n, kd))
    lhs = float(np.dot(S, oracle.sddmm(ro, col, A, BT)))
    rhs = float(np.sum(A * oracle.spmm(ro, col, S, BT)))
    assert abs(lhs - rhs) <= 1e-11 * (1 + abs(lhs))


# ------------------------------------------------------------------ row permutation and bins


@pytest.mark.parametrize("seed", range(3))
def test_sort_rows_definition(seed):
    rng = np.random.default_rng(400 + seed)
    m = int(rng.integers(1, 300))
    lens = rng.integers(0, 6, size=m)  # many ties
    ro = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    got = oracle.sort_rows(ro)
    # library routine: a stable argsort on -nnz keeps ascending row ids among equals
    assert np.array_equal(got, np.argsort(-lens, kind="stable"))
    assert sorted(got.tolist()) == list(range(m))
    nn = lens[got]
    assert np.all(nn[:-1] >= nn[1:])
    ties = nn[:-1] == nn[1:]
    assert np.all(got[:-1][ties] < got[1:][ties])


def test_row_bins_partition():
    rng = np.random.default_rng(7)
    lens = rng.integers(0, 300, size=500)
    lens[::7] = 0
    ro = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    for t in (1, 32, 128, 299, 1000):
        b = oracle.row_bins(ro, t)
        assert b[0] == 0 and b[3] == 500 and b[1] <= b[2] <= b[3]
        order = oracle.sort_rows(ro)
        nn = lens[order]
        assert np.all(nn[: b[1]] >= t) and np.all(nn[b[1]:b[2]] < max(t, 1)) and np.all(nn[b[1]:b[2]] >= 1)
        assert np.all(nn[b[2]:] == 0)


# ------------------------------------------------------------------ rounding


def _fp16_grid():
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    v = bits.view(np.float16).astype(np.float64)
    return v[np.isfinite(v)]


def test_round_fp16_exhaustive_and_midpoints():
    v = np.unique(_fp16_grid())
    assert np.array_equal(oracle.round_to(v, "f16"), v)
    mid = (v[:-1] + v[1:]) / 2  # exact in fp64
    r = oracle.round_to(mid, "f16")
    even = np.where((v[:-1].astype(np.float16).view(np.uint16) & 1) == 0, v[:-1], v[1:])
    assert np.array_equal(r, even)


def test_round_fp16_matches_numpy():
    rng = np.random.default_rng(8)
    x = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-9, 6, 20000),
                        [65504.0, 65519.99, 65520.0, 1e6, -1e6, 2.0 ** -25, 2.0 ** -24 * 1.5, -2.0 ** -26, 0.0,
                         -0.0]])
    got = oracle.round_to(x, "f16")
    with np.errstate(over="ignore"):
        want = x.astype(np.float16).astype(np.float64)
    assert np.array_equal(got, want)
    assert np.array_equal(np.signbit(got), np.signbit(want))


def test_round_fp32_matches_numpy():
    rng = np.random.default_rng(9)
    x = rng.standard_normal(20000) * 10.0 ** rng.integers(-44, 38, 20000)
    got = oracle.round_to(x, "f32")
    assert np.array_equal(got, x.astype(np.float32).astype(np.float64))


def test_round_bf16_matches_torch():
    rng = np.random.default_rng(10)
    x32 = (rng.standard_normal(20000) * 10.0 ** rng.integers(-38, 38, 20000)).astype(np.float32)
    x32 = np.concatenate([x32, np.array([2.0 ** -133, 2.0 ** -134, 3.3895314e38, 3.4e38], dtype=np.float32)])
    got = oracle.round_to(x32.astype(np.float64), "bf16")
    want = torch.from_numpy(x32).to(torch.bfloat16).double().numpy()
    assert np.array_equal(got, want)
    allb = torch.arange(0, 1 << 16, dtype=torch.int32).to(torch.int16).view(torch.bfloat16).double().numpy()
    allb = allb[np.isfinite(allb)]
    assert np.array_equal(oracle.round_to(allb, "bf16"), allb)


@pytest.mark.parametrize("fmt", ["f32", "f16", "bf16"])
def test_csr_add_is_correctly_rounded_sum(fmt):
    """One fp64 add then one rounding equals the dtype's own correctly rounded add
    (numpy for fp32/fp16, torch for bf16), including cancellation and overflow."""
    rng = np.random.default_rng(12)
    dt = wl.DTYPES[fmt]
    a = torch.from_numpy(rng.standard_normal(50000) * 10.0 ** rng.integers(-6, 4, 50000)).to(dt)
    b = torch.from_numpy(rng.standard_normal(50000) * 10.0 ** rng.integers(-6, 4, 50000)).to(dt)
    b[:100] = -a[:100]
    want = (a + b)
    if fmt == "f16":
        want = torch.from_numpy((a.numpy() + b.numpy()))
    elif fmt == "f32":
        want = torch.from_numpy(a.numpy() + b.numpy())
    ro = np.arange(a.numel() + 1, dtype=np.int32)
    col = np.zeros(a.numel(), dtype=np.int32)
    got = oracle.round_to(oracle.csr_add(ro, col, a, b.double().numpy()[:, None]).ravel(), fmt)
    assert np.array_equal(got, want.double().numpy())


# ------------------------------------------------------------------ butterfly, second restatement


def test_butterfly_blockwise_restatement():
    """The butterfly layout as dense blocks: per block-row, sum its dense block products
    (the two-stage block view of the pixelfly issue). Must equal the CSR oracle."""
    blk, nbr, nbc = 8, 16, 8
    m, n, N, kd = nbr * blk, nbc * blk, 12, 10
    ro, col = wl.butterfly_mask(m, n, block=blk, stages=3)
    rng = np.random.default_rng(13)
    val = rng.standard_normal(col.size)
    Dn = densify(ro, col, val, m, n)
    B = rng.standard_normal((n, N))
    C = np.zeros((m, N))
    for r in range(nbr):
        c = r % nbc
        for b in sorted({c, c ^ 1, c ^ 2, c ^ 4}):
            C[r * blk:(r + 1) * blk] += Dn[r * blk:(r + 1) * blk, b * blk:(b + 1) * blk] @ B[b * blk:(b + 1) * blk]
    np.testing.assert_allclose(oracle.spmm(ro, col, val, B), C, rtol=1e-12, atol=1e-12)
    A = rng.standard_normal((m, kd))
    BT = rng.standard_normal((n, kd))
    out = oracle.sddmm(ro, col, A, BT)
    blocks = {}
    for r in range(nbr):
        c = r % nbc
        for b in {c, c ^ 1, c ^ 2, c ^ 4}:
            blocks[(r, b)] = A[r * blk:(r + 1) * blk] @ BT[b * blk:(b + 1) * blk].T
    rows_of = np.repeat(np.arange(m), np.diff(ro))
    want = np.array([blocks[(i // blk, j // blk)][i % blk, j % blk] for i, j in zip(rows_of, col)])
    np.testing.assert_allclose(out, want, rtol=1e-12, atol=1e-12)
    assert np.all(np.diff(ro) == 4 * blk)


# ------------------------------------------------------------------ the workload recipes


def test_workload_recipes_small_and_structured():
    w = wl.generate("tiny")
    assert w.nnz == 3277 and w.B.shape == (256, 64) and w.W.shape == (256, 256)
    ro = w.row_offsets.numpy()
    assert ro[-1] == w.nnz and np.all(np.diff(ro) >= 0)
    col = w.col_idx.numpy()
    for i in range(w.m):
        seg = col[ro[i]:ro[i + 1]]
        assert np.all(np.diff(seg) > 0)
    r = wl.generate(wl.spec("rosa", m=1024, n=1024, N=16, kd=16))
    lens = np.diff(r.row_offsets.numpy())
    assert (lens > 0).sum() <= round(0.1 * 1024) and len(np.unique(r.col_idx.numpy())) <= round(0.1 * 1024)
    assert r.nnz == min(round(0.01 * 1024 * 1024), 102 * 102)  # capped by the 10 % x 10 % block


# ------------------------------------------------------------------ transpose and dB = A^T dC


def test_golden_ust_transpose(golden_dir):
    """The hand-derived transpose of the UST article's 4 x 8 COO example."""
    g = json.load(open(os.path.join(golden_dir, "ust_coo_4x8.json")))
    m, n = g["shape"]
    ro, col = wl.csr_from_coords(np.array(g["row"]), np.array(g["col"]), m)
    t = g["derived_by_hand"]["transpose"]
    ro_t, row_t, val_t, perm = oracle.csr_transpose(ro, col, np.array(g["val"], dtype=np.float64), n)
    assert ro_t.tolist() == t["row_offsets"]
    assert row_t.tolist() == t["row_ids"]
    assert val_t.tolist() == t["values"]
    assert perm.tolist() == t["perm"]


@pytest.mark.parametrize("seed", range(4))
def test_transpose_dense_and_involution(seed):
    rng = np.random.default_rng(400 + seed)
    m, n = int(rng.integers(1, 40)), int(rng.integers(1, 40))
    ro, col = rand_csr(rng, m, n, 0.2, empty_rows=(0,) if m > 2 else ())
    val = rng.standard_normal(ro[-1])
    ro_t, row_t, val_t, perm = oracle.csr_transpose(ro, col, val, n)
    np.testing.assert_array_equal(densify(ro_t, row_t, val_t, n, m), densify(ro, col, val, m, n).T)
    for j in range(n):  # canonical: ascending row ids inside every row of A^T
        assert np.all(np.diff(row_t[ro_t[j]:ro_t[j + 1]]) > 0)
    np.testing.assert_array_equal(val_t, val[perm])
    ro2, col2, val2, _ = oracle.csr_transpose(ro_t, row_t, val_t, m)
    np.testing.assert_array_equal(ro2, ro)
    np.testing.assert_array_equal(col2, col)
    np.testing.assert_array_equal(val2, val)


def test_transpose_matches_scipy():
    sparse = pytest.importorskip("scipy.sparse")
    rng = np.random.default_rng(410)
    m, n = 57, 91
    ro, col = rand_csr(rng, m, n, 0.1)
    val = rng.standard_normal(ro[-1])
    At = sparse.csr_matrix((val, col, ro), shape=(m, n)).transpose().tocsr()
    At.sort_indices()
    ro_t, row_t, val_t, _ = oracle.csr_transpose(ro, col, val, n)
    np.testing.assert_array_equal(ro_t, At.indptr)
    np.testing.assert_array_equal(row_t, At.indices)
    np.testing.assert_array_equal(val_t, At.data)


@pytest.mark.parametrize("seed", range(3))
def test_spmm_grad_b_brute_force_and_adjoint(seed):
    """dB = A^T dC: brute force on a dense copy, and <A X, Y> = <X, A^T Y>."""
    rng = np.random.default_rng(420 + seed)
    m, n, N = 23, 31, 7
    ro, col = rand_csr(rng, m, n, 0.25)
    val = rng.standard_normal(ro[-1])
    dC = rng.standard_normal((m, N))
    dB = oracle.spmm_grad_b(ro, col, val, dC, n)
    np.testing.assert_allclose(dB, densify(ro, col, val, m, n).T @ dC, rtol=1e-13, atol=1e-13)
    X = rng.standard_normal((n, N))
    lhs = np.sum(oracle.spmm(ro, col, val, X) * dC)
    rhs = np.sum(X * dB)
    assert abs(lhs - rhs) <= 1e-11 * max(1.0, abs(lhs))
    # integer-valued inputs: exact
    vi = rng.integers(-3, 4, ro[-1]).astype(np.float64)
    Ci = rng.integers(-3, 4, (m, N)).astype(np.float64)
    np.testing.assert_array_equal(oracle.spmm_grad_b(ro, col, vi, Ci, n), densify(ro, col, vi, m, n).T @ Ci)


# ------------------------------------------------------------------ masked Adam (SparseAdam page)


def test_sparse_adam_page_mask(golden_dir):
    """The page's example: only the entries under the gradient's mask move."""
    g = json.load(open(os.path.join(golden_dir, "sparse_adam_mask.json")))
    dense = np.array(g["gradient_dense"], dtype=np.float64)
    pos = np.nonzero(dense)[0]
    assert (dense != 0).astype(int).tolist() == g["mask"]
    rng = np.random.default_rng(430)
    p0 = rng.standard_normal(dense.size)
    m0 = rng.standard_normal(dense.size) * 0.1
    v0 = rng.random(dense.size) * 0.1
    d = g["defaults"]
    p, m1, v1 = oracle.masked_adam(p0, m0, v0, dense[pos], 3, lr=d["lr"], betas=d["betas"], eps=d["eps"],
                                   maximize=d["maximize"], positions=pos)
    off = np.array(g["mask"]) == 0
    np.testing.assert_array_equal(p[off], p0[off])
    np.testing.assert_array_equal(m1[off], m0[off])
    np.testing.assert_array_equal(v1[off], v0[off])
    assert np.all(p[~off] != p0[~off]) and np.all(m1[~off] != m0[~off]) and np.all(v1[~off] != v0[~off])


def test_masked_adam_first_step_closed_form():
    """From zero moments, step 1 moves each entry by lr * g / (|g| + eps)."""
    g = np.array([5.0, -9.0, 1e-3, -2.5])
    p, m1, v1 = oracle.masked_adam(np.zeros(4), np.zeros(4), np.zeros(4), g, 1)
    np.testing.assert_allclose(p, -1e-3 * g / (np.abs(g) + 1e-8), rtol=1e-13)
    np.testing.assert_allclose(m1, 0.1 * g, rtol=1e-15)
    np.testing.assert_allclose(v1, 0.001 * g * g, rtol=1e-13)


@pytest.mark.parametrize("maximize", [False, True])
def test_masked_adam_matches_torch_adam(maximize):
    """On the masked entries, several steps equal torch.optim.Adam (fp64, dense)."""
    rng = np.random.default_rng(440 + int(maximize))
    n = 37
    pos = np.sort(rng.choice(n, 11, replace=False))
    p0 = rng.standard_normal(n)
    w = torch.tensor(p0[pos], dtype=torch.float64, requires_grad=True)
    opt = torch.optim.Adam([w], lr=3e-3, betas=(0.8, 0.95), eps=1e-6, maximize=maximize)
    p, m1, v1 = p0.copy(), np.zeros(n), np.zeros(n)
    for t in range(1, 5):
        g = rng.standard_normal(pos.size)
        w.grad = torch.tensor(g, dtype=torch.float64)
        opt.step()
        p, m1, v1 = oracle.masked_adam(p, m1, v1, g, t, lr=3e-3, betas=(0.8, 0.95), eps=1e-6, maximize=maximize,
                                       positions=pos)
    np.testing.assert_allclose(p[pos], w.detach().numpy(), rtol=1e-13, atol=1e-15)
    rest = np.setdiff1d(np.arange(n), pos)
    np.testing.assert_array_equal(p[rest], p0[rest])
