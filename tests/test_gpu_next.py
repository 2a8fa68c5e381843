"""GPU parity of the widened operators against the fp64 oracle: csr_transpose (bit-exact
structure and values), dB = A^T dC (SpMM of the transpose) and masked Adam."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import (TOL, abs_of, as_f64, assert_bits_equal, assert_close, assert_elementwise, index_dtype,
                     spmm_terms)

pytestmark = pytest.mark.gpu

sp = pytest.importorskip("unstructured_sparse_linear_gb300")

DEV = torch.device("cuda:0")

TRANSPOSE_CASES = {
    "tiny": wl.spec("tiny"),
    "rosa_s": wl.spec("rosa", m=1000, n=1000, N=200, kd=200),
    "llama_s": wl.spec("llama_mlp", m=1100, n=512, N=520, kd=264),
    "zipf_s": wl.spec("zipf", m=4000, n=4000, N=36, mask_kw=(("max_len", 600), ("band", 700))),
    "butterfly_s": wl.spec("butterfly", m=1024, n=256, N=256, kd=136, mask_kw=(("block", 32),)),
    "wide": wl.spec("tiny", m=70, n=20000, density=0.01),  # 15-bit columns: two radix passes
}


def check_transpose(w, idx_dtype, values=True):
    ro = w.row_offsets.to(DEV)
    col = w.col_idx.to(idx_dtype).to(DEV)
    val = w.values.to(DEV) if values else None
    t = sp.csr_transpose(val, ro, col, w.n)
    torch.cuda.synchronize()
    ro_t, row_t, val_t, perm = oracle.csr_transpose(w.row_offsets.numpy(), w.col_idx.numpy(),
                                                    w.values.double().numpy(), w.n)
    assert np.array_equal(t.row_offsets.cpu().numpy(), ro_t)
    assert np.array_equal(t.col_idx.cpu().to(torch.int64).numpy(), row_t)
    assert np.array_equal(t.perm.cpu().numpy(), perm)
    if values:
        fmt = {torch.float32: "f32", torch.float16: "f16", torch.bfloat16: "bf16"}[w.values.dtype]
        assert_bits_equal(t.values, val_t, fmt, "csr_transpose values")
    return t


@pytest.mark.parametrize("name", list(TRANSPOSE_CASES))
def test_transpose_bit_exact(name):
    w = wl.generate(TRANSPOSE_CASES[name], operands=())
    check_transpose(w, index_dtype(w.m, w.n))


@pytest.mark.parametrize("name", ["rosa_s", "zipf_s"])
def test_transpose_int32_and_structure_only(name):
    w = wl.generate(TRANSPOSE_CASES[name], operands=())
    check_transpose(w, torch.int32)
    check_transpose(w, index_dtype(w.m, w.n), values=False)


def test_transpose_edge_cases():
    # empty matrix, one row, one column, empty rows and columns
    for m, n, coords in [(5, 7, []), (1, 9, [(0, 0), (0, 3), (0, 8)]), (6, 1, [(1, 0), (4, 0)]),
                         (8, 8, [(0, 7), (3, 0), (3, 7), (7, 3)])]:
        rows = np.array([r for r, _ in coords], dtype=np.int64)
        cols = np.array([c for _, c in coords], dtype=np.int64)
        ro, col = wl.csr_from_coords(rows, cols, m)
        vals = torch.arange(1, len(coords) + 1, dtype=torch.float32)
        w = wl.Workload("edge", "f32", m, n, torch.from_numpy(ro), torch.from_numpy(col), vals)
        check_transpose(w, torch.int16)


def test_permute_values_follows_transpose():
    w = wl.generate(TRANSPOSE_CASES["rosa_s"], operands=())
    ro = w.row_offsets.to(DEV)
    col = w.col_idx.to(torch.int16).to(DEV)
    t = sp.csr_transpose(None, ro, col, w.n)
    v2 = torch.randn(w.nnz, device=DEV).to(torch.float16)
    got = sp.permute_values(v2, t)
    torch.cuda.synchronize()
    assert torch.equal(got.cpu(), v2.cpu()[t.perm.cpu().long()])


@pytest.mark.parametrize("name", ["tiny", "rosa_s", "llama_s", "zipf_s", "butterfly_s"])
def test_spmm_grad_b(name):
    """dB = A^T dC against the oracle, every element."""
    s = TRANSPOSE_CASES[name]
    w = wl.generate(s, operands=())
    fmt = s.dtype
    dtype = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[fmt]
    rng = np.random.default_rng(7)
    N = 72
    dC = torch.from_numpy(rng.standard_normal((w.m, N))).to(dtype)
    it = index_dtype(w.m, w.n)
    dB = sp.spmm_grad_b(w.values.to(DEV), w.row_offsets.to(DEV), w.col_idx.to(it).to(DEV), dC.to(DEV), w.n)
    torch.cuda.synchronize()
    want = oracle.spmm_grad_b(w.row_offsets.numpy(), w.col_idx.numpy(), w.values, dC, w.n)
    assert dB.shape == (w.n, N)
    assert_close(dB, want, fmt, f"spmm_grad_b {name}")


def test_spmm_grad_b_integer_exact_and_reused_transpose():
    w = wl.generate(TRANSPOSE_CASES["rosa_s"], operands=(), integer_valued=True)
    rng = np.random.default_rng(8)
    dC = torch.from_numpy(rng.integers(-2, 3, (w.m, 40)).astype(np.float32))
    ro, col = w.row_offsets.to(DEV), w.col_idx.to(torch.int16).to(DEV)
    vals = w.values.to(torch.float32).to(DEV)
    t = sp.csr_transpose(None, ro, col, w.n)
    dB = sp.spmm_grad_b(vals, ro, col, dC.to(DEV), w.n, transpose=t)
    torch.cuda.synchronize()
    want = oracle.spmm_grad_b(w.row_offsets.numpy(), w.col_idx.numpy(), w.values, dC, w.n)
    assert_bits_equal(dB, want, "f32", "integer dB")


def test_spmm_grad_b_full_size_rosa():
    """The RoSA adapter at full size (4096 x 4096, 1 % clustered, fp16, 2048 tokens): every
    element of dB against the oracle's transpose + SpMM, by the Frobenius tolerance and the
    element-wise fp32-accumulation bound."""
    w = wl.generate("rosa", operands=())
    rng = np.random.default_rng(9)
    dC = torch.from_numpy(rng.standard_normal((w.m, 2048))).to(torch.float16)
    dB = sp.spmm_grad_b(w.values.to(DEV), w.row_offsets.to(DEV), w.col_idx.to(torch.int16).to(DEV), dC.to(DEV), w.n)
    torch.cuda.synchronize()
    ro_t, row_t, val_t, _ = oracle.csr_transpose(w.row_offsets.numpy(), w.col_idx.numpy(), w.values, w.n)
    want = oracle.spmm(ro_t, row_t, val_t, dC)
    absdot = oracle.spmm(ro_t, row_t, np.abs(val_t), abs_of(dC))
    assert_close(dB, want, "f16", "full-size dB")
    assert_elementwise(dB, want, absdot, spmm_terms(ro_t), "f16", "full-size dB")


def test_transpose_full_size_zipf():
    """131072 x 131072, int32 indices, about 6.4 M entries: bit-exact against the oracle."""
    w = wl.generate("zipf", operands=())
    check_transpose(w, torch.int32)


# ---------------------------------------------------------------- masked Adam


def adam_state(rng, n):
    p = rng.standard_normal(n).astype(np.float32)
    m = (rng.standard_normal(n) * 0.01).astype(np.float32)
    v = (rng.random(n) * 1e-3).astype(np.float32)
    return p, m, v


def assert_adam_close(got, want, what, lr=1e-3, steps=1, gmax=1.0):
    """fp32 against fp64. Each step rounds the parameter once (half an ulp: rtol) and
    computes the update lr * mhat / (sqrt(vhat) + eps) through about 15 fp32 operations,
    relative error below 1e-6 of an update no larger than 4 * lr here: atol. The first
    moment can cancel towards zero: its atol is steps * (1 - beta1) * |g| * 2 ulps."""
    p, m, v = (x.detach().cpu().double().numpy() for x in got)
    wp, wm, wv = want
    np.testing.assert_allclose(p, wp, rtol=5e-7, atol=steps * 4 * lr * 1e-6, err_msg=what + " param")
    np.testing.assert_allclose(m, wm, rtol=2e-6, atol=steps * 0.1 * gmax * 2.4e-7, err_msg=what + " exp_avg")
    np.testing.assert_allclose(v, wv, rtol=2e-6, atol=1e-14, err_msg=what + " exp_avg_sq")


@pytest.mark.parametrize("gdtype", [torch.float32, torch.float16, torch.bfloat16])
@pytest.mark.parametrize("maximize", [False, True])
def test_masked_adam_values(gdtype, maximize):
    rng = np.random.default_rng(11)
    n = 167_772 + 3  # the RoSA adapter's entries plus a ragged tail of the 4-wide loop
    p, m, v = adam_state(rng, n)
    P, M, V = (torch.from_numpy(x).to(DEV) for x in (p, m, v))
    wp, wm, wv = p.astype(np.float64), m.astype(np.float64), v.astype(np.float64)
    for step in range(1, 4):
        g = torch.from_numpy(rng.standard_normal(n) * 0.1).to(gdtype)
        sp.masked_adam(P, M, V, g.to(DEV), step, lr=2e-3, betas=(0.9, 0.99), eps=1e-8, maximize=maximize)
        wp, wm, wv = oracle.masked_adam(wp, wm, wv, g.double().numpy(), step, lr=2e-3, betas=(0.9, 0.99), eps=1e-8,
                                        maximize=maximize)
    torch.cuda.synchronize()
    assert_adam_close((P, M, V), (wp, wm, wv), "masked_adam", lr=2e-3, steps=3, gmax=0.6)


def test_masked_adam_unaligned_views():
    """Offsets that defeat the 16-byte path take the scalar loop."""
    rng = np.random.default_rng(12)
    n = 1001
    p, m, v = adam_state(rng, n + 1)
    P, M, V = (torch.from_numpy(x).to(DEV)[1:] for x in (p, m, v))
    g = torch.from_numpy(rng.standard_normal(n).astype(np.float32))
    sp.masked_adam(P, M, V, g.to(DEV), 1)
    torch.cuda.synchronize()
    want = oracle.masked_adam(p[1:], m[1:], v[1:], g.numpy(), 1)
    assert_adam_close((P, M, V), want, "masked_adam unaligned", gmax=4.0)


def test_masked_adam_csr_dense_param_page_example():
    """The SparseAdam page's example: gradient [0, 5, 0, 0, 9] over a 5-entry parameter."""
    ro = torch.tensor([0, 2], dtype=torch.int32, device=DEV)
    col = torch.tensor([1, 4], dtype=torch.int16, device=DEV)
    g = torch.tensor([5.0, 9.0], device=DEV)
    rng = np.random.default_rng(13)
    p, m, v = adam_state(rng, 5)
    P, M, V = (torch.from_numpy(x).reshape(1, 5).to(DEV) for x in (p, m, v))
    sp.masked_adam(P, M, V, g, 4, row_offsets=ro, col_idx=col)
    torch.cuda.synchronize()
    want = oracle.masked_adam(p, m, v, [5.0, 9.0], 4, positions=[1, 4])
    assert_adam_close((P.reshape(-1), M.reshape(-1), V.reshape(-1)), want, "page example", gmax=9.0)
    for i in (0, 2, 3):
        assert P.reshape(-1)[i].item() == p[i] and M.reshape(-1)[i].item() == m[i] and V.reshape(-1)[i].item() == v[i]


@pytest.mark.parametrize("idx_dtype", [torch.int16, torch.int32])
def test_masked_adam_csr_rosa_mask(idx_dtype):
    """Dense 1000 x 1000 parameter, gradient on a clustered mask: untouched entries keep
    their bits, masked entries match the oracle."""
    w = wl.generate(wl.spec("rosa", m=1000, n=1000), operands=())
    rng = np.random.default_rng(14)
    p, m, v = adam_state(rng, w.m * w.n)
    P, M, V = (torch.from_numpy(x).reshape(w.m, w.n).to(DEV) for x in (p, m, v))
    g = w.values.to(torch.bfloat16)
    sp.masked_adam(P, M, V, g.to(DEV), 2, lr=1e-3, row_offsets=w.row_offsets.to(DEV),
                   col_idx=w.col_idx.to(idx_dtype).to(DEV))
    torch.cuda.synchronize()
    ro, col = w.row_offsets.numpy(), w.col_idx.numpy().astype(np.int64)
    rows = np.repeat(np.arange(w.m), np.diff(ro))
    pos = rows * w.n + col
    want = oracle.masked_adam(p, m, v, g.double().numpy(), 2, lr=1e-3, positions=pos)
    assert_adam_close((P.reshape(-1), M.reshape(-1), V.reshape(-1)), want, "masked_adam_csr", gmax=0.1)
    untouched = np.ones(w.m * w.n, dtype=bool)
    untouched[pos] = False
    assert np.array_equal(P.reshape(-1).cpu().numpy()[untouched], p[untouched])


def test_masked_adam_rejects_bad_hyperparameters():
    x = torch.zeros(8, device=DEV)
    with pytest.raises(ValueError):
        sp.masked_adam(x, x.clone(), x.clone(), x.clone(), 0)
    with pytest.raises(ValueError):
        sp.masked_adam(x, x.clone(), x.clone(), x.clone(), 1, betas=(1.0, 0.9))
    with pytest.raises(ValueError):
        sp.masked_adam(x, x, x.clone(), x.clone(), 1)  # param and exp_avg alias


# ---------------------------------------------------------------- narrow-N SpMM (SpMV)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("N", [1, 3, 8, 16])
def test_spmm_narrow_all_elements(dtype, N):
    """N <= 16 takes the warp-per-row streaming kernel (vector or scalar B loads)."""
    s = wl.spec("spmv", m=3000, n=2500, density=0.05, dtype=dtype, N=N)
    w = wl.generate(s)
    it = index_dtype(w.m, w.n)
    ro, col = w.row_offsets.to(DEV), w.col_idx.to(it).to(DEV)
    row_idx = torch.from_numpy(oracle.sort_rows(w.row_offsets.numpy())).to(it).to(DEV)
    C = sp.spmm(w.values.to(DEV), ro, row_idx, col, w.B.to(DEV), w.m)
    torch.cuda.synchronize()
    want = oracle.spmm(w.row_offsets.numpy(), w.col_idx.numpy(), w.values, w.B)
    assert_close(C, want, dtype, f"narrow spmm N={N}")


def test_spmm_narrow_integer_exact_unaligned_b_and_empty_rows():
    s = wl.spec("spmv", m=500, n=700, density=0.03, dtype="f16", N=8)
    w = wl.generate(s, integer_valued=True)
    ro, col = w.row_offsets.to(DEV), w.col_idx.to(torch.int16).to(DEV)
    row_idx = torch.from_numpy(oracle.sort_rows(w.row_offsets.numpy())).to(torch.int16).to(DEV)
    Bbig = torch.zeros(w.n * 8 + 1, dtype=torch.float16, device=DEV)
    B = Bbig[1:].view(w.n, 8)  # 2-byte offset: the scalar path
    B.copy_(w.B.to(DEV))
    for b in (w.B.to(DEV), B):
        C = sp.spmm(w.values.to(DEV), ro, row_idx, col, b, w.m)
        torch.cuda.synchronize()
        want = oracle.spmm(w.row_offsets.numpy(), w.col_idx.numpy(), w.values, w.B)
        assert_bits_equal(C, want, "f16", "integer narrow spmm")
    # a matrix whose rows are all empty but one
    ro1 = torch.zeros(w.m + 1, dtype=torch.int32)
    ro1[5:] = 1
    C = sp.spmm(torch.ones(1, dtype=torch.float16, device=DEV), ro1.to(DEV), row_idx,
                torch.tensor([3], dtype=torch.int16, device=DEV), w.B.to(DEV), w.m)
    torch.cuda.synchronize()
    expect = torch.zeros((w.m, 8), dtype=torch.float16)
    expect[4] = w.B[3]
    assert torch.equal(C.cpu(), expect)


def test_spmm_narrow_full_size():
    """The 8192 x 8192, 90 %-sparse, N = 8 workload and its SpMV column (N = 1): every
    element against the oracle."""
    w = wl.generate("spmv")
    ro, col = w.row_offsets.to(DEV), w.col_idx.to(torch.int16).to(DEV)
    row_idx = sp.sort_rows(ro, nnz=w.nnz, index_dtype=torch.int16)
    ro_h, col_h = w.row_offsets.numpy(), w.col_idx.numpy()
    for B in (w.B, w.B[:, :1].contiguous()):
        C = sp.spmm(w.values.to(DEV), ro, row_idx, col, B.to(DEV), w.m)
        torch.cuda.synchronize()
        want = oracle.spmm(ro_h, col_h, w.values, B)
        absdot = oracle.spmm(ro_h, col_h, abs_of(w.values), abs_of(B))
        assert_close(C, want, "f16", f"narrow full size N={B.shape[1]}")
        assert_elementwise(C, want, absdot, spmm_terms(ro_h), "f16", f"narrow full size N={B.shape[1]}")


# ---------------------------------------------------------------- sparse linear layer (pixelfly)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_sparse_linear_forward_backward(dtype):
    """Feature-major butterfly layer: Y^T = W X^T, dW on the mask, dX^T = W^T dY^T, all
    against the oracle; the forward also against a dense fp64 product."""
    s = wl.spec("butterfly", m=512, n=256, N=136, kd=136, dtype=dtype, mask_kw=(("block", 32),))
    w = wl.generate(s, operands=("B", "A"))
    tdt = {"f16": torch.float16, "bf16": torch.bfloat16}[dtype]
    layer = sp.SparseLinear(w.row_offsets.to(DEV), w.col_idx.to(torch.int16).to(DEV), w.values.to(DEV).clone(),
                            in_features=w.n)
    Xt = w.B.to(DEV).clone().requires_grad_(True)      # in x tokens
    G = w.A.to(DEV)                                     # dY^T: out x tokens
    Yt = layer(Xt)
    Yt.backward(G)
    torch.cuda.synchronize()
    ro, col = w.row_offsets.numpy(), w.col_idx.numpy()
    assert_close(Yt.detach(), oracle.spmm(ro, col, w.values, w.B), dtype, "layer forward")
    assert_close(layer.values.grad, oracle.sddmm(ro, col, w.A, w.B), dtype, "layer dW")
    assert_close(Xt.grad, oracle.spmm_grad_b(ro, col, w.values, w.A, w.n), dtype, "layer dX")
    dense = torch.zeros((w.m, w.n), dtype=torch.float64)
    rows = np.repeat(np.arange(w.m), np.diff(ro))
    dense[rows, col] = w.values.double()
    ref = (dense @ w.B.double()).numpy()
    assert_close(Yt.detach(), ref, dtype, "layer forward vs dense fp64")


@pytest.mark.slow
@pytest.mark.parametrize("name", [n for mlp in wl.FLY_MLPS for n in wl.fly_layer_names(mlp)])
def test_pixelfly_mlp_layer_full_size(name):
    """The layers of the pixelfly issue's two MLPs at their own shapes (block 48: K chunks of
    the tensor-core panels end inside a block; block 256), 8192 tokens: forward Y^T = W X^T,
    dW = dY^T X on the mask and dX^T = W^T dY^T through SparseLinear's autograd function,
    every element against the oracle by the Frobenius tolerance and the element-wise
    fp32-accumulation bound."""
    w = wl.generate(name, operands=("B", "A"))
    layer = sp.SparseLinear(w.row_offsets.to(DEV), w.col_idx.to(torch.int16).to(DEV), w.values.to(DEV).clone(),
                            in_features=w.n)
    assert layer.plan.stats()["spmm_panels"] > 0  # the forward runs on the tensor cores
    Xt = w.B.to(DEV).clone().requires_grad_(True)
    Yt = layer(Xt)
    Yt.backward(w.A.to(DEV))
    torch.cuda.synchronize()
    ro, col = w.row_offsets.numpy(), w.col_idx.numpy()
    aval, aX, aG = abs_of(w.values), abs_of(w.B), abs_of(w.A)
    want = oracle.spmm(ro, col, w.values, w.B)
    assert_close(Yt.detach(), want, "bf16", f"{name} forward")
    assert_elementwise(Yt.detach(), want, oracle.spmm(ro, col, aval, aX), spmm_terms(ro), "bf16", f"{name} forward")
    del want
    want = oracle.sddmm(ro, col, w.A, w.B)
    assert_close(layer.values.grad, want, "bf16", f"{name} dW")
    assert_elementwise(layer.values.grad, want, oracle.sddmm(ro, col, aG, aX), w.A.shape[1], "bf16", f"{name} dW")
    del want
    ro_t, row_t, val_t, _ = oracle.csr_transpose(ro, col, w.values, w.n)
    want = oracle.spmm(ro_t, row_t, val_t, w.A)
    assert_close(Xt.grad, want, "bf16", f"{name} dX")
    assert_elementwise(Xt.grad, want, oracle.spmm(ro_t, row_t, np.abs(val_t), aG), spmm_terms(ro_t), "bf16",
                       f"{name} dX")
