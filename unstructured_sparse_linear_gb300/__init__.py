"""spops_gb300: CSR sparse-adapter operators (SpMM, SDDMM, csr_add) for GB300 (sm_103a).

Thin PyTorch binding over the C ABI in ``include/spops_gb300.h``. PyTorch provides device
memory and the current stream; every step of every operator runs in this package's CUDA
kernels. The functions keep the spops README signatures ("Sparse Operations (spops)",
section "Usage"):

    csr_add(A_val, A_row_offsets, A_row_indices, A_col_indices, B)
    spmm(A_val, A_row_offsets, A_row_indices, A_col_indices, B, m)
    sddmm(out_row_offsets, out_row_indices, out_col_indices, A, BT, backend="structure_aware")

plus the row scheduler helpers ``sort_rows`` (builds row_idx) and ``row_bins``, and
``check_csr`` (device-side structure check). Index lists are int16 (the README's type) or
int32 (for matrices with more than 32768 rows or columns); row_offsets is int32. All
inputs must be contiguous CUDA tensors on the same device.
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib

__all__ = ["spmm", "sddmm", "csr_add", "sort_rows", "row_bins", "check_csr", "plan_build", "Plan", "SpopsError", "library_path",
           "release_streams",
           "SPMM_LONG_ROW", "SDDMM_LONG_ROW"]

SPMM_LONG_ROW = 256
SDDMM_LONG_ROW = 64

_DTYPE = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}
_ITYPE = {torch.int16: 0, torch.int32: 1}
_BACKEND = {"structure_aware": 0, "general": 1, "sputnik": 1}
_SPMM_PATH = {"auto": 0, "general": 1}
_ERR_CLASS = {1: ValueError, 2: ValueError, 3: ValueError}


class SpopsError(RuntimeError):
    pass


def library_path() -> str:
    return _lib.lib_path()


def _L():
    return _lib.load()


def _check(status: int, what: str):
    if status != 0:
        lib = _L()
        name = lib.spops_status_string(status).decode()
        msg = lib.spops_last_error().decode()
        raise _ERR_CLASS.get(status, SpopsError)(f"{what}: {name}: {msg}")


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None and t.numel() > 0 else ctypes.c_void_p(0)


def _req(t, name, dtype=None, dtypes=None, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must have dtype {dtype}, got {t.dtype}")
    if dtypes is not None and t.dtype not in dtypes:
        raise ValueError(f"{name} dtype {t.dtype} not in {list(dtypes)}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    return t


def _itype(col_idx, row_idx=None):
    it = _ITYPE.get(col_idx.dtype)
    if it is None:
        raise ValueError(f"index lists must be int16 or int32, got {col_idx.dtype}")
    if row_idx is not None and row_idx.dtype != col_idx.dtype:
        raise ValueError("row_idx and col_idx must have the same dtype")
    return it


def _ws(nbytes: int, device):
    return torch.empty(max(int(nbytes), 16), dtype=torch.uint8, device=device)


def release_streams() -> None:
    """Destroy the calling thread's side streams and events (the library's only persistent
    host-side resources); later calls create them again."""
    _check(_L().spops_release_streams(), "release_streams")


def sort_rows(row_offsets: torch.Tensor, nnz: int | None = None, index_dtype=torch.int16) -> torch.Tensor:
    """row_idx: the rows ordered by nnz descending, ties by ascending row id."""
    _req(row_offsets, "row_offsets", torch.int32)
    m = row_offsets.numel() - 1
    if nnz is None:
        nnz = int(row_offsets[-1].item())
    out = torch.empty(m, dtype=index_dtype, device=row_offsets.device)
    lib = _L()
    with torch.cuda.device(row_offsets.device):
        ws = _ws(lib.spops_sort_rows_workspace_size(m), row_offsets.device)
        _check(lib.spops_sort_rows(_p(row_offsets), m, int(nnz), _p(out), _ITYPE[index_dtype], _p(ws), ws.numel(),
                                   _stream()), "sort_rows")
    return out


def row_bins(row_offsets: torch.Tensor, t_long: int) -> torch.Tensor:
    """Device int32[4] = {0, #rows with nnz >= t_long, #rows with nnz >= 1, m}."""
    _req(row_offsets, "row_offsets", torch.int32)
    m = row_offsets.numel() - 1
    out = torch.empty(4, dtype=torch.int32, device=row_offsets.device)
    with torch.cuda.device(row_offsets.device):
        _check(_L().spops_row_bins(_p(row_offsets), m, int(t_long), _p(out), _stream()), "row_bins")
    return out


class Plan:
    """A mask plan (row bins and dense panels) built once per CSR structure; pass it to
    spmm / sddmm on the same mask to skip rebuilding it in every call."""

    def __init__(self, buf: torch.Tensor, m: int, n: int, nnz: int):
        self.buf, self.m, self.n, self.nnz = buf, m, n, nnz

    def ptr(self):
        return ctypes.c_void_p(self.buf.data_ptr())

    def stats(self) -> dict:
        """Summary of the plan (synchronizes)."""
        out = torch.zeros(16, dtype=torch.int32, device=self.buf.device)
        with torch.cuda.device(self.buf.device):
            _check(_L().spops_plan_stats(self.ptr(), self.m, self.n, self.nnz, _p(out), _stream()), "plan_stats")
        s = out.cpu().tolist()
        return {"dense_panels": s[0], "sddmm_tiles": s[1], "spmm_panels": s[2], "dense_entries": s[3],
                "image_elems": s[4], "panels": s[5], "sddmm_groups": s[6], "bins_spmm": s[8:12],
                "bins_sddmm": s[12:16]}

    def row_order(self) -> torch.Tensor:
        """The row at each position of the plan's row order (int32 [m], on the plan's
        device): row_idx, or row_idx sorted by (nnz, column pattern) when rows with one
        pattern recur in separate runs. Masks wider than 65536 columns have no panels and
        raise."""
        out = torch.empty(self.m, dtype=torch.int32, device=self.buf.device)
        with torch.cuda.device(self.buf.device):
            _check(_L().spops_plan_row_order(self.ptr(), self.m, self.n, self.nnz, _p(out), _stream()),
                   "plan_row_order")
        return out


def plan_build(row_offsets, row_idx, col_idx, n: int) -> Plan:
    """Build the mask plan of an m x n CSR structure (asynchronous on the current stream)."""
    _req(row_offsets, "row_offsets", torch.int32)
    dev = row_offsets.device
    _req(col_idx, "col_idx", device=dev)
    _req(row_idx, "row_idx", device=dev)
    m = row_offsets.numel() - 1
    it = _itype(col_idx, row_idx)
    nnz = col_idx.numel()
    lib = _L()
    size = int(lib.spops_plan_size(m, int(n), nnz))
    raw = torch.empty(size + 1024, dtype=torch.uint8, device=dev)
    off = (-raw.data_ptr()) % 1024
    buf = raw[off:off + size]
    with torch.cuda.device(dev):
        _check(lib.spops_plan_build(_p(row_offsets), _p(row_idx), _p(col_idx), it, m, int(n), nnz, _p(buf), size,
                                    _stream()), "plan_build")
    plan = Plan(buf, m, int(n), nnz)
    plan._raw = raw
    return plan


def _plan_ptr(plan, m, n, nnz):
    if plan is None:
        return ctypes.c_void_p(0)
    if (plan.m, plan.n, plan.nnz) != (m, n, nnz):
        raise ValueError(f"plan was built for (m, n, nnz) = {(plan.m, plan.n, plan.nnz)}, not {(m, n, nnz)}")
    return plan.ptr()


def spmm(A_val, A_row_offsets, A_row_indices, A_col_indices, B, m: int, out: torch.Tensor | None = None,
         path: str = "auto", plan: Plan | None = None):
    """C = A @ B for a CSR matrix A (m rows) and a dense row-major B.
    path="auto" runs dense row panels on the tensor cores, "general" every row on the
    general row kernels. plan: a Plan of this mask (optional)."""
    if path not in _SPMM_PATH:
        raise ValueError(f"path must be one of {list(_SPMM_PATH)}")
    _req(B, "B", dtypes=_DTYPE)
    dev = B.device
    _req(A_val, "A_val", B.dtype, device=dev)
    _req(A_row_offsets, "A_row_offsets", torch.int32, device=dev)
    _req(A_col_indices, "A_col_indices", device=dev)
    _req(A_row_indices, "A_row_indices", device=dev)
    if B.dim() != 2:
        raise ValueError("B must be 2-D")
    m = int(m)
    if A_row_offsets.numel() != m + 1:
        raise ValueError(f"A_row_offsets must have m + 1 = {m + 1} entries")
    k, n = B.shape
    it = _itype(A_col_indices, A_row_indices)
    nnz = A_col_indices.numel()
    if A_val.numel() != nnz or A_row_indices.numel() != m:
        raise ValueError("A_val / A_row_indices lengths do not match col_idx / m")
    C = out if out is not None else torch.empty((m, n), dtype=B.dtype, device=dev)
    _req(C, "out", B.dtype, device=dev)
    lib = _L()
    dt = _DTYPE[B.dtype]
    with torch.cuda.device(dev):
        ws = _ws(lib.spops_spmm_workspace_size(m, k, n, nnz, dt, it), dev)
        _check(lib.spops_spmm(_p(A_val), _p(A_row_offsets), _p(A_row_indices), _p(A_col_indices), it, dt, m, k, nnz,
                              _p(B), n, _p(C), _SPMM_PATH[path], _plan_ptr(plan, m, k, nnz), _p(ws), ws.numel(),
                              _stream()), "spmm")
    return C


def sddmm(out_row_offsets, out_row_indices, out_col_indices, A, BT, backend: str = "structure_aware",
          out: torch.Tensor | None = None, plan: Plan | None = None):
    """out[k] = A[i, :] . BT[col[k], :] for every entry k (row i) of the CSR mask.
    plan: a Plan of this mask (optional)."""
    _req(A, "A", dtypes=_DTYPE)
    dev = A.device
    _req(BT, "BT", A.dtype, device=dev)
    _req(out_row_offsets, "out_row_offsets", torch.int32, device=dev)
    _req(out_col_indices, "out_col_indices", device=dev)
    _req(out_row_indices, "out_row_indices", device=dev)
    if A.dim() != 2 or BT.dim() != 2 or A.shape[1] != BT.shape[1]:
        raise ValueError("A (m x kd) and BT (n x kd) must be 2-D with the same kd")
    if backend not in _BACKEND:
        raise ValueError(f"backend must be one of {list(_BACKEND)}")
    m, kd = A.shape
    n = BT.shape[0]
    if out_row_offsets.numel() != m + 1 or out_row_indices.numel() != m:
        raise ValueError("mask row arrays do not match A's rows")
    it = _itype(out_col_indices, out_row_indices)
    nnz = out_col_indices.numel()
    res = out if out is not None else torch.empty(nnz, dtype=A.dtype, device=dev)
    _req(res, "out", A.dtype, device=dev)
    lib = _L()
    dt, be = _DTYPE[A.dtype], _BACKEND[backend]
    with torch.cuda.device(dev):
        ws = _ws(lib.spops_sddmm_workspace_size(m, n, kd, nnz, dt, it, be), dev)
        _check(lib.spops_sddmm(_p(out_row_offsets), _p(out_row_indices), _p(out_col_indices), it, dt, m, n, kd, nnz,
                               _p(A), _p(BT), _p(res), be, _plan_ptr(plan, m, n, nnz), _p(ws), ws.numel(),
                               _stream()), "sddmm")
    return res


def csr_add(A_val, A_row_offsets, A_row_indices, A_col_indices, B, out: torch.Tensor | None = None):
    """C = B + A for a CSR matrix A and a dense B of the same shape (out=B: in place)."""
    _req(B, "B", dtypes=_DTYPE)
    dev = B.device
    _req(A_val, "A_val", B.dtype, device=dev)
    _req(A_row_offsets, "A_row_offsets", torch.int32, device=dev)
    _req(A_col_indices, "A_col_indices", device=dev)
    if A_row_indices is not None:
        _req(A_row_indices, "A_row_indices", device=dev)
    if B.dim() != 2:
        raise ValueError("B must be 2-D")
    m, n = B.shape
    if A_row_offsets.numel() != m + 1:
        raise ValueError("A_row_offsets must have B.shape[0] + 1 entries")
    it = _itype(A_col_indices, A_row_indices)
    nnz = A_col_indices.numel()
    C = out if out is not None else torch.empty_like(B)
    _req(C, "out", B.dtype, device=dev)
    with torch.cuda.device(dev):
        _check(_L().spops_csr_add(_p(A_val), _p(A_row_offsets), _p(A_row_indices), _p(A_col_indices), it,
                                  _DTYPE[B.dtype], m, n, nnz, _p(B), _p(C), _stream()), "csr_add")
    return C


def check_csr(row_offsets, col_idx, row_idx, n: int) -> None:
    """Run the device-side CSR structure check; raise SpopsError on a violation."""
    _req(row_offsets, "row_offsets", torch.int32)
    dev = row_offsets.device
    _req(col_idx, "col_idx", device=dev)
    m = row_offsets.numel() - 1
    it = _itype(col_idx, row_idx)
    lib = _L()
    with torch.cuda.device(dev):
        ws = _ws(lib.spops_check_csr_workspace_size(m), dev)
        _check(lib.spops_check_csr(_p(row_offsets), _p(col_idx), _p(row_idx), it, m, int(n), col_idx.numel(), _p(ws),
                                   ws.numel(), _stream()), "check_csr")
        code = ctypes.c_int32(0)
        _check(lib.spops_get_device_error(_stream(), ctypes.byref(code)), "get_device_error")
    if code.value != 0:
        raise SpopsError(f"CSR check failed: device error code {code.value}")


# ---------------------------------------------------------------- transpose and dB = A^T dC


class Transpose:
    """A^T of a CSR matrix (n x m): row_offsets [n+1] int32, col_idx (row ids of A, the
    index dtype of A's col_idx), values (or None), perm [nnz] int32 (the entry of A at each
    position, for refreshing values with ``permute_values``)."""

    def __init__(self, row_offsets, col_idx, values, perm):
        self.row_offsets = row_offsets
        self.col_idx = col_idx
        self.values = values
        self.perm = perm


def csr_transpose(values, row_offsets, col_idx, n: int) -> Transpose:
    """A^T of the m x n CSR matrix (values may be None for the structure only). Canonical:
    row j of A^T lists column j of A by ascending row (spops README, "csr_transpose")."""
    _req(row_offsets, "row_offsets", torch.int32)
    dev = row_offsets.device
    _req(col_idx, "col_idx", device=dev)
    m = row_offsets.numel() - 1
    nnz = col_idx.numel()
    it = _itype(col_idx)
    if values is not None:
        _req(values, "values", dtypes=_DTYPE, device=dev)
        if values.numel() != nnz:
            raise ValueError("values and col_idx lengths differ")
    dt = _DTYPE[values.dtype] if values is not None else 0
    n = int(n)
    ro_t = torch.empty(n + 1, dtype=torch.int32, device=dev)
    col_t = torch.empty(nnz, dtype=col_idx.dtype, device=dev)
    val_t = torch.empty(nnz, dtype=values.dtype, device=dev) if values is not None else None
    perm = torch.empty(nnz, dtype=torch.int32, device=dev)
    lib = _L()
    with torch.cuda.device(dev):
        ws = _ws(lib.spops_csr_transpose_workspace_size(nnz), dev)
        _check(lib.spops_csr_transpose(_p(row_offsets), _p(col_idx), _p(values), it, dt, m, n, nnz, _p(ro_t), _p(col_t),
                                       _p(val_t), _p(perm), _p(ws), ws.numel(), _stream()), "csr_transpose")
    return Transpose(ro_t, col_t, val_t, perm)


def permute_values(values, t: Transpose, out: torch.Tensor | None = None) -> torch.Tensor:
    """New values of A in the order of an existing transpose: out[p] = values[t.perm[p]]."""
    _req(values, "values", dtypes=_DTYPE)
    dev = values.device
    _req(t.perm, "perm", torch.int32, device=dev)
    nnz = t.perm.numel()
    if values.numel() != nnz:
        raise ValueError("values and the transpose have different nnz")
    res = out if out is not None else torch.empty(nnz, dtype=values.dtype, device=dev)
    _req(res, "out", values.dtype, device=dev)
    with torch.cuda.device(dev):
        _check(_L().spops_csr_permute_values(_p(values), _p(t.perm), _DTYPE[values.dtype], nnz, _p(res), _stream()),
               "csr_permute_values")
    return res


def spmm_grad_b(A_val, A_row_offsets, A_col_indices, dC, n: int, transpose: Transpose | None = None,
                path: str = "auto"):
    """dB = A^T @ dC, the gradient of C = A @ B (A m x n in CSR) with respect to B: the
    transpose (built here unless given; its values are refreshed from A_val), its nnz-sorted
    row permutation, and one spmm of the transpose."""
    t = transpose if transpose is not None else csr_transpose(A_val, A_row_offsets, A_col_indices, n)
    vals = t.values if (transpose is None and t.values is not None) else permute_values(A_val, t)
    idx_dtype = t.col_idx.dtype
    row_idx = sort_rows(t.row_offsets, nnz=t.col_idx.numel(), index_dtype=idx_dtype)
    return spmm(vals, t.row_offsets, row_idx, t.col_idx, dC, int(n), path=path)


# ---------------------------------------------------------------- masked Adam


def masked_adam(param, exp_avg, exp_avg_sq, grad, step: int, lr: float = 1e-3, betas=(0.9, 0.999), eps: float = 1e-8,
                maximize: bool = False, row_offsets=None, col_idx=None):
    """One Adam step, in place, on the entries the sparse gradient materializes (SparseAdam
    page: moments and parameters move only under the gradient's mask).
    Without row_offsets: param / exp_avg / exp_avg_sq (fp32) and grad hold one value per
    entry of one CSR mask (the RoSA adapter's values). With row_offsets / col_idx: param and
    the moments are dense m x n fp32 and grad holds the CSR gradient's values."""
    _req(param, "param", torch.float32)
    dev = param.device
    _req(exp_avg, "exp_avg", torch.float32, device=dev)
    _req(exp_avg_sq, "exp_avg_sq", torch.float32, device=dev)
    _req(grad, "grad", dtypes=_DTYPE, device=dev)
    b1, b2 = float(betas[0]), float(betas[1])
    lib = _L()
    with torch.cuda.device(dev):
        if row_offsets is None:
            if not (param.numel() == exp_avg.numel() == exp_avg_sq.numel() == grad.numel()):
                raise ValueError("param, exp_avg, exp_avg_sq and grad must have the same number of entries")
            _check(lib.spops_masked_adam(_p(param), _p(exp_avg), _p(exp_avg_sq), _p(grad), _DTYPE[grad.dtype],
                                         param.numel(), int(step), float(lr), b1, b2, float(eps), int(bool(maximize)),
                                         _stream()), "masked_adam")
        else:
            _req(row_offsets, "row_offsets", torch.int32, device=dev)
            _req(col_idx, "col_idx", device=dev)
            if param.dim() != 2 or exp_avg.shape != param.shape or exp_avg_sq.shape != param.shape:
                raise ValueError("param and moments must be the same 2-D shape")
            m, n = param.shape
            if row_offsets.numel() != m + 1 or grad.numel() != col_idx.numel():
                raise ValueError("row_offsets / grad do not match param / col_idx")
            _check(lib.spops_masked_adam_csr(_p(param), _p(exp_avg), _p(exp_avg_sq), _p(grad), _DTYPE[grad.dtype],
                                             _p(row_offsets), _p(col_idx), _itype(col_idx), m, n, col_idx.numel(),
                                             int(step), float(lr), b1, b2, float(eps), int(bool(maximize)), _stream()),
                   "masked_adam_csr")
    return param


__all__ += ["Transpose", "csr_transpose", "permute_values", "spmm_grad_b", "masked_adam"]

from .layer import SparseLinear, SparseLinearFunction  # noqa: E402  (uses the functions above)

__all__ += ["SparseLinear", "SparseLinearFunction"]
