"""fp64 CPU oracle for the CSR sparse-adapter operators (spmm, sddmm, csr_add, sort_rows,
row_bins, csr_transpose, masked_adam) -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import this package. It shares no code with ``unstructured_sparse_linear_gb300`` and never
imports it. The arithmetic lives in ``spops_oracle.c`` (plain C, fp64, one row at a time);
this file only builds that library with gcc and marshals numpy arrays into it.

Each function follows the spops README ("Sparse Operations (spops)", section "Usage" and
the per-operation sections); see the C file's header for the readings taken where the
README is silent.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "spops_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libspops_oracle.so")
_lock = threading.Lock()
_lib = None

FMT = {"f32": 0, "f16": 1, "bf16": 2}


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP when the compiler has it). Returns the path."""
    os.makedirs(_BUILD, exist_ok=True)
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp,
            "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i32 = ctypes.c_int32
            lib.oracle_num_threads.restype = ctypes.c_int
            lib.oracle_set_threads.argtypes = [i32]
            lib.oracle_sort_rows.argtypes = [i32, P, P]
            lib.oracle_row_bins.argtypes = [i32, P, i32, P]
            lib.oracle_spmm.argtypes = [i32, i32, i32, P, P, P, P, P, P, i32]
            lib.oracle_sddmm.argtypes = [i32, i32, i32, P, P, P, P, P, P, i32]
            lib.oracle_csr_add.argtypes = [i32, i32, P, P, P, P, P, P, i32]
            lib.oracle_csr_transpose.argtypes = [i32, i32, P, P, P, P, P, P, P]
            lib.oracle_masked_adam.argtypes = [ctypes.c_int64, P, P, P, P, P, i32, ctypes.c_double, ctypes.c_double,
                                               ctypes.c_double, ctypes.c_double, i32]
            lib.oracle_round.argtypes = [ctypes.c_double, i32]
            lib.oracle_round.restype = ctypes.c_double
            lib.oracle_round_array.argtypes = [P, P, ctypes.c_int64, i32]
            _lib = lib
    return _lib


def _i32(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def _f64(x) -> np.ndarray:
    if hasattr(x, "detach"):  # a torch tensor: every supported dtype widens exactly to fp64
        x = x.detach().cpu().double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_threads(n: int) -> None:
    """Threads of the oracle's parallel loops from now on (results do not depend on it)."""
    _load().oracle_set_threads(int(n))


def sort_rows(row_offsets) -> np.ndarray:
    ro = _i32(row_offsets)
    m = ro.size - 1
    out = np.empty(m, dtype=np.int32)
    _load().oracle_sort_rows(m, _ptr(ro), _ptr(out))
    return out


def row_bins(row_offsets, t_long: int) -> np.ndarray:
    ro = _i32(row_offsets)
    out = np.empty(4, dtype=np.int32)
    _load().oracle_row_bins(ro.size - 1, _ptr(ro), int(t_long), _ptr(out))
    return out


def spmm(row_offsets, col_idx, values, B, rows=None) -> np.ndarray:
    """C = A @ B in fp64 (all rows, or the listed rows in the listed order)."""
    ro, col, val, b = _i32(row_offsets), _i32(col_idx), _f64(values), _f64(B)
    m = ro.size - 1
    kdim, n = b.shape
    if rows is None:
        out = np.empty((m, n), dtype=np.float64)
        _load().oracle_spmm(m, kdim, n, _ptr(ro), _ptr(col), _ptr(val), _ptr(b), _ptr(out), None, 0)
    else:
        r = _i32(rows)
        out = np.empty((r.size, n), dtype=np.float64)
        _load().oracle_spmm(m, kdim, n, _ptr(ro), _ptr(col), _ptr(val), _ptr(b), _ptr(out), _ptr(r), r.size)
    return out


def sddmm(row_offsets, col_idx, A, BT, rows=None) -> np.ndarray:
    """out[k] = A[i, :] . BT[col[k], :] in fp64. With ``rows``, A is either the full m-row
    matrix (sliced here) or already the listed rows; the result holds the listed rows'
    entries in order."""
    ro, col, bt = _i32(row_offsets), _i32(col_idx), _f64(BT)
    m = ro.size - 1
    n, kd = bt.shape
    if rows is None:
        a = _f64(A)
        out = np.empty(int(ro[-1]), dtype=np.float64)
        _load().oracle_sddmm(m, n, kd, _ptr(ro), _ptr(col), _ptr(a), _ptr(bt), _ptr(out), None, 0)
    else:
        r = _i32(rows)
        a = _f64(A[r.astype(np.int64)] if A.shape[0] == m else A)
        total = int(np.sum(ro[r + 1] - ro[r]))
        out = np.empty(total, dtype=np.float64)
        _load().oracle_sddmm(m, n, kd, _ptr(ro), _ptr(col), _ptr(a), _ptr(bt), _ptr(out), _ptr(r), r.size)
    return out


def csr_add(row_offsets, col_idx, values, B, rows=None) -> np.ndarray:
    """C = B + dense(A) in fp64. With ``rows``, B holds (or is sliced to) the listed rows."""
    ro, col, val = _i32(row_offsets), _i32(col_idx), _f64(values)
    m = ro.size - 1
    if rows is None:
        b = _f64(B)
        out = np.empty_like(b)
        _load().oracle_csr_add(m, b.shape[1], _ptr(ro), _ptr(col), _ptr(val), _ptr(b), _ptr(out), None, 0)
    else:
        r = _i32(rows)
        b = _f64(B[r.astype(np.int64)] if B.shape[0] == m else B)
        out = np.empty_like(b)
        _load().oracle_csr_add(m, b.shape[1], _ptr(ro), _ptr(col), _ptr(val), _ptr(b), _ptr(out), _ptr(r), r.size)
    return out


def csr_transpose(row_offsets, col_idx, values, n: int):
    """A^T of the m x n CSR matrix as (row_offsets_t [n+1], row_ids [nnz], values_t [nnz],
    perm [nnz]); perm[p] is the entry of A placed at position p (spops README operation
    list, "csr_transpose")."""
    ro, col, val = _i32(row_offsets), _i32(col_idx), _f64(values)
    m = ro.size - 1
    nnz = int(ro[-1]) if m >= 0 else 0
    ro_t = np.empty(n + 1, dtype=np.int32)
    row_t = np.empty(nnz, dtype=np.int32)
    val_t = np.empty(nnz, dtype=np.float64)
    perm = np.empty(nnz, dtype=np.int32)
    _load().oracle_csr_transpose(m, int(n), _ptr(ro), _ptr(col), _ptr(val), _ptr(ro_t), _ptr(row_t), _ptr(val_t),
                                 _ptr(perm))
    return ro_t, row_t, val_t, perm


def spmm_grad_b(row_offsets, col_idx, values, dC, n: int) -> np.ndarray:
    """dB = A^T @ dC in fp64 for C = A @ B with A m x n in CSR: the SpMM of the transpose."""
    ro_t, row_t, val_t, _ = csr_transpose(row_offsets, col_idx, values, n)
    return spmm(ro_t, row_t, val_t, dC)


def masked_adam(param, exp_avg, exp_avg_sq, grad, step: int, lr=1e-3, betas=(0.9, 0.999), eps=1e-8,
                maximize=False, positions=None):
    """One Adam step on the entries `positions` (all entries when None) of fp64 copies of
    param / exp_avg / exp_avg_sq; returns the three updated arrays (SparseAdam page: moments
    and parameters change only where the sparse gradient has a materialized value)."""
    p, m1, m2 = _f64(param).copy(), _f64(exp_avg).copy(), _f64(exp_avg_sq).copy()
    g = _f64(grad)
    pos = None if positions is None else np.ascontiguousarray(np.asarray(positions, dtype=np.int64))
    _load().oracle_masked_adam(g.size, None if pos is None else _ptr(pos), _ptr(g), _ptr(p), _ptr(m1), _ptr(m2),
                               int(step), float(lr), float(betas[0]), float(betas[1]), float(eps),
                               1 if maximize else 0)
    return p, m1, m2


def round_to(x, fmt: str) -> np.ndarray:
    """Round fp64 values to fp32 / fp16 / bf16 (ties to even); returned as fp64."""
    a = _f64(x)
    out = np.empty_like(a)
    _load().oracle_round_array(_ptr(a), _ptr(out), a.size, FMT[fmt])
    return out


def round_scalar(x: float, fmt: str) -> float:
    return float(_load().oracle_round(float(x), FMT[fmt]))
