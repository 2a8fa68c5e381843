"""Shared test helpers: move a workload to the GPU in the spops index layout, and compare
GPU results with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle

# Relative Frobenius-error bounds for floating-point outputs (fp32 operands; fp16/bf16
# operands with fp32 accumulation).
TOL = {"f32": 1e-5, "f16": 3e-3, "bf16": 3e-3}


def index_dtype(m: int, n: int):
    return torch.int16 if max(m, n) <= 32768 else torch.int32


def to_gpu(w, idx_dtype=None, row_idx=None):
    """CSR + operands on cuda:0. row_idx defaults to the oracle's sorted permutation."""
    it = idx_dtype or index_dtype(w.m, w.n)
    dev = torch.device("cuda:0")
    if row_idx is None:
        row_idx = torch.from_numpy(oracle.sort_rows(w.row_offsets.numpy()))
    g = {
        "ro": w.row_offsets.to(dev),
        "col": w.col_idx.to(it).to(dev),
        "row_idx": row_idx.to(it).to(dev),
        "val": w.values.to(dev),
    }
    for k in ("B", "A", "BT", "W"):
        t = getattr(w, k)
        if t is not None:
            g[k] = t.to(dev)
    return g


def rel_fro(got, want) -> float:
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    den = np.linalg.norm(want)
    num = np.linalg.norm(got - want)
    if den == 0:
        return float(num)
    return float(num / den)


def as_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().double().numpy()


def assert_close(got: torch.Tensor, want64: np.ndarray, fmt: str, what: str):
    g = as_f64(got)
    assert g.shape == want64.shape, (what, g.shape, want64.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    err = rel_fro(g, want64)
    assert err <= TOL[fmt], f"{what}: relative Frobenius error {err:.3e} > {TOL[fmt]:.0e}"
    return err


# Element-wise bound on fp32 accumulation (any order, any split into partial sums, tensor
# cores included): each of the `terms` additions of a result is off by at most one fp32 ulp
# of a partial sum, and every partial sum is at most sum |a_t b_t| in magnitude, so
#     |acc - exact| <= 2^-23 * terms * sum_t |a_t b_t|;
# rounding acc to the output dtype then adds half an ulp of the dtype at |acc|.
ACC_UNIT = 2.0 ** -23
_FMT_BITS = {"f32": (23, -126), "f16": (10, -14), "bf16": (7, -126)}  # mantissa bits, min normal exponent


def ulp(x: np.ndarray, fmt: str) -> np.ndarray:
    """Spacing of the dtype's representable numbers at |x| (subnormal spacing below the
    smallest normal)."""
    p, emin = _FMT_BITS[fmt]
    x = np.abs(np.asarray(x, dtype=np.float64))
    _, e2 = np.frexp(x)                      # x = f * 2^e2, f in [0.5, 1)
    e = np.maximum(e2 - 1, emin)
    return np.ldexp(1.0, e - p)


def assert_elementwise(got: torch.Tensor, want64: np.ndarray, absdot64: np.ndarray, terms, fmt: str, what: str):
    """Every element within 2^-23 * terms * sum|a b| + 1/2 ulp_fmt of the oracle's fp64 value.
    absdot64: the oracle run on |values| and |operands| (same shape as want64); terms: the
    number of products summed per element (scalar or broadcastable to want64)."""
    g = as_f64(got)
    assert g.shape == want64.shape == absdot64.shape, (what, g.shape, want64.shape, absdot64.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    acc_err = ACC_UNIT * np.asarray(terms, dtype=np.float64) * absdot64
    bound = acc_err + 0.5 * ulp(np.abs(want64) + acc_err, fmt)
    diff = np.abs(g - want64)
    bad = diff > bound
    if bad.any():
        i = np.unravel_index(int(np.argmax(diff - bound)), diff.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} of {diff.size} elements outside the fp32-accumulation bound; "
                             f"worst at {tuple(int(x) for x in i)}: got {g[i]!r} want {want64[i]!r} "
                             f"bound {bound[i]:.3e}")


def spmm_terms(row_offsets: np.ndarray, rows=None) -> np.ndarray:
    """Products summed per SpMM output row (the row's entry count), as a column vector."""
    lens = np.diff(np.asarray(row_offsets, dtype=np.int64))
    if rows is not None:
        lens = lens[np.asarray(rows, dtype=np.int64)]
    return lens[:, None]


def abs_of(t) -> np.ndarray:
    return np.abs(as_f64(t) if isinstance(t, torch.Tensor) else np.asarray(t, dtype=np.float64))


def assert_bits_equal(got: torch.Tensor, want64: np.ndarray, fmt: str, what: str):
    """Bit-for-bit equality with the oracle's fp64 result rounded to the dtype."""
    want = torch.from_numpy(oracle.round_to(want64, fmt)).to(got.dtype)
    g = got.detach().cpu()
    assert g.shape == want.shape
    view = torch.int32 if got.dtype == torch.float32 else torch.int16
    gv, wv = g.contiguous().view(view), want.contiguous().view(view)
    bad = (gv != wv).nonzero()
    assert bad.numel() == 0, f"{what}: {bad.shape[0]} elements differ, first at {bad[0].tolist()}: " \
                             f"got {g[tuple(bad[0].tolist())].item()} want {want[tuple(bad[0].tolist())].item()}"


def sample_rows(ro: np.ndarray, count: int, seed: int = 0) -> np.ndarray:
    """Rows to check at full size: the longest rows, some empty rows, random rows."""
    lens = np.diff(ro)
    rng = np.random.default_rng(seed)
    order = np.argsort(-lens, kind="stable")
    pick = list(order[: count // 4])
    empty = np.nonzero(lens == 0)[0]
    if empty.size:
        pick += list(rng.choice(empty, size=min(4, empty.size), replace=False))
    pick += list(rng.choice(len(lens), size=count - len(pick), replace=False))
    return np.unique(np.asarray(pick, dtype=np.int64))
