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
