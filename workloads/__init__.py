"""Seeded synthetic inputs shared by the oracle tests, the GPU parity tests and the bench.

This module only draws random numbers and lays them out as CSR index arrays and dense
operands. It contains none of the operators' arithmetic (no products, no sums of
values, no rounding of results), so the oracle and the CUDA path can both consume its
output without sharing any of the method.

CSR layout (spops README "Sparse Operations (spops)", section "Usage"): ``values`` of
length nnz, ``row_offsets`` of length m + 1 (int32), ``col_idx`` of length nnz and a
row permutation ``row_idx``. The generator returns canonical CSR: columns strictly
increasing inside each row. It does not compute ``row_idx``; that is an operator.

Every operand draws from its own stream, ``SeedSequence([config_seed, operand_id])``,
so any operand can be regenerated alone, at any size, with the same values.

Workloads (sizes, densities and distributions of the five named configurations):

1. ``tiny``      256x256 fp32, 5 % uniform mask, values N(0,1); B 256x64; SDDMM 256x64
                 operands; csr_add into a dense 256x256.
2. ``rosa``      4096x4096 fp16 RoSA adapter, 1 % density, all nonzeros inside a random
                 10 % of rows x 10 % of columns, values N(0, 0.02); B = tokens 4096x2048;
                 SDDMM A = dY^T 4096x2048, BT = X^T 4096x2048; csr_add into W N(0, 0.02).
3. ``llama_mlp`` 11008x4096 bf16, 0.5 % uniform, values N(0, 0.02); B 4096x4096;
                 SDDMM A 11008x4096, BT 4096x4096; csr_add into W N(0, 0.02).
4. ``zipf``      131072x131072 fp32, row lengths Zipf(1.5) on [1, 4096] (resampled above
                 4096), columns uniform without replacement within +-8192 of the diagonal,
                 values U(-1, 1); B 131072x128 N(0,1). SpMM only.
5. ``butterfly`` 8192x2048 bf16, 64x64 blocks, block-row r holds blocks at block-columns
                 {r mod 32} and {(r mod 32) XOR 2^s : s = 0, 1, 2}; values N(0, 0.02);
                 B 2048x8192; SDDMM A 8192x8192, BT 2048x8192. No csr_add.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

# operand stream ids
_MASK, _VALUES, _B, _A, _BT, _W = range(6)

DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


def _rng(seed: int, operand: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([int(seed), int(operand)]))


def _to_dtype(x64: np.ndarray, dtype: str) -> torch.Tensor:
    """Store fp64 draws in the operand dtype. The stored values are the inputs."""
    return torch.from_numpy(np.ascontiguousarray(x64)).to(DTYPES[dtype])


def normal(seed: int, operand: int, shape, sigma: float, dtype: str) -> torch.Tensor:
    x = _rng(seed, operand).standard_normal(size=shape) * sigma
    return _to_dtype(x, dtype)


def uniform(seed: int, operand: int, shape, lo: float, hi: float, dtype: str) -> torch.Tensor:
    x = _rng(seed, operand).uniform(lo, hi, size=shape)
    return _to_dtype(x, dtype)


def integers(seed: int, operand: int, shape, lo: int, hi: int, dtype: str) -> torch.Tensor:
    """Small integers in [lo, hi]; every product and partial sum of such inputs is exact."""
    x = _rng(seed, operand).integers(lo, hi + 1, size=shape).astype(np.float64)
    return _to_dtype(x, dtype)


# ----------------------------------------------------------------------------- masks


def csr_from_coords(rows: np.ndarray, cols: np.ndarray, m: int):
    """Sort (row, col) pairs row-major and return (row_offsets int32, col_idx int32)."""
    rows = np.asarray(rows, dtype=np.int64)
    cols = np.asarray(cols, dtype=np.int64)
    order = np.lexsort((cols, rows))
    rows, cols = rows[order], cols[order]
    counts = np.bincount(rows, minlength=m) if rows.size else np.zeros(m, dtype=np.int64)
    ro = np.zeros(m + 1, dtype=np.int64)
    np.cumsum(counts, out=ro[1:])
    return ro.astype(np.int32), cols.astype(np.int32)


def uniform_mask(seed: int, m: int, n: int, density: float):
    """Exactly round(density*m*n) positions, uniform without replacement."""
    nnz = int(round(density * m * n))
    pos = _rng(seed, _MASK).choice(m * n, size=nnz, replace=False)
    return csr_from_coords(pos // n, pos % n, m)


def clustered_mask(seed: int, m: int, n: int, density: float, row_frac=0.1, col_frac=0.1):
    """round(density*m*n) positions uniform inside a random row_frac x col_frac block."""
    rng = _rng(seed, _MASK)
    nr = max(1, int(round(row_frac * m)))
    nc = max(1, int(round(col_frac * n)))
    rsel = rng.choice(m, size=nr, replace=False)
    csel = rng.choice(n, size=nc, replace=False)
    nnz = min(int(round(density * m * n)), nr * nc)
    pos = rng.choice(nr * nc, size=nnz, replace=False)
    return csr_from_coords(rsel[pos // nc], csel[pos % nc], m)


def zipf_band_mask(seed: int, m: int, n: int, exponent=1.5, max_len=4096, band=8192):
    """Row lengths Zipf(exponent) resampled until <= max_len (and <= band width); columns
    uniform without replacement inside [i - band, i + band] clipped to the matrix."""
    rng = _rng(seed, _MASK)
    lens = rng.zipf(exponent, size=m)
    bad = lens > max_len
    while bad.any():
        lens[bad] = rng.zipf(exponent, size=int(bad.sum()))
        bad = lens > max_len
    lo = np.maximum(0, np.arange(m) - band)
    hi = np.minimum(n - 1, np.arange(m) + band)
    width = hi - lo + 1
    lens = np.minimum(lens, width)
    ro = np.zeros(m + 1, dtype=np.int64)
    np.cumsum(lens, out=ro[1:])
    cols = np.empty(int(ro[-1]), dtype=np.int64)
    # short rows: draw with replacement, redraw rows that hit a duplicate
    short = np.nonzero(lens <= 64)[0]
    pending = short
    while pending.size:
        l = lens[pending]
        rep = np.repeat(pending, l)
        draw = lo[rep] + (rng.random(rep.size) * width[rep]).astype(np.int64)
        starts = np.repeat(ro[pending], l)
        offs = np.arange(rep.size) - np.repeat(np.cumsum(l) - l, l)
        cols[starts + offs] = draw
        redo = []
        for i in pending:
            seg = cols[ro[i]:ro[i + 1]]
            seg.sort()
            if seg.size > 1 and np.any(seg[1:] == seg[:-1]):
                redo.append(i)
        pending = np.asarray(redo, dtype=np.int64)
    for i in np.nonzero(lens > 64)[0]:
        c = lo[i] + rng.choice(width[i], size=lens[i], replace=False)
        c.sort()
        cols[ro[i]:ro[i + 1]] = c
    return ro.astype(np.int32), cols.astype(np.int32)


def butterfly_mask(m: int, n: int, block=64, stages=3):
    """Block-row r holds blocks at block-columns {c} and {c XOR 2^s : s < stages}, with
    c = r mod (n/block); every block is fully dense."""
    nbc = n // block
    rows, cols = [], []
    for r in range(m // block):
        c = r % nbc
        bcs = sorted({c} | {c ^ (1 << s) for s in range(stages)})
        rr, cc = np.meshgrid(np.arange(block), np.concatenate([np.arange(b * block, (b + 1) * block) for b in bcs]),
                             indexing="ij")
        rows.append((r * block + rr).ravel())
        cols.append(cc.ravel())
    return csr_from_coords(np.concatenate(rows), np.concatenate(cols), m)


# ----------------------------------------------------------------------------- workloads


@dataclass
class Workload:
    name: str
    dtype: str
    m: int
    n: int            # columns of the sparse matrix (= rows of B for SpMM)
    row_offsets: torch.Tensor   # int32 [m+1]
    col_idx: torch.Tensor       # int32 [nnz]
    values: torch.Tensor        # dtype [nnz]
    B: torch.Tensor | None = None    # [n, N]   SpMM dense operand
    A: torch.Tensor | None = None    # [m, kd]  SDDMM left operand
    BT: torch.Tensor | None = None   # [n, kd]  SDDMM right operand (B transposed)
    W: torch.Tensor | None = None    # [m, n]   csr_add dense operand
    meta: dict = field(default_factory=dict)

    @property
    def nnz(self) -> int:
        return int(self.col_idx.numel())


@dataclass(frozen=True)
class Spec:
    """Shape and distribution recipe of one workload."""
    name: str
    seed: int
    dtype: str
    m: int
    n: int
    mask: str                 # uniform | clustered | zipf | butterfly
    density: float = 0.0
    val_dist: tuple = ("normal", 1.0)
    N: int = 0                # SpMM dense columns (0: no SpMM)
    kd: int = 0               # SDDMM inner dimension (0: no SDDMM)
    w_sigma: float | None = None   # csr_add dense W (None: no csr_add)
    act_sigma: float = 1.0
    mask_kw: tuple = ()


SPECS = {
    "tiny": Spec("tiny", 0, "f32", 256, 256, "uniform", 0.05, ("normal", 1.0), N=64, kd=64, w_sigma=1.0),
    "rosa": Spec("rosa", 1, "f16", 4096, 4096, "clustered", 0.01, ("normal", 0.02), N=2048, kd=2048, w_sigma=0.02),
    "llama_mlp": Spec("llama_mlp", 2, "bf16", 11008, 4096, "uniform", 0.005, ("normal", 0.02), N=4096, kd=4096,
                      w_sigma=0.02),
    "zipf": Spec("zipf", 3, "f32", 131072, 131072, "zipf", 0.0, ("uniform", 1.0), N=128, kd=0, w_sigma=None),
    "butterfly": Spec("butterfly", 4, "bf16", 8192, 2048, "butterfly", 0.0, ("normal", 0.02), N=8192, kd=8192,
                      w_sigma=None),
    # narrow-N SpMM (an SpMV regime): 8192 x 8192 at 90 % sparsity, 8 right-hand sides
    "spmv": Spec("spmv", 5, "f16", 8192, 8192, "uniform", 0.1, ("normal", 0.02), N=8, kd=0, w_sigma=None),
}
CONFIG_ORDER = ["tiny", "rosa", "llama_mlp", "zipf", "butterfly"]

# The two MLPs of the HazyResearch/fly issue "Pure torch implementaton of pixelfly" (the T4
# timing comment): layers (in, out) = [(384, 1536), (1536, 384)] with block size 48 and
# [(2048, 8192), (8192, 4096)] with block size 256, inputs [16, 512, in], i.e. 8192 tokens.
# Each layer's weight W (out x in) keeps the butterfly block pattern of the workload above at
# the issue's block size: block-row r holds block-columns c = r mod (in / block) and
# c XOR 2^s for s = 0, 1, 2 (four blocks per block-row). As a workload: m = out, n = in,
# B = X^T (in x tokens) for the forward product Y^T = W X^T, A = dY^T (out x tokens) and
# BT (in x tokens) for the weight gradient on the mask; bf16, values N(0, 0.02),
# activations and gradients N(0, 1).
FLY_MLPS = {
    "fly_small": {"layers": ((384, 1536), (1536, 384)), "block": 48, "tokens": 16 * 512},
    "fly_large": {"layers": ((2048, 8192), (8192, 4096)), "block": 256, "tokens": 16 * 512},
}
for _mlp, (_base, _d) in zip(FLY_MLPS, ((6, FLY_MLPS["fly_small"]), (8, FLY_MLPS["fly_large"]))):
    for _li, (_in, _out) in enumerate(_d["layers"]):
        SPECS[f"{_mlp}_{_li + 1}"] = Spec(f"{_mlp}_{_li + 1}", _base + _li, "bf16", _out, _in, "butterfly", 0.0,
                                          ("normal", 0.02), N=_d["tokens"], kd=_d["tokens"], w_sigma=None,
                                          mask_kw=(("block", _d["block"]),))


def fly_layer_names(mlp: str):
    """Workload names of the MLP's layers, first layer first."""
    return [f"{mlp}_{i + 1}" for i in range(len(FLY_MLPS[mlp]["layers"]))]


def spec(name: str, **over) -> Spec:
    """A named spec, optionally with fields replaced (for scaled-down parity cases)."""
    s = SPECS[name]
    if over:
        d = dict(s.__dict__)
        d.update(over)
        s = Spec(**d)
    return s


def mask_for(s: Spec):
    kw = dict(s.mask_kw)
    if s.mask == "uniform":
        return uniform_mask(s.seed, s.m, s.n, s.density)
    if s.mask == "clustered":
        return clustered_mask(s.seed, s.m, s.n, s.density, **kw)
    if s.mask == "zipf":
        return zipf_band_mask(s.seed, s.m, s.n, **kw)
    if s.mask == "butterfly":
        return butterfly_mask(s.m, s.n, **kw)
    raise ValueError(s.mask)


def generate(s: Spec | str, operands=("B", "A", "BT", "W"), integer_valued=False) -> Workload:
    """Build the workload. ``integer_valued`` replaces every distribution by small integers
    (values in [-4, 4], dense operands in [-2, 2]) so that all results are exact."""
    if isinstance(s, str):
        s = SPECS[s]
    ro, col = mask_for(s)
    nnz = col.size
    if integer_valued:
        vals = integers(s.seed, _VALUES, (nnz,), -4, 4, s.dtype)
    elif s.val_dist[0] == "normal":
        vals = normal(s.seed, _VALUES, (nnz,), s.val_dist[1], s.dtype)
    else:
        vals = uniform(s.seed, _VALUES, (nnz,), -s.val_dist[1], s.val_dist[1], s.dtype)

    def dense(op, shape, sigma):
        if integer_valued:
            return integers(s.seed, op, shape, -2, 2, s.dtype)
        return normal(s.seed, op, shape, sigma, s.dtype)

    w = Workload(s.name, s.dtype, s.m, s.n, torch.from_numpy(ro), torch.from_numpy(col), vals,
                 meta={"spec": s, "integer_valued": integer_valued})
    if s.N and "B" in operands:
        w.B = dense(_B, (s.n, s.N), s.act_sigma)
    if s.kd and "A" in operands:
        w.A = dense(_A, (s.m, s.kd), s.act_sigma)
    if s.kd and "BT" in operands:
        w.BT = dense(_BT, (s.n, s.kd), s.act_sigma)
    if s.w_sigma is not None and "W" in operands:
        w.W = dense(_W, (s.m, s.n), s.w_sigma)
    return w


def random_permutation(seed: int, m: int) -> torch.Tensor:
    """A seeded permutation of 0..m-1 (int32), for tests that pass an unsorted row_idx."""
    return torch.from_numpy(_rng(seed, 99).permutation(m).astype(np.int32))
