"""A sparse linear layer on a fixed CSR mask, forward and backward on this package's kernels.

HazyResearch/fly issue "Pure torch implementaton of pixelfly": a pixelfly layer is a
linear layer whose weight keeps only a butterfly pattern of dense blocks; the issue times
its forward and backward against nn.Linear. spops README ("Sparse Operations (spops)"):
SpMM is the forward product, SDDMM the weight gradient on the mask, and csr_transpose
gives the input gradient (torchsparsegradutils README, "Basic Sparse Matrix
Multiplication": both gradients of a sparse product keep the sparsity).

Activations are feature-major (features x tokens), the layout in which every product is
one call with no transposed copies:
    forward   Y^T  = W X^T                 spmm
    dW        dW   = (dY^T X) on the mask  sddmm(A = dY^T, BT = X^T)
    dX        dX^T = W^T dY^T              spmm of the cached transpose of W
The row permutation, the mask plan and the transpose's structure are built once per mask.
"""
from __future__ import annotations

import torch

from . import csr_transpose, permute_values, plan_build, sddmm, sort_rows, spmm


class SparseLinearFunction(torch.autograd.Function):
    @staticmethod
    def forward(ctx, values, Xt, layer):
        Yt = spmm(values, layer.row_offsets, layer.row_idx, layer.col_idx, Xt, layer.out_features, plan=layer.plan)
        ctx.save_for_backward(values, Xt)
        ctx.layer = layer
        return Yt

    @staticmethod
    def backward(ctx, dYt):
        values, Xt = ctx.saved_tensors
        L = ctx.layer
        dYt = dYt.contiguous()
        d_values = d_Xt = None
        if ctx.needs_input_grad[0]:
            d_values = sddmm(L.row_offsets, L.row_idx, L.col_idx, dYt, Xt, plan=L.plan)
        if ctx.needs_input_grad[1]:
            vt = permute_values(values, L.transpose)
            d_Xt = spmm(vt, L.transpose.row_offsets, L.row_idx_t, L.transpose.col_idx, dYt, L.in_features,
                        plan=L.plan_t)
        return d_values, d_Xt, None


class SparseLinear(torch.nn.Module):
    """Y^T = W X^T with W (out_features x in_features) stored as the values of a fixed CSR
    mask (row_offsets int32, col_idx int16/int32); inputs and outputs are feature-major
    (features x tokens), fp16 or bf16 (fp32 runs the general kernels)."""

    def __init__(self, row_offsets: torch.Tensor, col_idx: torch.Tensor, values: torch.Tensor, in_features: int):
        super().__init__()
        self.out_features = row_offsets.numel() - 1
        self.in_features = int(in_features)
        self.register_buffer("row_offsets", row_offsets)
        self.register_buffer("col_idx", col_idx)
        self.values = torch.nn.Parameter(values)
        self.row_idx = sort_rows(row_offsets, nnz=col_idx.numel(), index_dtype=col_idx.dtype)
        self.plan = plan_build(row_offsets, self.row_idx, col_idx, self.in_features)
        self.transpose = csr_transpose(None, row_offsets, col_idx, self.in_features)
        self.row_idx_t = sort_rows(self.transpose.row_offsets, nnz=col_idx.numel(), index_dtype=col_idx.dtype)
        self.plan_t = plan_build(self.transpose.row_offsets, self.row_idx_t, self.transpose.col_idx,
                                 self.out_features)

    def forward(self, Xt: torch.Tensor) -> torch.Tensor:
        return SparseLinearFunction.apply(self.values, Xt.contiguous(), self)
