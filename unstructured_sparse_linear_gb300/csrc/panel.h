// Operator dispatch between the general row kernels and the dense-panel (tensor core)
// path, and the workspace the panel path needs.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace spops {

size_t panel_spmm_workspace_bytes(int32_t m, int32_t k, int32_t n, int32_t nnz, int dt, int it);
size_t panel_sddmm_workspace_bytes(int32_t m, int32_t n, int32_t kd, int32_t nnz, int dt, int it);

// Build the panel plan alone and write {dense panels, entries in dense panels, SDDMM
// tiles, panels} to stats (device int32[4]). Requires n <= 65536.
size_t panel_plan_workspace_bytes(int32_t m, int32_t nnz);
cudaError_t launch_panel_plan(int it, const int32_t* ro, const void* row_idx, const void* col, int32_t m, int32_t n,
                              int32_t nnz, int32_t* stats, void* ws, cudaStream_t s);

// bins: device int32[4] already written by the row-bins kernel on the same stream.
cudaError_t launch_spmm(int dt, int it, const void* vals, const int32_t* ro, const void* row_idx, const void* col,
                        int32_t m, int32_t k, int32_t nnz, const void* B, int32_t n, void* C, const int32_t* bins,
                        void* ws, bool allow_panels, cudaStream_t s);
cudaError_t launch_sddmm(int dt, int it, const int32_t* ro, const void* row_idx, const void* col, int32_t m,
                         int32_t n, int32_t kd, int32_t nnz, const void* A, const void* BT, void* out,
                         bool structure_aware, const int32_t* bins, void* ws, cudaStream_t s);

}  // namespace spops
