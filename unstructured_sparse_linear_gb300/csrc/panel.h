// Operator dispatch between the general row kernels and the dense-panel (tensor core)
// path, and the workspace each operator needs.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace spops {

// Workspace of one call when it builds its own plan (a caller plan only lowers the need).
size_t spmm_workspace_bytes(int32_t m, int32_t k, int32_t n, int32_t nnz, int dt);
size_t sddmm_workspace_bytes(int32_t m, int32_t n, int32_t kd, int32_t nnz, int dt, bool structure_aware);

// plan: a mask plan built by launch_plan_build for this mask, or nullptr to build one in ws.
cudaError_t launch_spmm(int dt, int it, const void* vals, const int32_t* ro, const void* row_idx, const void* col,
                        int32_t m, int32_t k, int32_t nnz, const void* B, int32_t n, void* C, const void* plan,
                        void* ws, bool allow_panels, cudaStream_t s);
cudaError_t launch_sddmm(int dt, int it, const int32_t* ro, const void* row_idx, const void* col, int32_t m,
                         int32_t n, int32_t kd, int32_t nnz, const void* A, const void* BT, void* out,
                         bool structure_aware, const void* plan, void* ws, cudaStream_t s);

}  // namespace spops
