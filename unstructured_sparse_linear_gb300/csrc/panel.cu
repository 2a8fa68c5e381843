// Operator dispatch. This revision routes every operator to the general row kernels.
#include "internal.h"
#include "panel.h"

namespace spops {

size_t panel_spmm_workspace_bytes(int32_t, int32_t, int32_t, int32_t, int, int) { return 0; }
size_t panel_sddmm_workspace_bytes(int32_t, int32_t, int32_t, int32_t, int, int) { return 0; }

cudaError_t launch_spmm(int dt, int it, const void* vals, const int32_t* ro, const void* row_idx, const void* col,
                        int32_t m, int32_t k, int32_t nnz, const void* B, int32_t n, void* C, const int32_t* bins,
                        void* ws, cudaStream_t s) {
    (void)nnz;
    (void)ws;
    return launch_spmm_general(dt, it, vals, ro, row_idx, col, m, k, B, n, C, bins, s);
}

cudaError_t launch_sddmm(int dt, int it, const int32_t* ro, const void* row_idx, const void* col, int32_t m,
                         int32_t n, int32_t kd, int32_t nnz, const void* A, const void* BT, void* out,
                         bool structure_aware, const int32_t* bins, void* ws, cudaStream_t s) {
    (void)nnz;
    (void)ws;
    (void)structure_aware;
    return launch_sddmm_general(dt, it, ro, row_idx, col, m, n, kd, A, BT, out, bins, s);
}

}  // namespace spops
