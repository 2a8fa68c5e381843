// Internal launcher interface between the C-ABI layer (abi.cu) and the kernel files.
// Nothing here is exported from the shared library.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

namespace spops {

enum DType { kF32 = 0, kF16 = 1, kBF16 = 2 };
enum IType { kIdx16 = 0, kIdx32 = 1 };

struct DeviceProps {
    int device = -1;
    int sm_count = 0;
    int max_smem_optin = 0;
    int cc_major = 0, cc_minor = 0;
};

// Properties of the current device (queried once per device).
const DeviceProps& device_props();
// Device address of this library's error word on the current device.
int* device_error_word();
// Add n to the process-wide count of kernels this library has launched.
void count_launches(int n);
// A second stream for work that is independent of what follows on `s` (the general row
// kernels beside the tensor-core panels). side_fork records an event on s and makes the
// calling thread's side stream for the current device wait for it; side_join makes s wait
// for everything queued on the side stream since. Both are captured into CUDA graphs as a
// fork and a join. side_fork returns nullptr (run everything on s) if no side stream can
// be made.
cudaStream_t side_fork(cudaStream_t s);
cudaError_t side_join(cudaStream_t s);
// Destroy the calling thread's side streams and events (spops_release_streams).
cudaError_t release_sides();
// Record the calling thread's spops_last_error() text (printf format) and return status.
int set_last_error(int status, const char* fmt, ...);

// Launch with programmatic stream serialization: the kernel may start while the previous
// kernel in the stream finishes (its CTAs call pdl_wait before reading earlier results), so
// consecutive kernels overlap launch latency. Captured into CUDA graphs as programmatic edges.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// launch_pdl with the grid divided into thread-block clusters of `cluster` CTAs along x
// (grid.x a multiple of cluster).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, unsigned cluster,
                               cudaStream_t s, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

inline size_t dtype_size(int dt) { return dt == kF32 ? 4 : 2; }
inline size_t itype_size(int it) { return it == kIdx16 ? 2 : 4; }
__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Row-bin thresholds used by the operators (rows with nnz >= threshold are "long").
constexpr int32_t kSpmmLongRow = 256;
constexpr int32_t kSddmmLongRow = 64;

// csr_add.cu
cudaError_t launch_csr_add(int dt, int it, const void* vals, const int32_t* ro, const void* col, int32_t m,
                           int32_t n, int32_t nnz, const void* B, void* C, cudaStream_t s);

// sort_rows.cu
size_t sort_rows_workspace_bytes(int32_t m);
cudaError_t launch_sort_rows(const int32_t* ro, int32_t m, int32_t nnz, void* row_idx_out, int it, void* ws,
                             cudaStream_t s);
cudaError_t launch_row_bins(const int32_t* ro, int32_t m, int32_t t_long, int32_t* bins, cudaStream_t s);
cudaError_t launch_check_csr(const int32_t* ro, const void* col, const void* row_idx, int it, int32_t m, int32_t n,
                             int32_t nnz, uint32_t* perm_bits, int* err, cudaStream_t s);

// spmm.cu
cudaError_t launch_spmm_general(int dt, int it, const void* vals, const int32_t* ro, const void* row_idx,
                                const void* col, int32_t m, int32_t k, const void* B, int32_t n, void* C,
                                const int32_t* bins, const uint8_t* skip_panels, const int32_t* order,
                                cudaStream_t s);

// sddmm.cu
cudaError_t launch_sddmm_general(int dt, int it, const int32_t* ro, const void* row_idx, const void* col, int32_t m,
                                 int32_t n, int32_t kd, const void* A, const void* BT, void* out,
                                 const int32_t* bins, const uint8_t* skip_panels, const int32_t* order,
                                 cudaStream_t s);

// Rows are grouped in panels of kPanelRows consecutive positions of the plan's row order
// (row_idx, or row_idx refined by column pattern); the general kernels walk the same order
// (`order`, the plan's row at each position; row_idx when null) and skip positions whose
// panel flag in skip_panels is set (handled on tensor cores).
constexpr int kPanelRows = 128;

// transpose.cu
size_t csr_transpose_workspace_bytes(int32_t nnz);
cudaError_t launch_csr_transpose(int dt, int it, const int32_t* ro, const void* col, const void* val, int32_t m,
                                 int32_t n, int32_t nnz, int32_t* ro_t, void* row_t, void* val_t, int32_t* perm,
                                 void* ws, cudaStream_t s);
cudaError_t launch_permute_values(int dt, const void* val, const int32_t* perm, int32_t nnz, void* val_t,
                                  cudaStream_t s);

// adam.cu
cudaError_t launch_masked_adam(int gdt, float* param, float* exp_avg, float* exp_avg_sq, const void* grad,
                               int64_t count, int32_t step, double lr, double beta1, double beta2, double eps,
                               int maximize, cudaStream_t s);
cudaError_t launch_masked_adam_csr(int gdt, int it, float* param, float* exp_avg, float* exp_avg_sq, const void* grad,
                                   const int32_t* ro, const void* col, int32_t m, int32_t n, int32_t step, double lr,
                                   double beta1, double beta2, double eps, int maximize, cudaStream_t s);

// selftest.cu: one thread waits on an mbarrier nothing arrives on, with a limit of limit_ns;
// the wait gives up and records kDevErrMbarTimeout. waited_ns (device, may be null) receives
// the time the wait took.
cudaError_t launch_wait_selftest(uint64_t limit_ns, unsigned long long* waited_ns, cudaStream_t s);

}  // namespace spops
