// spops_sort_rows_static: the row permutation without any caller-provided or
// library-allocated device memory.
//
// Some callers cannot allocate device memory at the point where they need row_idx: a
// plugin inside a host application that owns every device allocation and hands out no
// allocator, or a latency-critical loop that must not call cudaMalloc (it can synchronize
// the device). For them this entry point runs the same radix sort as spops_sort_rows, with
// its scratch in a file-scope __device__ array instead of a workspace argument.
//
// The array holds the scratch for at most kStaticSortMaxRows rows (about 2.1 MB). Every GPU
// that loads this library keeps that much device memory reserved until the process exits.
// All calls on a device share the one array: calls whose work overlaps on the GPU (for
// example on two streams without ordering between them) race on it. The sort writes every
// scratch word it later reads, so nothing needs clearing between calls.
#include <mutex>

#include "../../include/spops_gb300.h"
#include "common.cuh"
#include "internal.h"

namespace spops {
namespace {

constexpr int32_t kStaticSortMaxRows = 131072;
// Same layout as the workspace of spops_sort_rows: four arrays of m 32-bit words (each
// rounded up to 256 bytes) and the digit histograms of ceil(m / 2048) blocks.
constexpr size_t kStaticSortBytes = 4 * ((size_t)kStaticSortMaxRows * 4) + ((kStaticSortMaxRows + 2047) / 2048) * 256 * 4;

static __device__ __align__(256) unsigned char g_sort_scratch[kStaticSortBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mutex;

// Device address of g_sort_scratch on the current device, looked up once per device.
// In host code the name g_sort_scratch is only a host-side stand-in for the symbol, so the
// address must come from cudaGetSymbolAddress with the device current.
cudaError_t scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_sort_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace
}  // namespace spops

using namespace spops;

extern "C" {

int32_t spops_sort_rows_static_max_rows(void) { return kStaticSortMaxRows; }

int spops_sort_rows_static(const int32_t* row_offsets, int32_t m, int32_t nnz, void* row_idx_out, int itype,
                           void* stream) {
    if (itype != SPOPS_IDX16 && itype != SPOPS_IDX32)
        return set_last_error(SPOPS_ERR_INVALID_ARG, "itype %d is not a spops_itype", itype);
    if (m < 0 || nnz < 0) return set_last_error(SPOPS_ERR_INVALID_ARG, "negative size (m=%d nnz=%d)", m, nnz);
    if (m > kStaticSortMaxRows)
        return set_last_error(SPOPS_ERR_UNSUPPORTED,
                              "sort_rows_static: m=%d exceeds the %d rows its static scratch holds; "
                              "use spops_sort_rows with a workspace",
                              m, kStaticSortMaxRows);
    if (itype == SPOPS_IDX16 && m > 32768)
        return set_last_error(SPOPS_ERR_UNSUPPORTED, "int16 row_idx holds at most 32768 rows (m=%d)", m);
    if (m == 0) return set_last_error(SPOPS_OK, "");
    if (!row_offsets || !row_idx_out)
        return set_last_error(SPOPS_ERR_INVALID_ARG, "row_offsets or row_idx_out is NULL");
    if ((uintptr_t)row_offsets % 4 || (uintptr_t)row_idx_out % (itype == SPOPS_IDX16 ? 2 : 4))
        return set_last_error(SPOPS_ERR_INVALID_ARG, "misaligned row_offsets or row_idx_out");
    if (sort_rows_workspace_bytes(m) > kStaticSortBytes)
        return set_last_error(SPOPS_ERR_UNSUPPORTED, "sort_rows_static: scratch for m=%d does not fit", m);
    void* scratch = nullptr;
    cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess)
        return set_last_error(SPOPS_ERR_CUDA, "sort_rows_static: scratch address: %s", cudaGetErrorString(e));
    e = launch_sort_rows(row_offsets, m, nnz, row_idx_out, itype, scratch, (cudaStream_t)stream);
    if (e != cudaSuccess) return set_last_error(SPOPS_ERR_CUDA, "sort_rows_static launch: %s", cudaGetErrorString(e));
    return set_last_error(SPOPS_OK, "");
}

}  // extern "C"
