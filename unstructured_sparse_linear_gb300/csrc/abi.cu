// C-ABI entry points: host-side argument validation, workspace carving and dispatch to
// the kernels. Declarations and the contract of every call are in include/spops_gb300.h.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "../../include/spops_gb300.h"
#include "common.cuh"
#include "internal.h"
#include "panel.h"
#include "plan.h"

namespace spops {

// The device error word: one per device (a __device__ variable exists once per device
// context). Kernels receive its address; spops_get_device_error reads and clears it.
static __device__ int g_device_error;

namespace {

constexpr int kMaxDevices = 64;
DeviceProps g_props[kMaxDevices];
// Device address of g_device_error per device, looked up once with the device current and
// kept for the life of the process (it does not survive cudaDeviceReset).
int* g_err_addr[kMaxDevices];
std::mutex g_err_mutex;
thread_local char g_last_error[320];
std::atomic<uint64_t> g_launches{0};

int current_device() {
    int d = 0;
    if (cudaGetDevice(&d) != cudaSuccess) return -1;
    return d;
}

}  // namespace

const DeviceProps& device_props() {
    static DeviceProps none;
    const int d = current_device();
    if (d < 0 || d >= kMaxDevices) return none;
    DeviceProps& p = g_props[d];
    if (p.device != d) {
        cudaDeviceGetAttribute(&p.sm_count, cudaDevAttrMultiProcessorCount, d);
        cudaDeviceGetAttribute(&p.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, d);
        cudaDeviceGetAttribute(&p.cc_major, cudaDevAttrComputeCapabilityMajor, d);
        cudaDeviceGetAttribute(&p.cc_minor, cudaDevAttrComputeCapabilityMinor, d);
        if (p.sm_count <= 0) p.sm_count = 1;
        p.device = d;
    }
    return p;
}

int* device_error_word() {
    const int d = current_device();
    if (d < 0 || d >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_err_mutex);
    if (!g_err_addr[d]) {
        void* addr = nullptr;
        if (cudaGetSymbolAddress(&addr, g_device_error) != cudaSuccess) return nullptr;
        g_err_addr[d] = static_cast<int*>(addr);
    }
    return g_err_addr[d];
}

void count_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

namespace {
// One side stream per (device, caller stream), so operators queued on different streams do
// not serialize on a shared side stream.
struct Side {
    int device = -1;
    cudaStream_t caller = nullptr;
    cudaStream_t stream = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};
constexpr int kMaxSides = 8;
thread_local Side g_side[kMaxSides];

Side* find_side(int d, cudaStream_t s) {
    for (Side& sd : g_side)
        if (sd.stream && sd.device == d && sd.caller == s) return &sd;
    return nullptr;
}
}  // namespace

cudaStream_t side_fork(cudaStream_t s) {
    const int d = current_device();
    if (d < 0) return nullptr;
    Side* sd = find_side(d, s);
    if (!sd) {
        // Streams are not created while s is being captured into a graph (no fork then).
        cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(s, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone) {
            cudaGetLastError();
            return nullptr;
        }
        for (Side& x : g_side)
            if (!x.stream) {
                sd = &x;
                break;
            }
        if (!sd) return nullptr;
        if (cudaStreamCreateWithFlags(&sd->stream, cudaStreamNonBlocking) != cudaSuccess) {
            cudaGetLastError();
            sd->stream = nullptr;
            return nullptr;
        }
        sd->fork = sd->join = nullptr;
        if (cudaEventCreateWithFlags(&sd->fork, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&sd->join, cudaEventDisableTiming) != cudaSuccess) {
            cudaGetLastError();
            if (sd->fork) cudaEventDestroy(sd->fork);
            cudaStreamDestroy(sd->stream);
            sd->stream = nullptr;
            return nullptr;
        }
        sd->device = d;
        sd->caller = s;
    }
    if (cudaEventRecord(sd->fork, s) != cudaSuccess || cudaStreamWaitEvent(sd->stream, sd->fork, 0) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    return sd->stream;
}

// Destroy the calling thread's side streams and their events (work already queued on them
// still runs to completion; the CUDA runtime releases the stream afterwards).
cudaError_t release_sides() {
    cudaError_t first = cudaSuccess;
    for (Side& sd : g_side) {
        if (!sd.stream) continue;
        cudaError_t e = cudaEventDestroy(sd.fork);
        if (first == cudaSuccess) first = e;
        e = cudaEventDestroy(sd.join);
        if (first == cudaSuccess) first = e;
        e = cudaStreamDestroy(sd.stream);
        if (first == cudaSuccess) first = e;
        sd = Side{};
    }
    return first;
}

cudaError_t side_join(cudaStream_t s) {
    Side* sd = find_side(current_device(), s);
    if (!sd) return cudaErrorInvalidResourceHandle;
    cudaError_t e = cudaEventRecord(sd->join, sd->stream);
    if (e != cudaSuccess) return e;
    return cudaStreamWaitEvent(s, sd->join, 0);
}

int set_last_error(int status, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
    return status;
}

}  // namespace spops

using namespace spops;

namespace {

int fail(int status, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
    return status;
}

int ok() {
    g_last_error[0] = 0;
    return SPOPS_OK;
}

int cuda_status(cudaError_t e, const char* what) {
    if (e == cudaSuccess) return ok();
    return fail(SPOPS_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Checks shared by the CSR-consuming calls. Returns SPOPS_OK or an error status.
int check_common(int itype, int dtype, int32_t m, int32_t ncols, int32_t nnz, const void* vals,
                 const int32_t* ro, const void* row_idx, const void* col, bool need_vals, bool need_row_idx) {
    if (dtype < SPOPS_F32 || dtype > SPOPS_BF16) return fail(SPOPS_ERR_INVALID_ARG, "dtype %d is not a spops_dtype", dtype);
    if (itype != SPOPS_IDX16 && itype != SPOPS_IDX32)
        return fail(SPOPS_ERR_INVALID_ARG, "itype %d is not a spops_itype", itype);
    if (m < 0 || ncols < 0 || nnz < 0) return fail(SPOPS_ERR_INVALID_ARG, "negative size (m=%d n=%d nnz=%d)", m, ncols, nnz);
    if (itype == SPOPS_IDX16 && (m > 32768 || ncols > 32768))
        return fail(SPOPS_ERR_UNSUPPORTED, "int16 indices hold at most 32768 rows/columns (m=%d n=%d); use SPOPS_IDX32",
                    m, ncols);
    if (!ro) return fail(SPOPS_ERR_INVALID_ARG, "row_offsets is NULL");
    if (!aligned(ro, 4)) return fail(SPOPS_ERR_INVALID_ARG, "row_offsets is not 4-byte aligned");
    const size_t is = itype_size(itype), ds = dtype_size(dtype);
    if (nnz > 0) {
        if (!col) return fail(SPOPS_ERR_INVALID_ARG, "col_idx is NULL with nnz=%d", nnz);
        if (!aligned(col, is)) return fail(SPOPS_ERR_INVALID_ARG, "col_idx is not aligned to its index size");
        if (need_vals && !vals) return fail(SPOPS_ERR_INVALID_ARG, "values is NULL with nnz=%d", nnz);
        if (need_vals && !aligned(vals, ds)) return fail(SPOPS_ERR_INVALID_ARG, "values is not aligned to its dtype");
    }
    if (need_row_idx && m > 0) {
        if (!row_idx) return fail(SPOPS_ERR_INVALID_ARG, "row_idx is NULL with m=%d", m);
        if (!aligned(row_idx, is)) return fail(SPOPS_ERR_INVALID_ARG, "row_idx is not aligned to its index size");
    }
    return SPOPS_OK;
}

bool overlaps(const void* a, size_t abytes, const void* b, size_t bbytes) {
    if (!a || !b || !abytes || !bbytes) return false;
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + bbytes && y < x + abytes;
}

int check_adam(const float* param, const float* exp_avg, const float* exp_avg_sq, const void* grad, int grad_dtype,
               int64_t entries, int64_t grad_count, int32_t step, double lr, double beta1, double beta2, double eps) {
    if (grad_dtype < SPOPS_F32 || grad_dtype > SPOPS_BF16)
        return fail(SPOPS_ERR_INVALID_ARG, "grad_dtype %d is not a spops_dtype", grad_dtype);
    if (step < 1) return fail(SPOPS_ERR_INVALID_ARG, "step must be >= 1 (got %d)", step);
    if (!(lr >= 0.0) || !(eps >= 0.0)) return fail(SPOPS_ERR_INVALID_ARG, "need lr >= 0 and eps >= 0");
    if (!(beta1 >= 0.0 && beta1 < 1.0) || !(beta2 >= 0.0 && beta2 < 1.0))
        return fail(SPOPS_ERR_INVALID_ARG, "betas must lie in [0, 1)");
    if (entries == 0 || grad_count == 0) return SPOPS_OK;
    if (!param || !exp_avg || !exp_avg_sq || !grad) return fail(SPOPS_ERR_INVALID_ARG, "a state or gradient pointer is NULL");
    const size_t gs = dtype_size(grad_dtype);
    if (!aligned(param, 4) || !aligned(exp_avg, 4) || !aligned(exp_avg_sq, 4) || !aligned(grad, gs))
        return fail(SPOPS_ERR_INVALID_ARG, "misaligned state or gradient");
    const size_t sb = (size_t)entries * 4, gb = (size_t)grad_count * gs;
    if (overlaps(param, sb, exp_avg, sb) || overlaps(param, sb, exp_avg_sq, sb) || overlaps(exp_avg, sb, exp_avg_sq, sb) ||
        overlaps(param, sb, grad, gb) || overlaps(exp_avg, sb, grad, gb) || overlaps(exp_avg_sq, sb, grad, gb))
        return fail(SPOPS_ERR_INVALID_ARG, "param, exp_avg, exp_avg_sq and grad must not overlap");
    return SPOPS_OK;
}

}  // namespace

extern "C" {

const char* spops_status_string(int status) {
    switch (status) {
        case SPOPS_OK: return "SPOPS_OK";
        case SPOPS_ERR_INVALID_ARG: return "SPOPS_ERR_INVALID_ARG";
        case SPOPS_ERR_UNSUPPORTED: return "SPOPS_ERR_UNSUPPORTED";
        case SPOPS_ERR_WORKSPACE: return "SPOPS_ERR_WORKSPACE";
        case SPOPS_ERR_CUDA: return "SPOPS_ERR_CUDA";
        case SPOPS_ERR_DEVICE_CHECK: return "SPOPS_ERR_DEVICE_CHECK";
        default: return "SPOPS_UNKNOWN_STATUS";
    }
}

const char* spops_last_error(void) { return g_last_error; }

const char* spops_version(void) { return "spops_gb300 0.1 sm_103a"; }

uint64_t spops_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

size_t spops_sort_rows_workspace_size(int32_t m) { return m > 0 ? sort_rows_workspace_bytes(m) : 16; }

int spops_sort_rows(const int32_t* row_offsets, int32_t m, int32_t nnz, void* row_idx_out, int itype,
                    void* workspace, size_t ws_bytes, void* stream) {
    if (itype != SPOPS_IDX16 && itype != SPOPS_IDX32) return fail(SPOPS_ERR_INVALID_ARG, "itype %d is not a spops_itype", itype);
    if (m < 0 || nnz < 0) return fail(SPOPS_ERR_INVALID_ARG, "negative size (m=%d nnz=%d)", m, nnz);
    if (itype == SPOPS_IDX16 && m > 32768) return fail(SPOPS_ERR_UNSUPPORTED, "int16 row_idx holds at most 32768 rows (m=%d)", m);
    if (m == 0) return ok();
    if (!row_offsets || !row_idx_out) return fail(SPOPS_ERR_INVALID_ARG, "row_offsets or row_idx_out is NULL");
    if (!aligned(row_offsets, 4) || !aligned(row_idx_out, itype_size(itype)))
        return fail(SPOPS_ERR_INVALID_ARG, "misaligned row_offsets or row_idx_out");
    if (!workspace || !aligned(workspace, 16) || ws_bytes < spops_sort_rows_workspace_size(m))
        return fail(SPOPS_ERR_WORKSPACE, "sort_rows needs a 16-byte aligned workspace of %zu bytes (got %zu)",
                    spops_sort_rows_workspace_size(m), ws_bytes);
    return cuda_status(launch_sort_rows(row_offsets, m, nnz, row_idx_out, itype, workspace, (cudaStream_t)stream),
                       "sort_rows launch");
}

int spops_row_bins(const int32_t* row_offsets, int32_t m, int32_t t_long, int32_t* bins_out, void* stream) {
    if (m < 0 || t_long < 1) return fail(SPOPS_ERR_INVALID_ARG, "need m >= 0 and t_long >= 1 (m=%d t_long=%d)", m, t_long);
    if (!row_offsets || !bins_out) return fail(SPOPS_ERR_INVALID_ARG, "row_offsets or bins_out is NULL");
    if (!aligned(row_offsets, 4) || !aligned(bins_out, 4)) return fail(SPOPS_ERR_INVALID_ARG, "misaligned pointer");
    return cuda_status(launch_row_bins(row_offsets, m, t_long, bins_out, (cudaStream_t)stream), "row_bins launch");
}

size_t spops_plan_size(int32_t m, int32_t n, int32_t nnz) {
    if (m < 0 || n < 0 || nnz < 0) return 0;
    return plan_bytes(m, n, nnz) + 1024;
}

int spops_plan_build(const int32_t* row_offsets, const void* row_idx, const void* col_idx, int itype, int32_t m,
                     int32_t n, int32_t nnz, void* plan, size_t plan_size, void* stream) {
    int st = check_common(itype, SPOPS_F16, m, n, nnz, nullptr, row_offsets, row_idx, col_idx, false, true);
    if (st != SPOPS_OK) return st;
    if (m == 0) return ok();
    if (!plan || !aligned(plan, 1024) || plan_size < spops_plan_size(m, n, nnz))
        return fail(SPOPS_ERR_WORKSPACE, "plan needs a 1024-byte aligned buffer of %zu bytes (got %zu)",
                    spops_plan_size(m, n, nnz), plan_size);
    const PlanView v = plan_view(plan, m, n, nnz);
    return cuda_status(launch_plan_build(itype, row_offsets, row_idx, col_idx, v,
                                         (int64_t)spmm_image_budget_elems(m, nnz), (cudaStream_t)stream),
                       "plan_build launch");
}

int spops_plan_stats(const void* plan, int32_t m, int32_t n, int32_t nnz, int32_t* stats_out, void* stream) {
    if (m <= 0 || n < 0 || nnz < 0) return fail(SPOPS_ERR_INVALID_ARG, "bad sizes (m=%d n=%d nnz=%d)", m, n, nnz);
    if (!plan || !aligned(plan, 1024)) return fail(SPOPS_ERR_INVALID_ARG, "plan is NULL or not 1024-byte aligned");
    if (!stats_out || !aligned(stats_out, 4)) return fail(SPOPS_ERR_INVALID_ARG, "stats_out is NULL or misaligned");
    const PlanView v = plan_view(const_cast<void*>(plan), m, n, nnz);
    return cuda_status(launch_plan_stats(v, stats_out, (cudaStream_t)stream), "plan_stats launch");
}

int spops_plan_row_order(const void* plan, int32_t m, int32_t n, int32_t nnz, int32_t* order_out, void* stream) {
    if (m <= 0 || n < 0 || nnz < 0) return fail(SPOPS_ERR_INVALID_ARG, "bad sizes (m=%d n=%d nnz=%d)", m, n, nnz);
    if (!plan || !aligned(plan, 1024)) return fail(SPOPS_ERR_INVALID_ARG, "plan is NULL or not 1024-byte aligned");
    if (!order_out || !aligned(order_out, 4)) return fail(SPOPS_ERR_INVALID_ARG, "order_out is NULL or misaligned");
    const PlanView v = plan_view(const_cast<void*>(plan), m, n, nnz);
    if (!v.panels) return fail(SPOPS_ERR_UNSUPPORTED, "the plan of an m x %d mask has no panels (n > 65536)", n);
    return cuda_status(cudaMemcpyAsync(order_out, v.prow, (size_t)m * sizeof(int32_t), cudaMemcpyDeviceToDevice,
                                       (cudaStream_t)stream),
                       "plan_row_order copy");
}

size_t spops_spmm_workspace_size(int32_t m, int32_t k, int32_t n, int32_t nnz, int dtype, int itype) {
    (void)itype;
    return spmm_workspace_bytes(m, k, n, nnz, dtype);
}

int spops_spmm(const void* A_val, const int32_t* row_offsets, const void* row_idx, const void* col_idx, int itype,
               int dtype, int32_t m, int32_t k, int32_t nnz, const void* B, int32_t n, void* C, int path,
               const void* plan, void* workspace, size_t ws_bytes, void* stream) {
    int st = check_common(itype, dtype, m, k, nnz, A_val, row_offsets, row_idx, col_idx, true, true);
    if (st != SPOPS_OK) return st;
    if (path != SPOPS_SPMM_AUTO && path != SPOPS_SPMM_GENERAL)
        return fail(SPOPS_ERR_INVALID_ARG, "path %d is not a spops_spmm_path", path);
    if (n < 0) return fail(SPOPS_ERR_INVALID_ARG, "negative n=%d", n);
    if ((int64_t)m * n == 0) return ok();
    const size_t ds = dtype_size(dtype);
    if (!C || !aligned(C, ds)) return fail(SPOPS_ERR_INVALID_ARG, "C is NULL or misaligned");
    if ((int64_t)k * n > 0 && (!B || !aligned(B, ds))) return fail(SPOPS_ERR_INVALID_ARG, "B is NULL or misaligned");
    if (overlaps(C, (size_t)m * n * ds, B, (size_t)k * n * ds)) return fail(SPOPS_ERR_INVALID_ARG, "C overlaps B");
    if (plan && !aligned(plan, 1024)) return fail(SPOPS_ERR_INVALID_ARG, "plan is not 1024-byte aligned");
    const size_t need = spops_spmm_workspace_size(m, k, n, nnz, dtype, itype);
    if (!workspace || !aligned(workspace, 16) || ws_bytes < need)
        return fail(SPOPS_ERR_WORKSPACE, "spmm needs a 16-byte aligned workspace of %zu bytes (got %zu)", need, ws_bytes);
    return cuda_status(launch_spmm(dtype, itype, A_val, row_offsets, row_idx, col_idx, m, k, nnz, B, n, C, plan,
                                   workspace, path == SPOPS_SPMM_AUTO, (cudaStream_t)stream),
                       "spmm launch");
}

size_t spops_sddmm_workspace_size(int32_t m, int32_t n, int32_t kd, int32_t nnz, int dtype, int itype, int backend) {
    (void)itype;
    return sddmm_workspace_bytes(m, n, kd, nnz, dtype, backend == SPOPS_SDDMM_STRUCTURE_AWARE);
}

int spops_sddmm(const int32_t* out_row_offsets, const void* out_row_idx, const void* out_col_idx, int itype,
                int dtype, int32_t m, int32_t n, int32_t kd, int32_t nnz, const void* A, const void* BT,
                void* out_val, int backend, const void* plan, void* workspace, size_t ws_bytes, void* stream) {
    int st = check_common(itype, dtype, m, n, nnz, out_val, out_row_offsets, out_row_idx, out_col_idx, true, true);
    if (st != SPOPS_OK) return st;
    if (backend != SPOPS_SDDMM_STRUCTURE_AWARE && backend != SPOPS_SDDMM_GENERAL)
        return fail(SPOPS_ERR_INVALID_ARG, "backend %d is not a spops_sddmm_backend", backend);
    if (kd < 0) return fail(SPOPS_ERR_INVALID_ARG, "negative kd=%d", kd);
    if (nnz == 0) return ok();
    const size_t ds = dtype_size(dtype);
    if (kd > 0 && (!A || !BT || !aligned(A, ds) || !aligned(BT, ds)))
        return fail(SPOPS_ERR_INVALID_ARG, "A or BT is NULL or misaligned");
    if (plan && !aligned(plan, 1024)) return fail(SPOPS_ERR_INVALID_ARG, "plan is not 1024-byte aligned");
    const size_t need = spops_sddmm_workspace_size(m, n, kd, nnz, dtype, itype, backend);
    if (!workspace || !aligned(workspace, 16) || ws_bytes < need)
        return fail(SPOPS_ERR_WORKSPACE, "sddmm needs a 16-byte aligned workspace of %zu bytes (got %zu)", need, ws_bytes);
    return cuda_status(launch_sddmm(dtype, itype, out_row_offsets, out_row_idx, out_col_idx, m, n, kd, nnz, A, BT,
                                    out_val, backend == SPOPS_SDDMM_STRUCTURE_AWARE, plan, workspace,
                                    (cudaStream_t)stream),
                       "sddmm launch");
}

int spops_csr_add(const void* A_val, const int32_t* row_offsets, const void* row_idx, const void* col_idx,
                  int itype, int dtype, int32_t m, int32_t n, int32_t nnz, const void* B, void* C, void* stream) {
    int st = check_common(itype, dtype, m, n, nnz, A_val, row_offsets, row_idx, col_idx, true, false);
    if (st != SPOPS_OK) return st;
    if (row_idx && !aligned(row_idx, itype_size(itype))) return fail(SPOPS_ERR_INVALID_ARG, "row_idx is misaligned");
    if ((int64_t)m * n == 0) return ok();
    const size_t ds = dtype_size(dtype);
    if (!B || !C || !aligned(B, ds) || !aligned(C, ds)) return fail(SPOPS_ERR_INVALID_ARG, "B or C is NULL or misaligned");
    const size_t bytes = (size_t)m * n * ds;
    if (B != C && overlaps(B, bytes, C, bytes)) return fail(SPOPS_ERR_INVALID_ARG, "C partially overlaps B");
    return cuda_status(launch_csr_add(dtype, itype, A_val, row_offsets, col_idx, m, n, nnz, B, C, (cudaStream_t)stream),
                       "csr_add launch");
}

size_t spops_csr_transpose_workspace_size(int32_t nnz) { return csr_transpose_workspace_bytes(nnz); }

int spops_csr_transpose(const int32_t* row_offsets, const void* col_idx, const void* values, int itype, int dtype,
                        int32_t m, int32_t n, int32_t nnz, int32_t* row_offsets_t, void* col_idx_t, void* values_t,
                        int32_t* perm, void* workspace, size_t ws_bytes, void* stream) {
    int st = check_common(itype, dtype, m, n, nnz, values, row_offsets, nullptr, col_idx, false, false);
    if (st != SPOPS_OK) return st;
    if ((values == nullptr) != (values_t == nullptr))
        return fail(SPOPS_ERR_INVALID_ARG, "values and values_t must both be given or both be NULL");
    if (!row_offsets_t || !aligned(row_offsets_t, 4)) return fail(SPOPS_ERR_INVALID_ARG, "row_offsets_t is NULL or misaligned");
    const size_t is = itype_size(itype), ds = dtype_size(dtype);
    if (nnz > 0) {
        if (!col_idx_t || !aligned(col_idx_t, is)) return fail(SPOPS_ERR_INVALID_ARG, "col_idx_t is NULL or misaligned");
        if (values && (!aligned(values, ds) || !aligned(values_t, ds)))
            return fail(SPOPS_ERR_INVALID_ARG, "values or values_t is misaligned");
        if (perm && !aligned(perm, 4)) return fail(SPOPS_ERR_INVALID_ARG, "perm is misaligned");
        const void* outs[3] = {col_idx_t, values_t, perm};
        const size_t osz[3] = {(size_t)nnz * is, (size_t)nnz * ds, (size_t)nnz * 4};
        const void* ins[3] = {col_idx, values, row_offsets};
        const size_t isz[3] = {(size_t)nnz * is, (size_t)nnz * ds, (size_t)(m + 1) * 4};
        for (int a = 0; a < 3; ++a)
            for (int b = 0; b < 3; ++b)
                if (outs[a] && ins[b] && overlaps(outs[a], osz[a], ins[b], isz[b]))
                    return fail(SPOPS_ERR_INVALID_ARG, "an output of csr_transpose overlaps an input");
        if (!workspace || !aligned(workspace, 16) || ws_bytes < spops_csr_transpose_workspace_size(nnz))
            return fail(SPOPS_ERR_WORKSPACE, "csr_transpose needs a 16-byte aligned workspace of %zu bytes (got %zu)",
                        spops_csr_transpose_workspace_size(nnz), ws_bytes);
    }
    return cuda_status(launch_csr_transpose(dtype, itype, row_offsets, col_idx, values, m, n, nnz, row_offsets_t,
                                            col_idx_t, values_t, perm, workspace, (cudaStream_t)stream),
                       "csr_transpose launch");
}

int spops_csr_permute_values(const void* values, const int32_t* perm, int dtype, int32_t nnz, void* values_t,
                             void* stream) {
    if (dtype < SPOPS_F32 || dtype > SPOPS_BF16) return fail(SPOPS_ERR_INVALID_ARG, "dtype %d is not a spops_dtype", dtype);
    if (nnz < 0) return fail(SPOPS_ERR_INVALID_ARG, "negative nnz=%d", nnz);
    if (nnz == 0) return ok();
    const size_t ds = dtype_size(dtype);
    if (!values || !perm || !values_t || !aligned(values, ds) || !aligned(values_t, ds) || !aligned(perm, 4))
        return fail(SPOPS_ERR_INVALID_ARG, "values, perm or values_t is NULL or misaligned");
    if (overlaps(values_t, (size_t)nnz * ds, values, (size_t)nnz * ds) ||
        overlaps(values_t, (size_t)nnz * ds, perm, (size_t)nnz * 4))
        return fail(SPOPS_ERR_INVALID_ARG, "values_t overlaps an input");
    return cuda_status(launch_permute_values(dtype, values, perm, nnz, values_t, (cudaStream_t)stream),
                       "csr_permute_values launch");
}

int spops_masked_adam(float* param, float* exp_avg, float* exp_avg_sq, const void* grad, int grad_dtype,
                      int64_t count, int32_t step, double lr, double beta1, double beta2, double eps, int maximize,
                      void* stream) {
    if (count < 0) return fail(SPOPS_ERR_INVALID_ARG, "negative count");
    int st = check_adam(param, exp_avg, exp_avg_sq, grad, grad_dtype, count, count, step, lr, beta1, beta2, eps);
    if (st != SPOPS_OK) return st;
    if (count == 0) return ok();
    return cuda_status(launch_masked_adam(grad_dtype, param, exp_avg, exp_avg_sq, grad, count, step, lr, beta1, beta2,
                                          eps, maximize, (cudaStream_t)stream),
                       "masked_adam launch");
}

int spops_masked_adam_csr(float* param, float* exp_avg, float* exp_avg_sq, const void* grad, int grad_dtype,
                          const int32_t* row_offsets, const void* col_idx, int itype, int32_t m, int32_t n, int32_t nnz,
                          int32_t step, double lr, double beta1, double beta2, double eps, int maximize, void* stream) {
    int st = check_common(itype, grad_dtype, m, n, nnz, grad, row_offsets, nullptr, col_idx, false, false);
    if (st != SPOPS_OK) return st;
    st = check_adam(param, exp_avg, exp_avg_sq, grad, grad_dtype, (int64_t)m * n, nnz, step, lr, beta1, beta2, eps);
    if (st != SPOPS_OK) return st;
    if (nnz == 0 || (int64_t)m * n == 0) return ok();
    return cuda_status(launch_masked_adam_csr(grad_dtype, itype, param, exp_avg, exp_avg_sq, grad, row_offsets, col_idx,
                                              m, n, step, lr, beta1, beta2, eps, maximize, (cudaStream_t)stream),
                       "masked_adam_csr launch");
}

size_t spops_check_csr_workspace_size(int32_t m) { return align_up(((size_t)(m > 0 ? m : 0) + 31) / 32 * 4, 256) + 16; }

int spops_check_csr(const int32_t* row_offsets, const void* col_idx, const void* row_idx, int itype, int32_t m,
                    int32_t n, int32_t nnz, void* workspace, size_t ws_bytes, void* stream) {
    int st = check_common(itype, SPOPS_F32, m, n, nnz, nullptr, row_offsets, row_idx, col_idx, false, false);
    if (st != SPOPS_OK) return st;
    if (row_idx && (!workspace || !aligned(workspace, 16) || ws_bytes < spops_check_csr_workspace_size(m)))
        return fail(SPOPS_ERR_WORKSPACE, "check_csr needs a workspace of %zu bytes to check row_idx",
                    spops_check_csr_workspace_size(m));
    int* err = device_error_word();
    if (!err) return fail(SPOPS_ERR_CUDA, "no device error word on the current device");
    return cuda_status(launch_check_csr(row_offsets, col_idx, row_idx, itype, m, n, nnz,
                                        static_cast<uint32_t*>(workspace), err, (cudaStream_t)stream),
                       "check_csr launch");
}

int spops_release_streams(void) { return cuda_status(release_sides(), "release side streams"); }

int spops_selftest_wait_timeout(int64_t limit_ns, uint64_t* waited_ns, void* stream) {
    if (limit_ns < 1000 || limit_ns > 1000000000)
        return fail(SPOPS_ERR_INVALID_ARG, "limit_ns must lie in [1e3, 1e9] (got %lld)", (long long)limit_ns);
    if (waited_ns && !aligned(waited_ns, 8)) return fail(SPOPS_ERR_INVALID_ARG, "waited_ns is not 8-byte aligned");
    return cuda_status(launch_wait_selftest((uint64_t)limit_ns, reinterpret_cast<unsigned long long*>(waited_ns),
                                            (cudaStream_t)stream),
                       "wait self-test launch");
}

int spops_get_device_error(void* stream, int32_t* code_out) {
    if (!code_out) return fail(SPOPS_ERR_INVALID_ARG, "code_out is NULL");
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_status(e, "stream synchronize");
    int* err = device_error_word();
    if (!err) return fail(SPOPS_ERR_CUDA, "no device error word on the current device");
    int v = 0;
    e = cudaMemcpy(&v, err, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_status(e, "read device error word");
    const int zero = 0;
    e = cudaMemcpy(err, &zero, sizeof(int), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_status(e, "clear device error word");
    *code_out = v;
    return ok();
}

}  // extern "C"
