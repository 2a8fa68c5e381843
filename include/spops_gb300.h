/*
 * spops_gb300.h -- C ABI of the GB300 (sm_103a) CSR sparse-adapter operators.
 *
 * The operators are the ones the spops README ("Sparse Operations (spops)") lists:
 *   csr_add  [dense = sparse + dense]      section "Sparse Addition"
 *   spmm     [dense = sparse x dense]      section "Sparse Matrix Multiplication (SpMM)"
 *   sddmm    [sparse = dense x dense]      section "Sampled Dense-Dense Matrix
 *                                          Multiplication (SDDMM)", with a general and a
 *                                          structure-aware backend (structure-aware is the
 *                                          default)
 * plus the row permutation row_idx and the row bins that schedule them.
 *
 * CSR layout (section "Usage"): an m x n matrix with nnz entries is
 *   values      [nnz]    entry values, dtype `dtype`;
 *   row_offsets [m + 1]  int32; row i holds entries row_offsets[i] .. row_offsets[i+1]-1;
 *   col_idx     [nnz]    column of each entry, int16 (SPOPS_IDX16) or int32 (SPOPS_IDX32);
 *   row_idx     [m]      permutation of 0..m-1 sorting rows by nnz, same width as col_idx.
 * Section "Important Notes" fixes int32 row_offsets and int16 index lists; int16 limits m
 * and n to 32768, so SPOPS_IDX32 is offered for larger matrices.
 * The library expects canonical CSR: row_offsets[0] = 0, non-decreasing, row_offsets[m] =
 * nnz, and columns strictly increasing inside each row. spops_check_csr verifies this on
 * the device. Results are correct for ANY permutation in row_idx; a sorted one (as
 * spops_sort_rows writes) only balances the work.
 *
 * Conventions for every call:
 *   - Every array is a DEVICE pointer into memory the caller owns and keeps alive until the
 *     work on `stream` finishes. All arrays are dense and contiguous (row-major for
 *     matrices). Element pointers must be aligned to their element size.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream). Calls are
 *     asynchronous on that stream and never synchronize, except spops_get_device_error.
 *   - The library allocates no device memory. Calls that need scratch take a caller
 *     `workspace` of at least the size the matching *_workspace_size function returns,
 *     16-byte aligned; it may be reused once the call's work on `stream` has finished.
 *     (Its persistent resources are listed above spops_release_streams.)
 *   - Return value: an spops_status. Argument errors are detected on the host before any
 *     work is queued and leave every output untouched. SPOPS_ERR_CUDA reports a failed
 *     launch. spops_last_error() gives a one-line description of the last failure on the
 *     calling thread.
 *   - Floating-point results accumulate in fp32 and are rounded once (round to nearest
 *     even) to the operand dtype. Values and dense operands share one dtype.
 */
#ifndef SPOPS_GB300_H
#define SPOPS_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SPOPS_API __attribute__((visibility("default")))
#else
#define SPOPS_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum spops_status {
    SPOPS_OK = 0,
    SPOPS_ERR_INVALID_ARG = 1,  /* bad enum, negative size, null or misaligned pointer */
    SPOPS_ERR_UNSUPPORTED = 2,  /* valid request this library does not serve (e.g. int16 overflow) */
    SPOPS_ERR_WORKSPACE = 3,    /* workspace missing, misaligned or smaller than required */
    SPOPS_ERR_CUDA = 4,         /* a CUDA runtime call or kernel launch failed */
    SPOPS_ERR_DEVICE_CHECK = 5  /* a device-side check recorded a violation */
} spops_status;

typedef enum spops_dtype { SPOPS_F32 = 0, SPOPS_F16 = 1, SPOPS_BF16 = 2 } spops_dtype;
typedef enum spops_itype { SPOPS_IDX16 = 0, SPOPS_IDX32 = 1 } spops_itype;
typedef enum spops_spmm_path {
    SPOPS_SPMM_AUTO = 0,   /* dense panels (fp16/bf16) on tensor cores, the other rows general */
    SPOPS_SPMM_GENERAL = 1 /* every row on the general row kernels */
} spops_spmm_path;
typedef enum spops_sddmm_backend {
    SPOPS_SDDMM_STRUCTURE_AWARE = 0, /* default: dense panels on tensor cores, the rest general */
    SPOPS_SDDMM_GENERAL = 1          /* any sparsity pattern, CUDA cores */
} spops_sddmm_backend;

/* Device error codes reported by spops_get_device_error. */
#define SPOPS_DEV_OK 0
#define SPOPS_DEV_MBAR_TIMEOUT 1 /* an asynchronous-copy or tensor-core wait exceeded its time limit */
#define SPOPS_DEV_ROW_OFFSETS 2  /* row_offsets not non-decreasing, or wrong first/last value */
#define SPOPS_DEV_COL_RANGE 3    /* a column index outside [0, n) */
#define SPOPS_DEV_COL_ORDER 4    /* columns not strictly increasing inside a row */
#define SPOPS_DEV_ROW_IDX 5      /* row_idx is not a permutation of 0..m-1 */
#define SPOPS_DEV_TMEM 6         /* tensor-memory allocation failed */

/* Row-bin thresholds the operators use: rows with at least this many entries are "long". */
#define SPOPS_SPMM_LONG_ROW 256
#define SPOPS_SDDMM_LONG_ROW 64

/* Human-readable name of a status code (static string). */
SPOPS_API const char* spops_status_string(int status);

/* One-line description of the most recent failed call on this thread ("" if none). */
SPOPS_API const char* spops_last_error(void);

/* Library version string, e.g. "spops_gb300 0.1 sm_103a". */
SPOPS_API const char* spops_version(void);

/* Number of kernels this library has launched in this process (all devices, all
 * threads). A call captured into a CUDA graph counts once, at capture. */
SPOPS_API uint64_t spops_kernel_launches(void);

/* Persistent resources. Besides two static device arrays (the 4-byte device error word and
 * the scratch of spops_sort_rows_static), the only thing the library keeps between calls is,
 * per calling host thread, up to 8 side streams with two events each: spops_spmm and
 * spops_sddmm run their general row kernels on a side stream of the caller's stream beside
 * the tensor-core panels (forked and joined with the events, so both are captured into CUDA
 * graphs as a fork and a join). They are created on the first such call for a (device,
 * caller stream) pair, never while that stream is being captured. spops_release_streams
 * destroys the calling thread's side streams and events (work already queued on them
 * completes); the next call creates them again. Call it when no capture that uses them is
 * in progress, e.g. before a thread exits. Returns SPOPS_ERR_CUDA if a destroy call fails. */
SPOPS_API int spops_release_streams(void);

/* ---------------------------------------------------------------- row scheduler */

/* Scratch bytes spops_sort_rows needs for m rows. */
SPOPS_API size_t spops_sort_rows_workspace_size(int32_t m);

/* row_idx_out[0..m) = the rows ordered by nnz_i = row_offsets[i+1] - row_offsets[i],
 * largest first, ties by ascending row id (spops README, section "Usage": row_idx sorts
 * the rows by their number of non-zeros; the README leaves the direction open).
 * row_offsets: [m+1] int32 device; nnz = row_offsets[m] (bounds the sort key);
 * row_idx_out: [m] device, int16 or int32 per `itype` (int16 needs m <= 32768).
 * Deterministic: bit-identical output on every call. */
SPOPS_API int spops_sort_rows(const int32_t* row_offsets, int32_t m, int32_t nnz, void* row_idx_out, int itype,
                    void* workspace, size_t ws_bytes, void* stream);

/* spops_sort_rows without a workspace, for callers that cannot allocate device memory
 * where they need row_idx (a plugin whose host application owns every device allocation,
 * or a loop that must not call cudaMalloc because it can synchronize the device). The
 * pages have no counterpart of this call; it exists for such callers only.
 * Same arguments and result as spops_sort_rows minus the workspace: the scratch is a
 * static device array inside this library that holds at most
 * spops_sort_rows_static_max_rows() rows (131072; about 2.1 MB reserved on every GPU that
 * loads the library, until the process exits). Larger m returns SPOPS_ERR_UNSUPPORTED.
 * The call allocates nothing. Its first call on a device looks up the array's device
 * address (cudaGetSymbolAddress) with that device current; make that first call before any
 * stream capture. All calls on a device share the array, so calls whose GPU work overlaps
 * (e.g. on unordered streams) race and must be serialized by the caller. */
SPOPS_API int spops_sort_rows_static(const int32_t* row_offsets, int32_t m, int32_t nnz, void* row_idx_out,
                                     int itype, void* stream);
SPOPS_API int32_t spops_sort_rows_static_max_rows(void);
/* (The array's device address is looked up once per device and kept for the life of the
 * process, so it does not survive cudaDeviceReset: do not use the library again in that
 * process after a reset.) */

/* bins_out[0..4) (device int32) = {0, #rows with nnz >= t_long, #rows with nnz >= 1, m}:
 * prefix offsets that split a sorted row_idx into long, short and empty rows. The counts
 * do not depend on row_idx, so the call takes only row_offsets. t_long >= 1. */
SPOPS_API int spops_row_bins(const int32_t* row_offsets, int32_t m, int32_t t_long, int32_t* bins_out, void* stream);

/* ---------------------------------------------------------------- mask plan */

/* Bytes of a mask plan for an m x n mask with nnz entries (callers allocate it 1024-byte
 * aligned). */
SPOPS_API size_t spops_plan_size(int32_t m, int32_t n, int32_t nnz);

/* Build the mask plan: everything the operators derive from the CSR structure alone, so a
 * plan built once serves every spmm / sddmm call on the same mask (same row_offsets,
 * row_idx, col_idx, m, n, nnz), like row_idx itself. It holds
 *   - the row bins of each operator (spops README, "Usage": row_idx sorts the rows by
 *     nnz; long rows get a CTA each, short rows a group of lanes), and, when n <= 65536,
 *   - the panel decomposition behind the structure-aware paths (README, "Sampled
 *     Dense-Dense Matrix Multiplication": the structure-aware kernel exploits non-zeros
 *     that cluster in a few rows and columns): panels of 128 consecutive row_idx
 *     positions; a panel is filled when it has at least 16 non-empty rows and its entries
 *     fill at least a quarter of (non-empty rows) x |U|, U the union of its columns. Filled
 *     panels run SDDMM on the tensor cores when |U| <= 1024 and SpMM when |U| <= 4096
 *     (and their SpMM image fits the workspace's budget).
 * plan: device buffer of spops_plan_size bytes, 1024-byte aligned, owned by the caller and
 * left unchanged by the operators. Deterministic: the same mask gives the same plan. */
SPOPS_API int spops_plan_build(const int32_t* row_offsets, const void* row_idx, const void* col_idx, int itype,
                               int32_t m, int32_t n, int32_t nnz, void* plan, size_t plan_size, void* stream);

/* stats_out (device int32[16]) = {dense panels, SDDMM tiles, panels with a SpMM image,
 * entries in dense panels, SpMM image elements, panels, SDDMM tile groups (up to 4
 * consecutive tiles of a panel), 0, SpMM row bins [4], SDDMM row bins [4]} of a built plan. */
SPOPS_API int spops_plan_stats(const void* plan, int32_t m, int32_t n, int32_t nnz, int32_t* stats_out, void* stream);

/* order_out (device int32[m]) = the row at each position of the plan's row order, the order
 * in which the panels (128 consecutive positions each) and the operators' row kernels take
 * the rows. It is row_idx, refined for masks of at most 16384 rows: when two runs of at least
 * 32 positions of row_idx (stretches of non-empty rows with equal keys) share a key, the
 * positions are sorted stably by key = (65535 - min(nnz, 65535)) << 16 | a 16-bit hash of the
 * row's first, middle and last column, so that rows with one column pattern share panels.
 * Returns SPOPS_ERR_UNSUPPORTED when the plan has no panels (n > 65536: the operators walk
 * row_idx itself). */
SPOPS_API int spops_plan_row_order(const void* plan, int32_t m, int32_t n, int32_t nnz, int32_t* order_out,
                                   void* stream);

/* ---------------------------------------------------------------- operators */

/* Scratch bytes spops_spmm needs (enough to build its own plan and the dense-panel images). */
SPOPS_API size_t spops_spmm_workspace_size(int32_t m, int32_t k, int32_t n, int32_t nnz, int dtype, int itype);

/* SpMM (spops README, "Sparse Matrix Multiplication (SpMM)"): C = A * B.
 * A: m x k CSR (A_val [nnz] dtype, row_offsets [m+1], row_idx [m], col_idx [nnz]);
 * B: k x n row-major dtype; C: m x n row-major dtype, every element written (rows without
 * entries become zeros). C must not overlap B or A's arrays. path: spops_spmm_path; AUTO
 * runs the plan's dense panels on the tensor cores (fp16/bf16, n > 16 and a multiple of 8,
 * 16-byte aligned B and C), the other rows on the general row kernels; n <= 16 takes a
 * streaming warp-per-row kernel. plan: a plan built by
 * spops_plan_build for this mask (m x k), or NULL to build one inside the workspace. */
SPOPS_API int spops_spmm(const void* A_val, const int32_t* row_offsets, const void* row_idx, const void* col_idx,
                         int itype, int dtype, int32_t m, int32_t k, int32_t nnz, const void* B, int32_t n, void* C,
                         int path, const void* plan, void* workspace, size_t ws_bytes, void* stream);

/* Scratch bytes spops_sddmm needs for the chosen backend (including its own plan). */
SPOPS_API size_t spops_sddmm_workspace_size(int32_t m, int32_t n, int32_t kd, int32_t nnz, int dtype, int itype,
                                            int backend);

/* SDDMM (spops README, "Sampled Dense-Dense Matrix Multiplication (SDDMM)"):
 * out_val[k] = sum_t A[i, t] * BT[col_idx[k], t] for every entry k of row i of the m x n
 * mask (out_row_offsets [m+1], out_row_idx [m], out_col_idx [nnz]).
 * A: m x kd row-major; BT: n x kd row-major (the right operand transposed);
 * out_val: [nnz] dtype, in CSR order. backend: spops_sddmm_backend (STRUCTURE_AWARE runs
 * the plan's dense panels on the tensor cores for fp16/bf16 with kd a multiple of 8 and
 * 16-byte aligned A and BT). No scaling by mask values (the call takes none). plan: as for
 * spops_spmm (an m x n plan), or NULL. */
SPOPS_API int spops_sddmm(const int32_t* out_row_offsets, const void* out_row_idx, const void* out_col_idx,
                          int itype, int dtype, int32_t m, int32_t n, int32_t kd, int32_t nnz, const void* A,
                          const void* BT, void* out_val, int backend, const void* plan, void* workspace,
                          size_t ws_bytes, void* stream);

/* csr_add (spops README, "Sparse Addition"): C = B + A with A an m x n CSR matrix and B, C
 * dense m x n row-major. C == B (in place) is allowed; partial overlap is not. Each entry
 * is the correctly rounded sum of the two dtype values (bit-exact). row_idx is accepted
 * for signature parity with the README and may be NULL. */
SPOPS_API int spops_csr_add(const void* A_val, const int32_t* row_offsets, const void* row_idx, const void* col_idx,
                            int itype, int dtype, int32_t m, int32_t n, int32_t nnz, const void* B, void* C,
                            void* stream);

/* ---------------------------------------------------------------- transpose, dB = A^T dC */

/* Scratch bytes spops_csr_transpose needs for nnz entries (radix-sort key and index
 * buffers and per-block digit histograms). */
SPOPS_API size_t spops_csr_transpose_workspace_size(int32_t nnz);

/* A^T of the m x n CSR matrix (row_offsets, col_idx, values) as an n x m CSR matrix
 * (row_offsets_t [n+1] int32, col_idx_t [nnz] = row ids of A, values_t [nnz]).
 * spops README, operation list: "csr_transpose"; with it the gradient of C = A B with
 * respect to B is dB = A^T dC, one spops_spmm call on the transpose (torchsparsegradutils
 * README, "Basic Sparse Matrix Multiplication", gradients of sparse products).
 * Output is canonical: row j of A^T lists column j of A by ascending row (a stable order
 * by column), bit-exact and identical run to run. perm [nnz] int32 (may be NULL) receives,
 * for every position p of A^T, the entry of A placed there, for spops_csr_permute_values.
 * values and values_t may both be NULL (structure only). itype applies to col_idx and
 * col_idx_t: int16 needs m, n <= 32768. All buffers are caller-owned device memory; the
 * outputs must not overlap the inputs. workspace: 16-byte aligned, at least
 * spops_csr_transpose_workspace_size(nnz) bytes. Returns SPOPS_ERR_INVALID_ARG /
 * SPOPS_ERR_UNSUPPORTED / SPOPS_ERR_WORKSPACE before queueing anything, SPOPS_ERR_CUDA if
 * a launch fails. */
SPOPS_API int spops_csr_transpose(const int32_t* row_offsets, const void* col_idx, const void* values, int itype,
                                  int dtype, int32_t m, int32_t n, int32_t nnz, int32_t* row_offsets_t,
                                  void* col_idx_t, void* values_t, int32_t* perm, void* workspace, size_t ws_bytes,
                                  void* stream);

/* values_t[p] = values[perm[p]] for p < nnz: new values of A carried through a transpose
 * computed earlier (the structure of a RoSA mask is fixed while its values train). */
SPOPS_API int spops_csr_permute_values(const void* values, const int32_t* perm, int dtype, int32_t nnz,
                                       void* values_t, void* stream);

/* ---------------------------------------------------------------- masked Adam */

/* One Adam step on the entries a sparse gradient materializes (SparseAdam page,
 * tensorplay.optim.sparse_adam.SparseAdam: moments and parameters change only where the
 * sparse gradient holds a value). With d = grad (negated when maximize != 0):
 *   exp_avg = beta1 exp_avg + (1 - beta1) d;  exp_avg_sq = beta2 exp_avg_sq + (1 - beta2) d^2;
 *   param -= lr * (exp_avg / (1 - beta1^step)) / (sqrt(exp_avg_sq / (1 - beta2^step)) + eps)
 * in fp32. Here the gradient holds one value per parameter entry (count entries, the
 * values of the parameter's own CSR mask, as for the RoSA adapter): entry g updates
 * param[g], exp_avg[g], exp_avg_sq[g] in place. param / exp_avg / exp_avg_sq are fp32
 * device arrays of count entries; grad is count values of grad_dtype. The four arrays must
 * not overlap. Requires step >= 1, lr >= 0, eps >= 0, 0 <= beta1, beta2 < 1, else
 * SPOPS_ERR_INVALID_ARG before anything is queued. */
SPOPS_API int spops_masked_adam(float* param, float* exp_avg, float* exp_avg_sq, const void* grad, int grad_dtype,
                                int64_t count, int32_t step, double lr, double beta1, double beta2, double eps,
                                int maximize, void* stream);

/* The same step for a dense m x n row-major fp32 parameter (and moments) with a CSR
 * gradient (row_offsets, col_idx, nnz values of grad_dtype): entry k of row i updates
 * position i * n + col_idx[k]; every other position is left untouched (the page's
 * "parameters of a dense layout with gradients of a sparse layout"). The CSR must be
 * canonical (no repeated column in a row). */
SPOPS_API int spops_masked_adam_csr(float* param, float* exp_avg, float* exp_avg_sq, const void* grad, int grad_dtype,
                                    const int32_t* row_offsets, const void* col_idx, int itype, int32_t m, int32_t n,
                                    int32_t nnz, int32_t step, double lr, double beta1, double beta2, double eps,
                                    int maximize, void* stream);

/* ---------------------------------------------------------------- checks */

/* Scratch bytes spops_check_csr needs (a bitmap of m bits for the permutation check). */
SPOPS_API size_t spops_check_csr_workspace_size(int32_t m);

/* Queue device-side checks of the CSR structure (row_offsets ends and order, column range
 * and order) and, when row_idx is non-NULL, that row_idx is a permutation of 0..m-1.
 * Violations are recorded in the device error word; read them with
 * spops_get_device_error. */
SPOPS_API int spops_check_csr(const int32_t* row_offsets, const void* col_idx, const void* row_idx, int itype, int32_t m,
                    int32_t n, int32_t nnz, void* workspace, size_t ws_bytes, void* stream);

/* Synchronize `stream`, then return in *code_out the first device error recorded on the
 * current device since the last call (SPOPS_DEV_*), and clear it. The error word's device
 * address is looked up once per device and kept for the life of the process: after
 * cudaDeviceReset this library must not be used again in that process. */
SPOPS_API int spops_get_device_error(void* stream, int32_t* code_out);

/* Self-test of failure detection. Every wait of the library's TMA and tensor-core kernels
 * on an asynchronous copy or an MMA gives up after a time limit (2 s), records
 * SPOPS_DEV_MBAR_TIMEOUT in the device error word and lets its kernel return, so a copy
 * that never completes cannot hang the GPU. This call queues one kernel whose single
 * thread waits on a shared-memory barrier that nothing ever arrives on (no copy, TMA load
 * or MMA is in flight) with the limit limit_ns, in [1e3, 1e9] nanoseconds; the wait gives
 * up and records SPOPS_DEV_MBAR_TIMEOUT. waited_ns (device pointer to one uint64, 8-byte
 * aligned, may be NULL) receives the nanoseconds the wait lasted (%globaltimer). Read and
 * clear the code with spops_get_device_error; the context stays usable. The pages have no
 * counterpart of this call. */
SPOPS_API int spops_selftest_wait_timeout(int64_t limit_ns, uint64_t* waited_ns, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SPOPS_GB300_H */
