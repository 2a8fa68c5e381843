// csr_transpose: A^T of an m x n CSR matrix as an n x m CSR matrix, and the gather that
// carries new values through an existing transpose.
//
// spops README ("Sparse Operations (spops)"): csr_transpose is one of the listed sparse
// operations; with it the gradient of C = A B with respect to the dense operand is
// dB = A^T dC, an SpMM of the transpose (torchsparsegradutils README, "Basic Sparse Matrix
// Multiplication", on gradients of sparse products).
//
// Output is canonical: row j of A^T lists column j of A by ascending row, i.e. the entries
// are ordered stably by column. Steps:
//   1. a stable least-significant-digit radix sort of the entry indices 0..nnz-1 by column,
//      8 bits per pass (per-block digit histograms, a two-step parallel scan of them, a
//      stable scatter that ranks equal digits inside a block with warp match masks);
//   2. the last pass scatters the finished entries directly: the entry's row (from an
//      entry -> row map written once, a warp per row), its value and its index (perm), and
//      keeps the sorted columns;
//   3. ro_t[j] = the first position whose column is >= j (binary search per j).
// perm lets later calls move new values through the same structure (csr_permute_values).
#include "common.cuh"
#include "internal.h"
#include "scan.cuh"

namespace spops {
namespace {

constexpr int kTThreads = 256;
constexpr int kTRounds = 8;
constexpr int kTRadix = 256;

// Key of position i in a pass: the column of entry i (first pass) or the carried key.
template <typename I>
__device__ __forceinline__ uint32_t tkey(const I* col, const uint32_t* keys_in, int32_t i) {
    return keys_in ? keys_in[i] : (uint32_t)idx_of(col[i]);
}

template <typename I>
__global__ void __launch_bounds__(kTThreads)
tr_hist_kernel(const I* __restrict__ col, const uint32_t* __restrict__ keys_in, int32_t nnz, int shift, int rounds,
               uint32_t* __restrict__ hist) {
    __shared__ uint32_t cnt[kTRadix];
    cnt[threadIdx.x] = 0;
    __syncthreads();
    const int32_t base = blockIdx.x * rounds * kTThreads;
    for (int r = 0; r < rounds; ++r) {
        const int32_t i = base + r * kTThreads + threadIdx.x;
        if (i < nnz) atomicAdd(&cnt[(tkey(col, keys_in, i) >> shift) & (kTRadix - 1)], 1u);
    }
    __syncthreads();
    hist[threadIdx.x * gridDim.x + blockIdx.x] = cnt[threadIdx.x];
}

// entry_row[k] = the row of entry k: a warp per row writes its id over the row's entries.
__global__ void __launch_bounds__(256) tr_entry_rows_kernel(const int32_t* __restrict__ ro, int32_t m,
                                                           int32_t* __restrict__ entry_row) {
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t i = warp; i < m; i += nwarps)
        for (int32_t k = ro[i] + lane; k < ro[i + 1]; k += 32) entry_row[k] = (int32_t)i;
}

// Stable scatter of one pass. Intermediate passes carry (key, entry index); the last pass
// writes the entry's row id, value and index at its final position.
template <typename T, typename I>
__global__ void __launch_bounds__(kTThreads)
tr_scatter_kernel(const I* __restrict__ col, const uint32_t* __restrict__ keys_in, const int32_t* __restrict__ vals_in,
                  int32_t nnz, int shift, int rounds, const uint32_t* __restrict__ offsets,
                  const uint32_t* __restrict__ sums, uint32_t* __restrict__ keys_out, int32_t* __restrict__ vals_out,
                  bool last, const int32_t* __restrict__ entry_row, const T* __restrict__ val, I* __restrict__ row_t,
                  T* __restrict__ val_t, int32_t* __restrict__ perm) {
    __shared__ uint32_t warp_cnt[kTThreads / 32][kTRadix];
    __shared__ uint32_t running[kTRadix];
    __shared__ uint32_t dbase[kTRadix];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    running[tid] = 0;
    {
        const int64_t at = (int64_t)tid * gridDim.x + blockIdx.x;
        dbase[tid] = offsets[at] + sums[at / kScanChunk];
    }
    const uint32_t lt_mask = (1u << lane) - 1u;
    const int32_t base = blockIdx.x * rounds * kTThreads;
    for (int r = 0; r < rounds; ++r) {
#pragma unroll
        for (int w = 0; w < kTThreads / 32; ++w) warp_cnt[w][tid] = 0;
        __syncthreads();
        const int32_t i = base + r * kTThreads + tid;
        const bool valid = i < nnz;
        uint32_t key = 0;
        int32_t k = 0;
        int d = kTRadix + lane;  // unique per invalid lane: never matches a real digit
        if (valid) {
            key = tkey(col, keys_in, i);
            k = vals_in ? vals_in[i] : i;
            d = (int)((key >> shift) & (kTRadix - 1));
        }
        const uint32_t peers = __match_any_sync(0xffffffffu, d);
        const uint32_t rank = __popc(peers & lt_mask);
        if (valid && lane == __ffs(peers) - 1) warp_cnt[warp][d] = __popc(peers);
        __syncthreads();
        {  // digit tid: exclusive prefix over warps, continuing from earlier rounds
            uint32_t acc = running[tid];
#pragma unroll
            for (int w = 0; w < kTThreads / 32; ++w) {
                const uint32_t c = warp_cnt[w][tid];
                warp_cnt[w][tid] = acc;
                acc += c;
            }
            running[tid] = acc;
        }
        __syncthreads();
        if (valid) {
            const uint32_t pos = dbase[d] + warp_cnt[warp][d] + rank;
            keys_out[pos] = key;
            if (!last) {
                vals_out[pos] = k;
            } else {
                row_t[pos] = static_cast<I>(entry_row[k]);
                if (val_t) val_t[pos] = val[k];
                if (perm) perm[pos] = k;
            }
        }
        __syncthreads();
    }
}

// ro_t[j] = number of entries with column < j: a lower bound of j in the sorted columns.
__global__ void __launch_bounds__(256) tr_offsets_kernel(const uint32_t* __restrict__ keys, int32_t nnz, int32_t n,
                                                        int32_t* __restrict__ ro_t) {
    for (int32_t j = blockIdx.x * blockDim.x + threadIdx.x; j <= n; j += gridDim.x * blockDim.x) {
        int32_t lo = 0, hi = nnz;  // first position with keys[p] >= j lies in [lo, hi]
        while (lo < hi) {
            const int32_t mid = (lo + hi) >> 1;
            if (keys[mid] < (uint32_t)j) lo = mid + 1;
            else hi = mid;
        }
        ro_t[j] = lo;
    }
}

template <typename T>
__global__ void __launch_bounds__(256) permute_values_kernel(const T* __restrict__ val, const int32_t* __restrict__ perm,
                                                            int32_t nnz, T* __restrict__ val_t) {
    for (int32_t p = blockIdx.x * blockDim.x + threadIdx.x; p < nnz; p += gridDim.x * blockDim.x)
        val_t[p] = val[perm[p]];
}

// Entries per CTA = rounds * 256: enough CTAs to fill the GPU twice for small matrices,
// up to 8 rounds (2048 entries) per CTA for large ones.
int tr_rounds(int32_t nnz) {
    const int64_t target = (int64_t)device_props().sm_count * 2 * kTThreads;
    const int64_t r = nnz / (target > 0 ? target : 1);
    return (int)max64(1, min64(kTRounds, r));
}

int bits_for(uint32_t x) {
    int b = 0;
    while (b < 32 && (x >> b) != 0) ++b;
    return b;
}

template <typename T, typename I>
cudaError_t run_transpose(const int32_t* ro, const void* col_v, const void* val_v, int32_t m, int32_t n, int32_t nnz,
                          int32_t* ro_t, void* row_t_v, void* val_t_v, int32_t* perm, void* ws, cudaStream_t s) {
    const I* col = static_cast<const I*>(col_v);
    const T* val = static_cast<const T*>(val_v);
    I* row_t = static_cast<I*>(row_t_v);
    T* val_t = static_cast<T*>(val_t_v);
    if (nnz == 0) {
        cudaError_t e = cudaMemsetAsync(ro_t, 0, (size_t)(n + 1) * sizeof(int32_t), s);
        return e;
    }
    const int passes = max(1, (bits_for((uint32_t)(n - 1)) + 7) / 8);
    const int rounds = tr_rounds(nnz);
    const int nb = (nnz + rounds * kTThreads - 1) / (rounds * kTThreads);
    const int64_t counters = (int64_t)nb * kTRadix;
    const int nchunks = (int)scan_chunks(counters);
    const size_t arr = align_up((size_t)nnz * 4, 256);
    char* w = static_cast<char*>(ws);
    uint32_t* keys[2] = {reinterpret_cast<uint32_t*>(w), reinterpret_cast<uint32_t*>(w + arr)};
    int32_t* vals[2] = {reinterpret_cast<int32_t*>(w + 2 * arr), reinterpret_cast<int32_t*>(w + 3 * arr)};
    uint32_t* hist = reinterpret_cast<uint32_t*>(w + 4 * arr);
    uint32_t* sums = reinterpret_cast<uint32_t*>(w + 4 * arr + align_up((size_t)counters * 4, 256));
    // entry -> row map, after the scan sums
    int32_t* entry_row = reinterpret_cast<int32_t*>(reinterpret_cast<char*>(sums) +
                                                    align_up((size_t)scan_chunks(counters) * 4, 256));
    const int sms = device_props().sm_count;
    tr_entry_rows_kernel<<<(int)min64((int64_t)sms * 8, ((int64_t)m + 7) / 8), 256, 0, s>>>(ro, m, entry_row);
    int launches = 1;
    for (int p = 0; p < passes; ++p) {
        const uint32_t* kin = p == 0 ? nullptr : keys[(p - 1) & 1];
        const int32_t* vin = p == 0 ? nullptr : vals[(p - 1) & 1];
        const bool last = p == passes - 1;
        tr_hist_kernel<I><<<nb, kTThreads, 0, s>>>(col, kin, nnz, 8 * p, rounds, hist);
        chunk_scan_kernel<<<nchunks, kScanThreads1k, 0, s>>>(hist, counters, sums);
        chunk_sums_kernel<<<1, kScanThreads1k, 0, s>>>(sums, nchunks);
        tr_scatter_kernel<T, I><<<nb, kTThreads, 0, s>>>(col, kin, vin, nnz, 8 * p, rounds, hist, sums, keys[p & 1],
                                                         vals[p & 1], last, entry_row, val, row_t, val_t, perm);
        launches += 4;
    }
    const int grid = (int)min64((int64_t)sms * 4, ((int64_t)n + 256) / 256);
    tr_offsets_kernel<<<grid, 256, 0, s>>>(keys[(passes - 1) & 1], nnz, n, ro_t);
    count_launches(launches + 1);
    return cudaGetLastError();
}

template <typename T>
cudaError_t run_tr_dt(int it, const int32_t* ro, const void* col, const void* val, int32_t m, int32_t n, int32_t nnz,
                      int32_t* ro_t, void* row_t, void* val_t, int32_t* perm, void* ws, cudaStream_t s) {
    return it == kIdx16 ? run_transpose<T, uint16_t>(ro, col, val, m, n, nnz, ro_t, row_t, val_t, perm, ws, s)
                        : run_transpose<T, int32_t>(ro, col, val, m, n, nnz, ro_t, row_t, val_t, perm, ws, s);
}

}  // namespace

size_t csr_transpose_workspace_bytes(int32_t nnz) {
    if (nnz <= 0) return 256;
    const size_t arr = align_up((size_t)nnz * 4, 256);
    const size_t nb = ((size_t)nnz + kTThreads - 1) / kTThreads;  // the most CTAs (one round each)
    const size_t counters = nb * kTRadix;
    return 5 * arr + align_up(counters * 4, 256) + align_up((size_t)scan_chunks((int64_t)counters) * 4, 256);
}

cudaError_t launch_csr_transpose(int dt, int it, const int32_t* ro, const void* col, const void* val, int32_t m,
                                 int32_t n, int32_t nnz, int32_t* ro_t, void* row_t, void* val_t, int32_t* perm,
                                 void* ws, cudaStream_t s) {
    if (dt == kF32) return run_tr_dt<float>(it, ro, col, val, m, n, nnz, ro_t, row_t, val_t, perm, ws, s);
    if (dt == kF16) return run_tr_dt<__half>(it, ro, col, val, m, n, nnz, ro_t, row_t, val_t, perm, ws, s);
    return run_tr_dt<__nv_bfloat16>(it, ro, col, val, m, n, nnz, ro_t, row_t, val_t, perm, ws, s);
}

cudaError_t launch_permute_values(int dt, const void* val, const int32_t* perm, int32_t nnz, void* val_t,
                                  cudaStream_t s) {
    if (nnz <= 0) return cudaSuccess;
    const int grid = (int)min64((int64_t)device_props().sm_count * 8, ((int64_t)nnz + 255) / 256);
    if (dt == kF32)
        permute_values_kernel<float><<<grid, 256, 0, s>>>(static_cast<const float*>(val), perm, nnz,
                                                          static_cast<float*>(val_t));
    else if (dt == kF16)
        permute_values_kernel<__half><<<grid, 256, 0, s>>>(static_cast<const __half*>(val), perm, nnz,
                                                           static_cast<__half*>(val_t));
    else
        permute_values_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(val), perm, nnz,
                                                                  static_cast<__nv_bfloat16*>(val_t));
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace spops
