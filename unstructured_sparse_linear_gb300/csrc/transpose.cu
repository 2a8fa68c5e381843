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
//   1. column counts with integer atomics (order-free, so the counts are exact), one block
//      scan over n + 1 counters: ro_t;
//   2. a stable least-significant-digit radix sort of the entry indices 0..nnz-1 by column,
//      8 bits per pass (per-block digit histograms, one scan, a stable scatter that ranks
//      equal digits inside a block with warp match masks);
//   3. the last pass scatters the finished entries directly: the entry's row (binary search
//      in row_offsets), its value and its index (perm).
// perm lets later calls move new values through the same structure (csr_permute_values).
#include "common.cuh"
#include "internal.h"

namespace spops {
namespace {

constexpr int kTThreads = 256;
constexpr int kTRounds = 8;
constexpr int kTTile = kTThreads * kTRounds;
constexpr int kTRadix = 256;
constexpr int kTScanThreads = 1024;

template <typename I>
__global__ void __launch_bounds__(256) col_count_kernel(const I* __restrict__ col, int32_t nnz,
                                                       int32_t* __restrict__ cnt) {
    for (int32_t k = blockIdx.x * blockDim.x + threadIdx.x; k < nnz; k += gridDim.x * blockDim.x)
        atomicAdd(&cnt[idx_of(col[k]) + 1], 1);
}

// Inclusive scan, in place, of `total` int32 counters with one block (cnt[0] = 0 stays 0,
// so the result is the exclusive prefix of the column counts: row offsets of A^T).
__global__ void __launch_bounds__(kTScanThreads) scan_counts_kernel(int32_t* __restrict__ cnt, int32_t total) {
    __shared__ int32_t part[kTScanThreads];
    const int32_t per = (total + kTScanThreads - 1) / kTScanThreads;
    const int32_t b = threadIdx.x * per, e = min(total, b + per);
    int32_t s = 0;
    for (int32_t i = b; i < e; ++i) s += cnt[i];
    part[threadIdx.x] = s;
    __syncthreads();
    for (int off = 1; off < kTScanThreads; off <<= 1) {
        const int32_t v = threadIdx.x >= off ? part[threadIdx.x - off] : 0;
        __syncthreads();
        part[threadIdx.x] += v;
        __syncthreads();
    }
    int32_t run = threadIdx.x ? part[threadIdx.x - 1] : 0;
    for (int32_t i = b; i < e; ++i) {
        run += cnt[i];
        cnt[i] = run;
    }
}

// Key of position i in a pass: the column of entry i (first pass) or the carried key.
template <typename I>
__device__ __forceinline__ uint32_t tkey(const I* col, const uint32_t* keys_in, int32_t i) {
    return keys_in ? keys_in[i] : (uint32_t)idx_of(col[i]);
}

template <typename I>
__global__ void __launch_bounds__(kTThreads)
tr_hist_kernel(const I* __restrict__ col, const uint32_t* __restrict__ keys_in, int32_t nnz, int shift,
               uint32_t* __restrict__ hist) {
    __shared__ uint32_t cnt[kTRadix];
    cnt[threadIdx.x] = 0;
    __syncthreads();
    const int32_t base = blockIdx.x * kTTile;
    for (int r = 0; r < kTRounds; ++r) {
        const int32_t i = base + r * kTThreads + threadIdx.x;
        if (i < nnz) atomicAdd(&cnt[(tkey(col, keys_in, i) >> shift) & (kTRadix - 1)], 1u);
    }
    __syncthreads();
    hist[threadIdx.x * gridDim.x + blockIdx.x] = cnt[threadIdx.x];
}

// Exclusive scan, in place, of `total` uint32 counters with one block.
__global__ void __launch_bounds__(kTScanThreads) tr_scan_kernel(uint32_t* __restrict__ hist, int32_t total) {
    __shared__ uint32_t part[kTScanThreads];
    const int32_t per = (total + kTScanThreads - 1) / kTScanThreads;
    const int32_t b = threadIdx.x * per, e = min(total, b + per);
    uint32_t s = 0;
    for (int32_t i = b; i < e; ++i) s += hist[i];
    part[threadIdx.x] = s;
    __syncthreads();
    for (int off = 1; off < kTScanThreads; off <<= 1) {
        const uint32_t v = threadIdx.x >= off ? part[threadIdx.x - off] : 0;
        __syncthreads();
        part[threadIdx.x] += v;
        __syncthreads();
    }
    uint32_t run = threadIdx.x ? part[threadIdx.x - 1] : 0;
    for (int32_t i = b; i < e; ++i) {
        const uint32_t c = hist[i];
        hist[i] = run;
        run += c;
    }
}

// Row of entry k: the last i with ro[i] <= k (rows with no entries are skipped over).
__device__ __forceinline__ int32_t row_of(const int32_t* __restrict__ ro, int32_t m, int32_t k) {
    int32_t lo = 0, hi = m;  // ro[lo] <= k < ro[hi]
    while (hi - lo > 1) {
        const int32_t mid = (lo + hi) >> 1;
        if (__ldg(ro + mid) <= k) lo = mid;
        else hi = mid;
    }
    return lo;
}

// Stable scatter of one pass. Intermediate passes carry (key, entry index); the last pass
// writes the entry's row id, value and index at its final position.
template <typename T, typename I>
__global__ void __launch_bounds__(kTThreads)
tr_scatter_kernel(const I* __restrict__ col, const uint32_t* __restrict__ keys_in, const int32_t* __restrict__ vals_in,
                  int32_t nnz, int shift, const uint32_t* __restrict__ offsets, uint32_t* __restrict__ keys_out,
                  int32_t* __restrict__ vals_out, const int32_t* __restrict__ ro, int32_t m,
                  const T* __restrict__ val, I* __restrict__ row_t, T* __restrict__ val_t, int32_t* __restrict__ perm) {
    __shared__ uint32_t warp_cnt[kTThreads / 32][kTRadix];
    __shared__ uint32_t running[kTRadix];
    __shared__ uint32_t dbase[kTRadix];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    running[tid] = 0;
    dbase[tid] = offsets[tid * gridDim.x + blockIdx.x];
    const uint32_t lt_mask = (1u << lane) - 1u;
    const int32_t base = blockIdx.x * kTTile;
    const bool last = keys_out == nullptr;
    for (int r = 0; r < kTRounds; ++r) {
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
            if (!last) {
                keys_out[pos] = key;
                vals_out[pos] = k;
            } else {
                row_t[pos] = static_cast<I>(row_of(ro, m, k));
                if (val_t) val_t[pos] = val[k];
                if (perm) perm[pos] = k;
            }
        }
        __syncthreads();
    }
}

template <typename T>
__global__ void __launch_bounds__(256) permute_values_kernel(const T* __restrict__ val, const int32_t* __restrict__ perm,
                                                            int32_t nnz, T* __restrict__ val_t) {
    for (int32_t p = blockIdx.x * blockDim.x + threadIdx.x; p < nnz; p += gridDim.x * blockDim.x)
        val_t[p] = val[perm[p]];
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
    cudaError_t e = cudaMemsetAsync(ro_t, 0, (size_t)(n + 1) * sizeof(int32_t), s);
    if (e != cudaSuccess) return e;
    if (nnz == 0) return cudaSuccess;
    const int sms = device_props().sm_count;
    const int gcount = (int)min64((int64_t)sms * 8, ((int64_t)nnz + 255) / 256);
    col_count_kernel<I><<<gcount, 256, 0, s>>>(col, nnz, ro_t);
    scan_counts_kernel<<<1, kTScanThreads, 0, s>>>(ro_t, n + 1);
    int launches = 2;

    const int passes = max(1, (bits_for((uint32_t)(n - 1)) + 7) / 8);
    const int nb = (nnz + kTTile - 1) / kTTile;
    const size_t arr = align_up((size_t)nnz * 4, 256);
    char* w = static_cast<char*>(ws);
    uint32_t* keys[2] = {reinterpret_cast<uint32_t*>(w), reinterpret_cast<uint32_t*>(w + arr)};
    int32_t* vals[2] = {reinterpret_cast<int32_t*>(w + 2 * arr), reinterpret_cast<int32_t*>(w + 3 * arr)};
    uint32_t* hist = reinterpret_cast<uint32_t*>(w + 4 * arr);
    for (int p = 0; p < passes; ++p) {
        const uint32_t* kin = p == 0 ? nullptr : keys[(p - 1) & 1];
        const int32_t* vin = p == 0 ? nullptr : vals[(p - 1) & 1];
        const bool last = p == passes - 1;
        tr_hist_kernel<I><<<nb, kTThreads, 0, s>>>(col, kin, nnz, 8 * p, hist);
        tr_scan_kernel<<<1, kTScanThreads, 0, s>>>(hist, nb * kTRadix);
        tr_scatter_kernel<T, I><<<nb, kTThreads, 0, s>>>(col, kin, vin, nnz, 8 * p, hist, last ? nullptr : keys[p & 1],
                                                         last ? nullptr : vals[p & 1], ro, m, val, row_t, val_t, perm);
        launches += 3;
    }
    count_launches(launches);
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
    const size_t nb = ((size_t)nnz + kTTile - 1) / kTTile;
    return 4 * arr + align_up(nb * kTRadix * 4, 256);
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
