// SpMM, general path: C = A * B with A an m x k CSR matrix, B dense k x n row-major and C
// dense m x n row-major, accumulated in fp32 and rounded once to the operand dtype.
//
// spops README ("Sparse Operations (spops)"), section "Sparse Matrix Multiplication
// (SpMM) [dense = sparse x dense]".
//
// Row scheduler: rows are visited in row_idx order (nnz descending) and split by the row
// bins into
//   * long rows (nnz >= kSpmmLongRow): one CTA per (row, 32*V-column chunk); the 8 warps
//     take interleaved slices of the row's entries and their partial sums are combined in
//     shared memory in warp order, so the result does not depend on timing;
//   * short and empty rows: a group of G lanes per (row, G*V-column chunk), G the smallest
//     power of two that covers n (at most 32); empty rows write zeros.
// Each lane owns V = 16 / sizeof(T) consecutive output columns and gathers them from B with
// one 16-byte load per entry. The group loads G (col, value) pairs at once, coalesced, and
// broadcasts them with warp shuffles; four B rows are gathered before their FMAs so that
// four loads are in flight per lane. Correctness does not depend on row_idx being sorted:
// any row is valid in any bin, sortedness only balances the work.
#include "common.cuh"
#include "internal.h"

namespace spops {
namespace {

constexpr int kSpmmThreads = 256;
constexpr int kSpmmWarps = kSpmmThreads / 32;
constexpr int kNarrowN = 16;  // B this narrow takes the warp-per-row streaming kernel

template <typename T, int V>
__device__ __forceinline__ void load_b(const T* __restrict__ Brow, int col0, int N, float (&b)[V]) {
    if constexpr (V == 1) {
        b[0] = col0 < N ? Elt<T>::to_f(Brow[col0]) : 0.f;
    } else {
        if (col0 < N) {
            Elt<T>::unpack(ld_nc_v4(Brow + col0), b);
        } else {
#pragma unroll
            for (int e = 0; e < V; ++e) b[e] = 0.f;
        }
    }
}

// acc += sum over the cnt entries held by lanes src0 .. src0+cnt-1 (col cj, value vj).
template <typename T, int V>
__device__ __forceinline__ void accumulate(float (&acc)[V], int cj, float vj, int cnt, const T* __restrict__ B,
                                           int N, int col0, unsigned mask, int src0) {
    constexpr int U = V == 1 ? 8 : 32 / V;  // B rows gathered before their FMAs (8 for 16-bit, 4 for fp32)
    int j = 0;
    for (; j + U <= cnt; j += U) {
        int c[U];
        float v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            c[u] = __shfl_sync(mask, cj, src0 + j + u);
            v[u] = __shfl_sync(mask, vj, src0 + j + u);
        }
        if constexpr (V == 1) {
            float b[U][V];
#pragma unroll
            for (int u = 0; u < U; ++u) load_b<T, V>(B + (int64_t)c[u] * N, col0, N, b[u]);
#pragma unroll
            for (int u = 0; u < U; ++u)
#pragma unroll
                for (int e = 0; e < V; ++e) acc[e] = fmaf(v[u], b[u][e], acc[e]);
        } else {
            uint4 r[U];  // raw 16-byte slices: 4 registers each, widened at their FMAs
#pragma unroll
            for (int u = 0; u < U; ++u)
                r[u] = col0 < N ? ld_nc_v4(B + (int64_t)c[u] * N + col0) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int u = 0; u < U; ++u) {
                float b[V];
                Elt<T>::unpack(r[u], b);
#pragma unroll
                for (int e = 0; e < V; ++e) acc[e] = fmaf(v[u], b[e], acc[e]);
            }
        }
    }
    for (; j < cnt; ++j) {
        const int c = __shfl_sync(mask, cj, src0 + j);
        const float v = __shfl_sync(mask, vj, src0 + j);
        float b[V];
        load_b<T, V>(B + (int64_t)c * N, col0, N, b);
#pragma unroll
        for (int e = 0; e < V; ++e) acc[e] = fmaf(v, b[e], acc[e]);
    }
}

template <typename T, int V>
__device__ __forceinline__ void store_c(T* __restrict__ Crow, int col0, int N, const float (&acc)[V]) {
    if (col0 >= N) return;
    if constexpr (V == 1) {
        Crow[col0] = Elt<T>::from_f(acc[0]);
    } else {
        *reinterpret_cast<uint4*>(Crow + col0) = Elt<T>::pack(acc);
    }
}

template <typename T, typename I, int V>
__global__ void __launch_bounds__(kSpmmThreads, 4)
spmm_rows_kernel(const T* __restrict__ vals, const int32_t* __restrict__ ro, const I* __restrict__ row_idx,
                 const I* __restrict__ col, const T* __restrict__ B, T* __restrict__ C, int32_t m, int32_t N, int G,
                 const int32_t* __restrict__ bins, const uint8_t* __restrict__ skip, const int32_t* __restrict__ order) {
    __shared__ float red[kSpmmWarps][32 * V];
    __shared__ uint8_t skip_cache[kSkipCache];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    pdl_trigger();
    pdl_wait();
    static_assert(kPanelRows == 128, "skip flags are per 128 positions");
    const SkipFlags skipped = load_skip_flags(skip, m, skip_cache);
    if (skipped.all) return;  // every row is on the tensor cores
    const int32_t n_long = bins[1];

    // ---- long rows: one CTA per (row, chunk of 32*V columns). Items are numbered row-major
    // over positions [0, n_long) and dealt round-robin to the CTAs; the loop walks the panels
    // carrying this CTA's next item: a panel without one costs a compare, a skipped panel
    // (on the tensor cores) one division to jump past it, an item a 32-bit division.
    {
        const int chunk = 32 * V;
        const int nch = (N + chunk - 1) / chunk;
        const int64_t g = gridDim.x;
        const int64_t items = (int64_t)n_long * nch;
        int64_t item = blockIdx.x;
        for (int64_t pan0 = 0; pan0 < n_long && item < items; pan0 += kPanelRows) {
            const int64_t i0 = pan0 * nch, i1 = min64(n_long, pan0 + kPanelRows) * nch;
            if (item >= i1) continue;  // uniform across the CTA
            if (skipped(pan0)) {
                item += (i1 - item + g - 1) / g * g;
                continue;
            }
            for (; item < i1; item += g) {
                const int64_t rel = item - i0;  // < 128 * nch
                const int32_t p = (int32_t)(pan0 + (uint32_t)rel / (uint32_t)nch);
                const int c = (int)((uint32_t)rel % (uint32_t)nch);
                const int row = order ? order[p] : idx_of(row_idx[p]);
                const int32_t k0 = ro[row], k1 = ro[row + 1];
                const int col0 = c * chunk + lane * V;
                float acc[V];
#pragma unroll
                for (int e = 0; e < V; ++e) acc[e] = 0.f;
                for (int32_t kb = k0 + warp * 32; kb < k1; kb += kSpmmThreads) {
                    const int32_t kk = kb + lane;
                    int cj = 0;
                    float vj = 0.f;
                    if (kk < k1) {
                        cj = idx_of(col[kk]);
                        vj = Elt<T>::to_f(vals[kk]);
                    }
                    accumulate<T, V>(acc, cj, vj, min(32, k1 - kb), B, N, col0, 0xffffffffu, 0);
                }
#pragma unroll
                for (int e = 0; e < V; ++e) red[warp][lane * V + e] = acc[e];
                __syncthreads();
                if (warp == 0) {
#pragma unroll
                    for (int e = 0; e < V; ++e) {
                        float sum = red[0][lane * V + e];
#pragma unroll
                        for (int w = 1; w < kSpmmWarps; ++w) sum += red[w][lane * V + e];
                        acc[e] = sum;
                    }
                    store_c<T, V>(C + (int64_t)row * N, col0, N, acc);
                }
                __syncthreads();
            }
        }
    }

    // ---- short and empty rows: a group of G lanes per (row, chunk of G*V columns)
    {
        const int chunk = G * V;
        const int nch = (N + chunk - 1) / chunk;
        const int gpw = 32 / G;
        const int gw = lane / G, gl = lane % G;
        const unsigned gmask = G == 32 ? 0xffffffffu : (((1u << G) - 1u) << (gw * G));
        const int64_t gid = ((int64_t)blockIdx.x * kSpmmWarps + warp) * gpw + gw;
        const int64_t ngroups = (int64_t)gridDim.x * kSpmmWarps * gpw;
        const int64_t items = (int64_t)(m - n_long) * nch;
        const bool items32 = items < (int64_t)0x7fffffff;
        // Items go in batches of kBatch: their row ids, then their row offsets, are loaded
        // together before any is processed, so short and empty rows do not wait on one
        // dependent load chain each.
        constexpr int kBatch = 2;
        for (int64_t base = gid; base < items; base += kBatch * ngroups) {
            int rowq[kBatch], cq[kBatch];
            int32_t k0q[kBatch], k1q[kBatch];
            bool live[kBatch];
#pragma unroll
            for (int q = 0; q < kBatch; ++q) {
                const int64_t item = base + q * ngroups;
                int32_t p;
                if (items32) {  // 32-bit division where the item numbers fit
                    const uint32_t it = (uint32_t)min64(item, items);
                    p = n_long + (int32_t)(it / (uint32_t)nch);
                    cq[q] = (int)(it % (uint32_t)nch);
                } else {
                    p = n_long + (int32_t)(item / nch);
                    cq[q] = (int)(item % nch);
                }
                live[q] = item < items && !skipped(p);  // uniform across the group
                rowq[q] = live[q] ? (order ? order[p] : idx_of(row_idx[p])) : 0;
            }
#pragma unroll
            for (int q = 0; q < kBatch; ++q) {
                k0q[q] = live[q] ? ro[rowq[q]] : 0;
                k1q[q] = live[q] ? ro[rowq[q] + 1] : 0;
            }
#pragma unroll
            for (int q = 0; q < kBatch; ++q) {
                if (!live[q]) continue;
                const int32_t k0 = k0q[q], k1 = k1q[q];
                const int col0 = cq[q] * chunk + gl * V;
                float acc[V];
#pragma unroll
                for (int e = 0; e < V; ++e) acc[e] = 0.f;
                for (int32_t kb = k0; kb < k1; kb += G) {
                    const int32_t kk = kb + gl;
                    int cj = 0;
                    float vj = 0.f;
                    if (kk < k1) {
                        cj = idx_of(col[kk]);
                        vj = Elt<T>::to_f(vals[kk]);
                    }
                    accumulate<T, V>(acc, cj, vj, min(G, k1 - kb), B, N, col0, gmask, gw * G);
                }
                store_c<T, V>(C + (int64_t)rowq[q] * N, col0, N, acc);
            }
        }
    }

}

// Narrow B (N <= 16, SpMV at N = 1): streaming A dominates, so a warp takes one row at a
// time and its lanes read the row's (col, val) pairs coalesced, 32 at a time, each lane
// gathering its entries' B rows (N elements, at most 64 bytes) and accumulating N fp32
// sums; a butterfly of shuffles then adds the 32 lanes' sums in a fixed order and lanes
// 0 .. N-1 write the row's outputs. NV 16-byte vectors per B row when N * sizeof(T) is a
// multiple of 16 and B is aligned; NV = 0 loads N scalars; NV = -1 is N = 1 (eight entries
// in flight per lane). Rows go round-robin over the warps in row_idx order (long rows
// first); empty rows write zeros.
template <typename T, typename I, int NV>
__global__ void __launch_bounds__(kSpmmThreads)
spmm_narrow_kernel(const T* __restrict__ vals, const int32_t* __restrict__ ro, const I* __restrict__ row_idx,
                   const I* __restrict__ col, const T* __restrict__ B, T* __restrict__ C, int32_t m, int32_t N,
                   const uint8_t* __restrict__ skip) {
    constexpr int kMaxN = 16;
    constexpr int VE = 16 / (int)sizeof(T);  // elements per 16-byte vector
    const int lane = threadIdx.x & 31;
    pdl_trigger();
    pdl_wait();
    const int64_t warp = ((int64_t)blockIdx.x * kSpmmThreads + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * kSpmmThreads) >> 5;
    for (int64_t p = warp; p < m; p += nwarps) {
        if (skip && skip[p / kPanelRows]) continue;  // uniform across the warp
        const int row = idx_of(row_idx[p]);
        const int32_t k0 = ro[row], k1 = ro[row + 1];
        float acc[kMaxN];
#pragma unroll
        for (int c = 0; c < kMaxN; ++c) acc[c] = 0.f;
        // kU entries per lane per round: their (col, val) loads, then their B rows, are all
        // in flight before the first FMA.
        constexpr int kU = NV > 2 ? 2 : (NV < 0 ? 8 : 4);
        for (int32_t kb = k0; kb < k1; kb += 32 * kU) {
            int jq[kU];
            float aq[kU];
            bool ok[kU];
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int32_t k = kb + u * 32 + lane;
                ok[u] = k < k1;
                jq[u] = ok[u] ? idx_of(col[k]) : 0;
                aq[u] = ok[u] ? Elt<T>::to_f(vals[k]) : 0.f;
            }
            if constexpr (NV < 0) {  // N == 1: gather kU values, then multiply
                float bv[kU];
#pragma unroll
                for (int u = 0; u < kU; ++u) bv[u] = ok[u] ? Elt<T>::to_f(B[jq[u]]) : 0.f;
#pragma unroll
                for (int u = 0; u < kU; ++u) acc[0] = fmaf(aq[u], bv[u], acc[0]);
            } else if constexpr (NV > 0) {
                uint4 raw[kU][NV];
#pragma unroll
                for (int u = 0; u < kU; ++u)
#pragma unroll
                    for (int q = 0; q < NV; ++q)  // past the row end: zeros, so nothing is added
                        raw[u][q] = ok[u] ? ld_nc_v4(B + (int64_t)jq[u] * N + q * VE) : make_uint4(0, 0, 0, 0);
#pragma unroll
                for (int u = 0; u < kU; ++u)
#pragma unroll
                    for (int q = 0; q < NV; ++q) {
                        float f[VE];
                        Elt<T>::unpack(raw[u][q], f);
#pragma unroll
                        for (int e = 0; e < VE; ++e) acc[q * VE + e] = fmaf(aq[u], f[e], acc[q * VE + e]);
                    }
            } else {
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    if (!ok[u]) continue;
                    const T* b = B + (int64_t)jq[u] * N;
#pragma unroll
                    for (int c = 0; c < kMaxN; ++c)
                        if (c < N) acc[c] = fmaf(aq[u], Elt<T>::to_f(b[c]), acc[c]);
                }
            }
        }
        constexpr int kUsed = NV > 0 ? NV * VE : (NV < 0 ? 1 : kMaxN);
#pragma unroll
        for (int c = 0; c < kUsed; ++c) {
            if (NV == 0 && c >= N) break;
            float x = acc[c];
#pragma unroll
            for (int o = 16; o; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
            acc[c] = x;
        }
        T* crow = C + (int64_t)row * N;
#pragma unroll
        for (int c = 0; c < kUsed; ++c)
            if (lane == c && c < N) crow[c] = Elt<T>::from_f(acc[c]);
    }
}

template <typename T, typename I>
cudaError_t run_narrow(const void* vals, const int32_t* ro, const void* row_idx, const void* col, int32_t m,
                       const void* B, int32_t N, void* C, const uint8_t* skip, cudaStream_t s) {
    constexpr int VE = 16 / (int)sizeof(T);
    const int grid = (int)max64(1, min64((int64_t)device_props().sm_count * 8, ((int64_t)m + 7) / 8));
    const bool vec = (N % VE) == 0 && (uintptr_t)B % 16 == 0;
    const T* v = static_cast<const T*>(vals);
    const I* ri = static_cast<const I*>(row_idx);
    const I* ci = static_cast<const I*>(col);
    const T* b = static_cast<const T*>(B);
    T* c = static_cast<T*>(C);
    cudaError_t e;
    if (N == 1) e = launch_pdl(spmm_narrow_kernel<T, I, -1>, grid, kSpmmThreads, 0, s, v, ro, ri, ci, b, c, m, N, skip);
    else if (vec && N / VE == 1) e = launch_pdl(spmm_narrow_kernel<T, I, 1>, grid, kSpmmThreads, 0, s, v, ro, ri, ci, b, c, m, N, skip);
    else if (vec && N / VE == 2) e = launch_pdl(spmm_narrow_kernel<T, I, 2>, grid, kSpmmThreads, 0, s, v, ro, ri, ci, b, c, m, N, skip);
    else if (vec && N / VE == 4) e = launch_pdl(spmm_narrow_kernel<T, I, 4>, grid, kSpmmThreads, 0, s, v, ro, ri, ci, b, c, m, N, skip);
    else e = launch_pdl(spmm_narrow_kernel<T, I, 0>, grid, kSpmmThreads, 0, s, v, ro, ri, ci, b, c, m, N, skip);
    if (e != cudaSuccess) return e;
    count_launches(1);
    return cudaGetLastError();
}

int pow2_cover(int64_t units) {
    int g = 1;
    while (g < 32 && g < units) g <<= 1;
    return g;
}

template <typename T, typename I>
cudaError_t run(const void* vals, const int32_t* ro, const void* row_idx, const void* col, int32_t m,
                const void* B, int32_t N, void* C, const int32_t* bins, const uint8_t* skip, const int32_t* order,
                cudaStream_t s) {
    if (N <= kNarrowN) return run_narrow<T, I>(vals, ro, row_idx, col, m, B, N, C, skip, s);
    constexpr int VV = Elt<T>::kVec;
    const bool vec = ((int64_t)N * sizeof(T)) % 16 == 0 && (uintptr_t)B % 16 == 0 && (uintptr_t)C % 16 == 0;
    auto kern = vec ? spmm_rows_kernel<T, I, VV> : spmm_rows_kernel<T, I, 1>;
    const int V = vec ? VV : 1;
    const int G = pow2_cover(((int64_t)N + V - 1) / V);
    int occ = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kSpmmThreads, 0);
    if (e != cudaSuccess) return e;
    const int grid = device_props().sm_count * (occ > 0 ? occ : 1);
    // Beside tensor-core panels (skip flags set) the kernel runs on a side stream after an
    // event wait: an ordinary launch there; on the caller's stream a programmatic dependent.
    if (skip)
        kern<<<grid, kSpmmThreads, 0, s>>>(static_cast<const T*>(vals), ro, static_cast<const I*>(row_idx),
                                           static_cast<const I*>(col), static_cast<const T*>(B), static_cast<T*>(C), m,
                                           N, G, bins, skip, order);
    else
        e = launch_pdl(kern, grid, kSpmmThreads, 0, s, static_cast<const T*>(vals), ro, static_cast<const I*>(row_idx),
                       static_cast<const I*>(col), static_cast<const T*>(B), static_cast<T*>(C), m, N, G, bins, skip,
                       order);
    if (e != cudaSuccess) return e;
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_spmm_general(int dt, int it, const void* vals, const int32_t* ro, const void* row_idx,
                                const void* col, int32_t m, int32_t k, const void* B, int32_t n, void* C,
                                const int32_t* bins, const uint8_t* skip, const int32_t* order, cudaStream_t s) {
    (void)k;
    if (dt == kF32)
        return it == kIdx16 ? run<float, uint16_t>(vals, ro, row_idx, col, m, B, n, C, bins, skip, order, s)
                            : run<float, int32_t>(vals, ro, row_idx, col, m, B, n, C, bins, skip, order, s);
    if (dt == kF16)
        return it == kIdx16 ? run<__half, uint16_t>(vals, ro, row_idx, col, m, B, n, C, bins, skip, order, s)
                            : run<__half, int32_t>(vals, ro, row_idx, col, m, B, n, C, bins, skip, order, s);
    return it == kIdx16 ? run<__nv_bfloat16, uint16_t>(vals, ro, row_idx, col, m, B, n, C, bins, skip, order, s)
                        : run<__nv_bfloat16, int32_t>(vals, ro, row_idx, col, m, B, n, C, bins, skip, order, s);
}

}  // namespace spops
