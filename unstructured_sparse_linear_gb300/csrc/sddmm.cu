// SDDMM, general path: out[k] = sum_t A[i, t] * BT[col[k], t] for every entry k (row i)
// of an m x n CSR mask; A is m x kd and BT is n x kd, both row-major; fp32 accumulation,
// one rounding to the operand dtype.
//
// spops README ("Sparse Operations (spops)"), section "Sampled Dense-Dense Matrix
// Multiplication (SDDMM) [sparse = dense x dense]": the first kernel listed there works
// for any sparsity pattern; BT is the transposed right operand.
//
// Row scheduler: rows in row_idx order (longest first), split by the row bins into
//   * long rows (nnz >= kSddmmLongRow): one CTA per row, its 8 warps take interleaved
//     batches of entries, so all of them stream the same A row through L1;
//   * short rows: a group of G lanes per row (G covers kd in 16-byte vectors, at most 32);
//     where rows are fewer than groups, a team of P consecutive groups of one CTA splits each
//     row's entries evenly (sharing its A row through L1); empty rows cost one row_offsets read.
// Both deal rows in bands of one row per CTA (group, team), the direction reversing every band:
// with the rows sorted by length, whoever took one of the longest rows of a band takes one of
// the shortest of the next, so the work per warp evens out even at a few rows each.
// A batch holds NB entries: the group walks kd once, loading each A vector once and the NB
// BT vectors beside it, keeps NB per-lane partial dot products and finishes them with an
// xor-shuffle butterfly inside the group. Empty rows are skipped.
// The gathers come from L2 and their latency, not L2 bandwidth, sets the pace; NB = 4 at 64
// registers (4 CTAs, 32 warps per SM) keeps more bytes in flight per SM than NB = 8 at 80
// registers (3 CTAs), and more CTAs at fewer registers spill.
#include "common.cuh"
#include "internal.h"

namespace spops {
namespace {

constexpr int kSddmmThreads = 256;
constexpr int kSddmmWarps = kSddmmThreads / 32;
constexpr int kNB = 4;  // entries per batch: 1 A load + up to 4 BT loads per lane per K step

// Raw operand words: one 16-byte vector (V elements), or one element for the scalar path.
template <typename T, int V>
struct Raw {
    uint4 v;
};
template <typename T>
struct Raw<T, 1> {
    T v;
};

template <typename T, int V>
__device__ __forceinline__ Raw<T, V> load_raw(const T* __restrict__ p) {
    Raw<T, V> r;
    if constexpr (V == 1) r.v = *p;
    else r.v = ld_nc_v4(p);
    return r;
}

template <typename T, int V>
__device__ __forceinline__ void widen(const Raw<T, V>& r, float (&f)[V]) {
    if constexpr (V == 1) f[0] = Elt<T>::to_f(r.v);
    else Elt<T>::unpack(r.v, f);
}

template <typename T, typename I, int V>
__device__ __forceinline__ void sddmm_batch(int row, int32_t kb, int cnt, const I* __restrict__ col,
                                            const T* __restrict__ A, const T* __restrict__ BT,
                                            T* __restrict__ out, int32_t kd, int G, int gl, unsigned gmask) {
    int c[kNB];
#pragma unroll
    for (int j = 0; j < kNB; ++j) c[j] = j < cnt ? idx_of(col[kb + j]) : 0;
    float acc[kNB];
#pragma unroll
    for (int j = 0; j < kNB; ++j) acc[j] = 0.f;
    const T* Arow = A + (int64_t)row * kd;
    for (int32_t t = gl * V; t < kd; t += G * V) {
        // all loads of the step first (packed), then widen and multiply
        const Raw<T, V> ar = load_raw<T, V>(Arow + t);
        Raw<T, V> br[kNB];
#pragma unroll
        for (int j = 0; j < kNB; ++j)
            if (j < cnt) br[j] = load_raw<T, V>(BT + (int64_t)c[j] * kd + t);
        float a[V];
        widen<T, V>(ar, a);
#pragma unroll
        for (int j = 0; j < kNB; ++j) {
            if (j < cnt) {
                float b[V];
                widen<T, V>(br[j], b);
#pragma unroll
                for (int e = 0; e < V; ++e) acc[j] = fmaf(a[e], b[e], acc[j]);
            }
        }
    }
#pragma unroll
    for (int j = 0; j < kNB; ++j)
        for (int off = G >> 1; off; off >>= 1) acc[j] += __shfl_xor_sync(gmask, acc[j], off);
    if (gl == 0) {
#pragma unroll
        for (int j = 0; j < kNB; ++j)
            if (j < cnt) out[kb + j] = Elt<T>::from_f(acc[j]);
    }
}

template <typename T, typename I, int V>
__global__ void __launch_bounds__(kSddmmThreads, 4)
sddmm_rows_kernel(const int32_t* __restrict__ ro, const I* __restrict__ row_idx, const I* __restrict__ col,
                  const T* __restrict__ A, const T* __restrict__ BT, T* __restrict__ out, int32_t kd, int G,
                  const int32_t* __restrict__ bins, const uint8_t* __restrict__ skip,
                  const int32_t* __restrict__ order, int lp) {
    __shared__ uint8_t skip_cache[kSkipCache];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    pdl_trigger();
    pdl_wait();
    // Short rows run over every position up to m, not only up to bins[2]: with an unsorted
    // row_idx, rows with entries may sit past the count of non-empty rows.
    const int32_t n_long = bins[1], n_rows = bins[3];
    static_assert(kPanelRows == 128, "skip flags are per 128 positions");
    const SkipFlags skipped = load_skip_flags(skip, n_rows, skip_cache);
    if (skipped.all) return;  // every row is on the tensor cores

    // ---- long rows: a CTA per row, dealt in alternating directions
    const int32_t g = gridDim.x;
    bool odd_l = false;
    for (int32_t b0 = 0; b0 < n_long; b0 += g, odd_l = !odd_l) {
        const int32_t p = b0 + (odd_l ? g - 1 - (int32_t)blockIdx.x : (int32_t)blockIdx.x);
        if (p >= n_long || skipped(p)) continue;
        const int row = order ? order[p] : idx_of(row_idx[p]);
        const int32_t k0 = ro[row], k1 = ro[row + 1];
        for (int32_t kb = k0 + warp * kNB; kb < k1; kb += kSddmmWarps * kNB)
            sddmm_batch<T, I, V>(row, kb, min(kNB, k1 - kb), col, A, BT, out, kd, 32, lane, 0xffffffffu);
    }

    // ---- short rows: a team of 2^lp groups of G lanes per row, dealt in alternating
    // directions; member j of a team takes the j-th of 2^lp even slices of the row's entries
    const int gpw = 32 / G;
    const int gw = lane / G, gl = lane % G;
    const unsigned gmask = G == 32 ? 0xffffffffu : (((1u << G) - 1u) << (gw * G));
    // 32-bit positions: n_rows <= m < 2^31 and the groups of one grid number far fewer
    const int32_t gid = ((int32_t)blockIdx.x * kSddmmWarps + warp) * gpw + gw;
    const int32_t ngroups = (int32_t)gridDim.x * kSddmmWarps * gpw;
    const int32_t team = gid >> lp, nteams = ngroups >> lp;  // 2^lp divides kSddmmWarps * gpw
    const int32_t member = gid & ((1 << lp) - 1);
    const int32_t n_short = n_rows - n_long;
    bool odd = false;
    for (int32_t b0 = 0; b0 < n_short; b0 += nteams, odd = !odd) {
        const int32_t q = b0 + (odd ? nteams - 1 - team : team);
        const int32_t p = n_long + q;
        if (q >= n_short || skipped(p)) continue;
        const int row = order ? order[p] : idx_of(row_idx[p]);
        const int32_t k0 = ro[row], len = ro[row + 1] - k0;
        const int32_t lo = k0 + (int32_t)(((int64_t)len * member) >> lp);
        const int32_t hi = k0 + (int32_t)(((int64_t)len * (member + 1)) >> lp);
        for (int32_t kb = lo; kb < hi; kb += kNB)
            sddmm_batch<T, I, V>(row, kb, min(kNB, hi - kb), col, A, BT, out, kd, G, gl, gmask);
    }
}

template <typename T, typename I>
cudaError_t run(const int32_t* ro, const void* row_idx, const void* col, int32_t m, int32_t kd, const void* A,
                const void* BT, void* out, const int32_t* bins, const uint8_t* skip, const int32_t* order,
                cudaStream_t s) {
    constexpr int VV = Elt<T>::kVec;
    const bool vec = ((int64_t)kd * sizeof(T)) % 16 == 0 && (uintptr_t)A % 16 == 0 && (uintptr_t)BT % 16 == 0;
    auto kern = vec ? sddmm_rows_kernel<T, I, VV> : sddmm_rows_kernel<T, I, 1>;
    const int V = vec ? VV : 1;
    int G = 1;
    while (G < 32 && (int64_t)G * V < kd) G <<= 1;
    int occ = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kSddmmThreads, 0);
    if (e != cudaSuccess) return e;
    const int grid = device_props().sm_count * (occ > 0 ? occ : 1);
    // Team size: with fewer rows than groups, up to 8 groups (one CTA) share a row, so more
    // of the grid works; otherwise one group per row: a row's entries in whole batches of
    // kNB keep the most loads in flight per warp, which sets this gather-bound kernel's pace.
    const int64_t ngroups = (int64_t)grid * kSddmmWarps * (32 / G);
    int lp = 0;
    while (lp < 3 && ((int64_t)m << (lp + 1)) <= ngroups) ++lp;
    // Beside tensor-core panels (skip flags set) the kernel runs on a side stream after an
    // event wait: an ordinary launch there; on the caller's stream a programmatic dependent.
    if (skip)
        kern<<<grid, kSddmmThreads, 0, s>>>(ro, static_cast<const I*>(row_idx), static_cast<const I*>(col),
                                            static_cast<const T*>(A), static_cast<const T*>(BT), static_cast<T*>(out),
                                            kd, G, bins, skip, order, lp);
    else
        e = launch_pdl(kern, grid, kSddmmThreads, 0, s, ro, static_cast<const I*>(row_idx), static_cast<const I*>(col),
                       static_cast<const T*>(A), static_cast<const T*>(BT), static_cast<T*>(out), kd, G, bins, skip,
                       order, lp);
    if (e != cudaSuccess) return e;
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_sddmm_general(int dt, int it, const int32_t* ro, const void* row_idx, const void* col, int32_t m,
                                 int32_t n, int32_t kd, const void* A, const void* BT, void* out,
                                 const int32_t* bins, const uint8_t* skip, const int32_t* order, cudaStream_t s) {
    (void)n;
    if (dt == kF32)
        return it == kIdx16 ? run<float, uint16_t>(ro, row_idx, col, m, kd, A, BT, out, bins, skip, order, s)
                            : run<float, int32_t>(ro, row_idx, col, m, kd, A, BT, out, bins, skip, order, s);
    if (dt == kF16)
        return it == kIdx16 ? run<__half, uint16_t>(ro, row_idx, col, m, kd, A, BT, out, bins, skip, order, s)
                            : run<__half, int32_t>(ro, row_idx, col, m, kd, A, BT, out, bins, skip, order, s);
    return it == kIdx16 ? run<__nv_bfloat16, uint16_t>(ro, row_idx, col, m, kd, A, BT, out, bins, skip, order, s)
                        : run<__nv_bfloat16, int32_t>(ro, row_idx, col, m, kd, A, BT, out, bins, skip, order, s);
}

}  // namespace spops
