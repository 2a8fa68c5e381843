// csr_add: C = B + A, A an m x n CSR matrix, B and C dense m x n row-major (C may be B).
//
// spops README ("Sparse Operations (spops)"), section "Sparse Addition [dense = sparse +
// dense]": a sparse CSR matrix is added to a dense matrix.
//
// The operation is a dense stream (2 * m * n * sizeof(T) bytes) with a sparse scatter on
// top, so the kernel is built around the copy engine: each CTA owns a ring of 16 KB shared
// memory stages. One thread moves a tile of B into a stage with a 1-D bulk async copy
// (TMA, completion on an mbarrier), the CTA adds the tile's CSR entries in place, and the
// same thread streams the stage back to C with a bulk store. Tiles are flat 16 KB slices
// of the row-major matrix, so the only alignment requirement is a 16-byte aligned B and
// C; otherwise a plain-load variant of the same kernel runs.
//
// A tile covers the tail of row r0, whole rows and the head of row r1. Columns increase
// inside a row, so when an edge row holds more than kSearchMin entries two warps find the
// tile's first entry in r0 and its end in r1 by a 32-way search (each step one load per
// lane and a ballot), and a row wider than a tile is scanned once in total, not once per
// tile it spans.
//
// Each entry is added in fp32 and rounded once to T. For fp32 that is the IEEE sum. For
// fp16/bf16 the fp32 sum of two such values is rounded twice (to fp32, then to T), which
// gives the correctly rounded result because fp32 has at least 2p+2 significand bits
// (Figueroa's double-rounding theorem), so the output matches the exact sum rounded once.
#include "common.cuh"
#include "internal.h"

namespace spops {
namespace {

constexpr int kAddThreads = 256;
constexpr int kAddTileBytes = 16384;
constexpr int kAddStages = 3;
constexpr int kAddSmem = kAddTileBytes * kAddStages;
constexpr int kRoCache = 512;  // row offsets of a tile kept in shared memory (tiles spanning fewer rows)
constexpr int kPre = 4;        // entries per thread loaded before the tile arrives
constexpr int kSearchMin = 2 * kAddThreads;  // edge rows with more entries are searched

// First k in [lo, hi) with col[k] >= c (hi if none), columns increasing; all 32 lanes call it
// with the same arguments and get the same result. Each step samples 32 evenly spaced
// entries and keeps the gap in which the columns reach c.
template <typename I>
__device__ __forceinline__ int32_t warp_lower_bound(const I* __restrict__ col, int32_t lo, int32_t hi, int32_t c,
                                                    int lane) {
    while (hi - lo > 32) {
        const int32_t step = (hi - lo + 31) / 32;
        const int32_t x = lo + lane * step;
        const bool below = x < hi && idx_of(col[x]) < c;
        const int cnt = __popc(__ballot_sync(0xffffffffu, below));
        if (cnt == 0) return lo;
        const int32_t nlo = lo + (cnt - 1) * step + 1;
        hi = min(hi, lo + cnt * step);
        lo = nlo;
    }
    const int32_t x = lo + lane;
    const bool below = x < hi && idx_of(col[x]) < c;
    return lo + __popc(__ballot_sync(0xffffffffu, below));
}

template <typename T, typename I, bool kBulk>
__global__ void __launch_bounds__(kAddThreads) csr_add_kernel(const T* __restrict__ vals,
                                                               const int32_t* __restrict__ ro,
                                                               const I* __restrict__ col, int32_t n, const T* B,
                                                               T* C, int64_t total, int* err) {
    extern __shared__ __align__(1024) unsigned char smem[];
    __shared__ __align__(8) uint64_t full_bar[kAddStages];
    __shared__ int32_t ro_s[kRoCache];
    __shared__ int32_t s_edge[2];
    constexpr int64_t E = kAddTileBytes / sizeof(T);
    const int tid = threadIdx.x;
    pdl_trigger();
    pdl_wait();
    const int64_t ntiles = (total + E - 1) / E;
    const int64_t my_tiles = (int64_t)blockIdx.x < ntiles ? (ntiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;

    auto stage = [&](int s) { return reinterpret_cast<T*>(smem + s * kAddTileBytes); };
    auto tile_elems = [&](int64_t t) { return (int)min64(E, total - t * E); };
    auto bulk_elems = [&](int cnt) { return (int)((cnt * (int)sizeof(T)) / 16 * 16 / (int)sizeof(T)); };
    auto issue_load = [&](int64_t j, int s) {
        const int64_t t = blockIdx.x + j * gridDim.x;
        const int be = bulk_elems(tile_elems(t));
        const uint32_t bar = smem_u32(&full_bar[s]);
        mbar_arrive_expect_tx(bar, (uint32_t)(be * sizeof(T)));
        if (be) bulk_g2s(smem_u32(stage(s)), B + t * E, (uint32_t)(be * sizeof(T)), bar);
    };

    if (kBulk) {
        if (tid == 0) {
            for (int s = 0; s < kAddStages; ++s) mbar_init(smem_u32(&full_bar[s]), 1);
            fence_mbar_init();
        }
        __syncthreads();
        if (tid == 0)
            for (int64_t j = 0; j < min64(kAddStages, my_tiles); ++j) issue_load(j, (int)j);
    }

    for (int64_t j = 0; j < my_tiles; ++j) {
        const int s = (int)(j % kAddStages);
        const int64_t t = blockIdx.x + j * gridDim.x;
        const int64_t f0 = t * E;
        const int cnt = tile_elems(t);
        const int64_t f1 = f0 + cnt;
        T* buf = stage(s);
        // Entries whose flat position falls in [f0, f1): rows r0..r1, CSR range [kb, ke).
        // Their row offsets go to shared memory and the first kPre entries per thread are
        // loaded before waiting for the tile, so those loads overlap the tile's copy.
        const int32_t r0 = (int32_t)(f0 / n), r1 = (int32_t)((f1 - 1) / n);
        const int nro = r1 - r0 + 2;
        const bool cached = nro <= kRoCache;
        if (cached)
            for (int x = tid; x < nro; x += kAddThreads) ro_s[x] = ro[r0 + x];
        __syncthreads();
        int32_t kb = cached ? ro_s[0] : ro[r0];
        int32_t ke = cached ? ro_s[nro - 1] : ro[r1 + 1];
        {
            // entries of r0 before the tile's first column and of r1 from its end column on
            const int32_t r0_end = cached ? ro_s[1] : ro[r0 + 1];
            const int32_t r1_beg = cached ? ro_s[nro - 2] : ro[r1];
            const bool w0 = r0_end - kb > kSearchMin, w1 = ke - r1_beg > kSearchMin;
            if (w0 || w1) {  // uniform over the CTA
                const int warp = tid >> 5, lane = tid & 31;
                if (warp == 0 && w0)
                    s_edge[0] = warp_lower_bound(col, kb, r0_end, (int32_t)(f0 - (int64_t)r0 * n), lane);
                if (warp == 1 && w1)
                    s_edge[1] = warp_lower_bound(col, r1_beg, ke, (int32_t)(f1 - (int64_t)r1 * n), lane);
                __syncthreads();
                if (w0) kb = s_edge[0];
                if (w1) ke = s_edge[1];  // s_edge is next written after two more barriers
            }
        }
        auto row_of = [&](int32_t k) {  // largest r in [r0, r1] with ro[r] <= k
            int32_t lo = 0, hi = nro - 2;
            while (lo < hi) {
                const int32_t mid = (lo + hi + 1) >> 1;
                if ((cached ? ro_s[mid] : ro[r0 + mid]) <= k) lo = mid;
                else hi = mid - 1;
            }
            return r0 + lo;
        };
        int cq[kPre];
        float vq[kPre];
#pragma unroll
        for (int q = 0; q < kPre; ++q) {
            const int32_t k = kb + tid + q * kAddThreads;
            cq[q] = k < ke ? idx_of(col[k]) : 0;
            vq[q] = k < ke ? Elt<T>::to_f(vals[k]) : 0.f;
        }
        bool ok = true;
        if (kBulk) {
            ok = mbar_wait(smem_u32(&full_bar[s]), (uint32_t)((j / kAddStages) & 1), err);
            const int be = bulk_elems(cnt);
            if (tid < cnt - be) buf[be + tid] = B[f0 + be + tid];
        } else {
            for (int e = tid; e < cnt; e += kAddThreads) buf[e] = B[f0 + e];
        }
        if (!__syncthreads_and(ok)) {
            if (tid == 0) bulk_wait<0>();
            return;
        }
        auto add = [&](int32_t k, int c, float a) {
            const int64_t f = (int64_t)row_of(k) * n + c;
            if (f >= f0 && f < f1) {
                T& x = buf[f - f0];
                x = Elt<T>::from_f(Elt<T>::to_f(x) + a);
            }
        };
#pragma unroll
        for (int q = 0; q < kPre; ++q) {
            const int32_t k = kb + tid + q * kAddThreads;
            if (k < ke) add(k, cq[q], vq[q]);
        }
        for (int32_t k = kb + tid + kPre * kAddThreads; k < ke; k += kAddThreads)
            add(k, idx_of(col[k]), Elt<T>::to_f(vals[k]));
        if (kBulk) fence_proxy_async_smem();
        __syncthreads();
        if (kBulk) {
            if (tid == 0) {
                const int be = bulk_elems(cnt);
                if (be) {
                    bulk_s2g(C + f0, smem_u32(buf), (uint32_t)(be * sizeof(T)));
                    bulk_commit();
                }
                for (int e = be; e < cnt; ++e) C[f0 + e] = buf[e];
                if (j + kAddStages < my_tiles) {
                    bulk_wait_read<0>();  // stage s is free once the store has read it
                    issue_load(j + kAddStages, s);
                }
            }
        } else {
            for (int e = tid; e < cnt; e += kAddThreads) C[f0 + e] = buf[e];
            __syncthreads();
        }
    }
    if (kBulk && tid == 0) bulk_wait<0>();
}

template <typename T, typename I>
cudaError_t run(const void* vals, const int32_t* ro, const void* col, int32_t m, int32_t n, const void* B, void* C,
                cudaStream_t s) {
    const int64_t total = (int64_t)m * n;
    if (total == 0) return cudaSuccess;
    const int64_t E = kAddTileBytes / sizeof(T);
    const int64_t ntiles = (total + E - 1) / E;
    const DeviceProps& p = device_props();
    const int grid = (int)min64(ntiles, (int64_t)p.sm_count * 4);
    const bool bulk = ((uintptr_t)B % 16 == 0) && ((uintptr_t)C % 16 == 0);
    auto kern = bulk ? csr_add_kernel<T, I, true> : csr_add_kernel<T, I, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kAddSmem);
    if (e != cudaSuccess) return e;
    e = launch_pdl(kern, grid, kAddThreads, kAddSmem, s, static_cast<const T*>(vals), ro, static_cast<const I*>(col), n,
                   static_cast<const T*>(B), static_cast<T*>(C), total, device_error_word());
    if (e != cudaSuccess) return e;
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_csr_add(int dt, int it, const void* vals, const int32_t* ro, const void* col, int32_t m,
                           int32_t n, int32_t nnz, const void* B, void* C, cudaStream_t s) {
    (void)nnz;
    if (dt == kF32) return it == kIdx16 ? run<float, uint16_t>(vals, ro, col, m, n, B, C, s)
                                        : run<float, int32_t>(vals, ro, col, m, n, B, C, s);
    if (dt == kF16) return it == kIdx16 ? run<__half, uint16_t>(vals, ro, col, m, n, B, C, s)
                                        : run<__half, int32_t>(vals, ro, col, m, n, B, C, s);
    return it == kIdx16 ? run<__nv_bfloat16, uint16_t>(vals, ro, col, m, n, B, C, s)
                        : run<__nv_bfloat16, int32_t>(vals, ro, col, m, n, B, C, s);
}

}  // namespace spops
