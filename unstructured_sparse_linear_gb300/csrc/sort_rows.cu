// Row scheduler support: the nnz-sorted row permutation (row_idx), the row bins that
// split it into long / short / empty rows, and an on-device CSR structure check.
//
// spops README ("Sparse Operations (spops)"), section "Usage": row_idx is a permutation
// of 0..m-1 that sorts the rows by their number of non-zeros. The README does not give
// the direction; this library sorts by nnz descending and keeps ascending row ids among
// rows with equal counts, so long rows come first and empty rows last.
//
// sort_rows: up to 1024 rows, a rank sort in one CTA; up to 16384 rows, a one-CTA radix sort
// in shared memory; beyond, a stable least-significant-digit radix sort on the key
// (nnz - nnz_i), 8 bits per pass: a per-block digit histogram, one exclusive scan over all
// blocks' histograms, and a stable scatter that ranks equal digits inside a block with warp
// match masks. The first pass derives the key from row_offsets directly.
#include "common.cuh"
#include "internal.h"

namespace spops {
namespace {

constexpr int kSortThreads = 256;
constexpr int kSortRounds = 8;
constexpr int kSortTile = kSortThreads * kSortRounds;
constexpr int kRadix = 256;
constexpr int kScanThreads = 1024;

__device__ __forceinline__ uint32_t sort_key(const int32_t* ro, const uint32_t* keys_in, int32_t i,
                                             uint32_t key_base) {
    return keys_in ? keys_in[i] : key_base - (uint32_t)(ro[i + 1] - ro[i]);
}

__global__ void __launch_bounds__(kSortThreads)
radix_hist_kernel(const int32_t* __restrict__ ro, const uint32_t* __restrict__ keys_in, int32_t m,
                  uint32_t key_base, int shift, uint32_t* __restrict__ hist) {
    __shared__ uint32_t cnt[kRadix];
    cnt[threadIdx.x] = 0;
    __syncthreads();
    const int32_t base = blockIdx.x * kSortTile;
    for (int r = 0; r < kSortRounds; ++r) {
        const int32_t i = base + r * kSortThreads + threadIdx.x;
        if (i < m) atomicAdd(&cnt[(sort_key(ro, keys_in, i, key_base) >> shift) & (kRadix - 1)], 1u);
    }
    __syncthreads();
    hist[threadIdx.x * gridDim.x + blockIdx.x] = cnt[threadIdx.x];
}

// Exclusive scan, in place, of `total` counters (a multiple of kRadix) with one block, in
// tiles of kScanThreads x kScanPer: each thread loads its kScanPer consecutive counters with
// independent 16-byte loads (one memory latency per tile, not one per counter), the block
// scans the per-thread sums, and each thread writes its counters' running offsets.
constexpr int kScanPer = 16;
static_assert(kRadix % kScanPer == 0, "tiles hold whole vectors of counters");

__global__ void __launch_bounds__(kScanThreads) radix_scan_kernel(uint32_t* __restrict__ hist, int32_t total) {
    __shared__ uint32_t wsum[kScanThreads / 32];
    __shared__ uint32_t carry_sh;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint32_t carry = 0;  // sum of the tiles before this one
    for (int32_t t0 = 0; t0 < total; t0 += kScanThreads * kScanPer) {
        const int32_t i0 = t0 + tid * kScanPer;
        uint4 v[kScanPer / 4];
#pragma unroll
        for (int q = 0; q < kScanPer / 4; ++q)
            v[q] = i0 < total ? reinterpret_cast<const uint4*>(hist + i0)[q] : make_uint4(0u, 0u, 0u, 0u);
        uint32_t s = 0;
#pragma unroll
        for (int q = 0; q < kScanPer / 4; ++q) s += v[q].x + v[q].y + v[q].z + v[q].w;
        // block exclusive scan of s
        uint32_t x = s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) wsum[warp] = x;
        __syncthreads();
        if (warp == 0) {
            uint32_t w = lane < kScanThreads / 32 ? wsum[lane] : 0u;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += y;
            }
            wsum[lane] = w;  // inclusive sums of the warps
            if (lane == kScanThreads / 32 - 1) carry_sh = w;
        }
        __syncthreads();
        uint32_t run = carry + (warp ? wsum[warp - 1] : 0u) + x - s;
        if (i0 < total) {
#pragma unroll
            for (int q = 0; q < kScanPer / 4; ++q) {
                uint4 o;
                o.x = run;
                run += v[q].x;
                o.y = run;
                run += v[q].y;
                o.z = run;
                run += v[q].z;
                o.w = run;
                run += v[q].w;
                reinterpret_cast<uint4*>(hist + i0)[q] = o;
            }
        }
        carry += carry_sh;
        __syncthreads();  // wsum and carry_sh are rewritten by the next tile
    }
}

template <typename OutI>
__global__ void __launch_bounds__(kSortThreads)
radix_scatter_kernel(const int32_t* __restrict__ ro, const uint32_t* __restrict__ keys_in,
                     const int32_t* __restrict__ vals_in, int32_t m, uint32_t key_base, int shift,
                     const uint32_t* __restrict__ offsets, uint32_t* __restrict__ keys_out,
                     OutI* __restrict__ vals_out) {
    __shared__ uint32_t warp_cnt[kSortThreads / 32][kRadix];
    __shared__ uint32_t running[kRadix];
    __shared__ uint32_t dbase[kRadix];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    running[tid] = 0;
    dbase[tid] = offsets[tid * gridDim.x + blockIdx.x];
    const uint32_t lt_mask = (1u << lane) - 1u;
    const int32_t base = blockIdx.x * kSortTile;
    for (int r = 0; r < kSortRounds; ++r) {
#pragma unroll
        for (int w = 0; w < kSortThreads / 32; ++w) warp_cnt[w][tid] = 0;
        __syncthreads();
        const int32_t i = base + r * kSortThreads + tid;
        const bool valid = i < m;
        uint32_t key = 0;
        int32_t val = 0;
        int d = kRadix + lane;  // unique per invalid lane: never matches a real digit
        if (valid) {
            key = sort_key(ro, keys_in, i, key_base);
            val = vals_in ? vals_in[i] : i;
            d = (int)((key >> shift) & (kRadix - 1));
        }
        const uint32_t peers = __match_any_sync(0xffffffffu, d);
        const uint32_t rank = __popc(peers & lt_mask);
        if (valid && lane == __ffs(peers) - 1) warp_cnt[warp][d] = __popc(peers);
        __syncthreads();
        {  // digit tid: exclusive prefix over warps, continuing from earlier rounds
            uint32_t acc = running[tid];
#pragma unroll
            for (int w = 0; w < kSortThreads / 32; ++w) {
                const uint32_t c = warp_cnt[w][tid];
                warp_cnt[w][tid] = acc;
                acc += c;
            }
            running[tid] = acc;
        }
        __syncthreads();
        if (valid) {
            const uint32_t pos = dbase[d] + warp_cnt[warp][d] + rank;
            if (keys_out) keys_out[pos] = key;
            vals_out[pos] = static_cast<OutI>(val);
        }
        __syncthreads();
    }
}

// Up to kRankSortRows rows: one CTA, a thread per row, sorts by rank. The key
// (0xFFFFFFFF - nnz_i) << 32 | i is distinct per row and orders rows by nnz descending, then by
// ascending row id, so each row's position is the number of keys below its own: one barrier
// and at most kRankSortRows broadcast shared-memory compares per thread, where the radix
// passes below cost several block-wide phases each.
constexpr int kRankSortRows = 1024;

template <typename OutI>
__global__ void __launch_bounds__(kRankSortRows) sort_rank_kernel(const int32_t* __restrict__ ro, int32_t m,
                                                                   OutI* __restrict__ out) {
    __shared__ unsigned long long key[kRankSortRows];
    const int i = threadIdx.x;
    pdl_trigger();
    pdl_wait();
    unsigned long long k = 0;
    if (i < m) {
        const uint32_t len = (uint32_t)(ro[i + 1] - ro[i]);
        k = ((unsigned long long)(0xFFFFFFFFu - len) << 32) | (uint32_t)i;
        key[i] = k;
    }
    __syncthreads();
    if (i < m) {
        int r = 0;
#pragma unroll 8
        for (int j = 0; j < m; ++j) r += key[j] < k ? 1 : 0;
        out[r] = static_cast<OutI>(i);
    }
}

// One CTA sorts up to kSmallSortRows rows in shared memory by a stable LSD radix sort of
// the key (longest row - nnz_i), with digits of up to kSmallBits bits and as many passes as
// the key range (longest - shortest row) needs: none when every row has the same length.
// Warp w owns the contiguous positions [w*L, (w+1)*L), L = ceil(m / 32). Per pass:
//   1. each warp counts its digits, 32 positions at a time (match_any gives each lane its
//      rank among equal digits in the group, the group leader adds the group's count);
//   2. one thread per digit turns the 32 warp counts into exclusive prefixes and a block
//      scan over digits gives each digit's first position;
//   3. each warp walks its positions again in the same order and scatters each row to
//      digit start + earlier warps' count + running count in the warp + rank in the group.
// Walking each warp's block in order and the warps in order keeps equal keys in input
// order (stability), so ties stay by ascending row id.
constexpr int kSmallSortRows = 16384;
constexpr int kSmallThreads = 1024;
constexpr int kSmallWarps = kSmallThreads / 32;
constexpr int kSmallBits = 9;
constexpr int kSmallBins = 1 << kSmallBits;
constexpr size_t kSmallSortSmem = kSmallSortRows * 4 + 2 * kSmallSortRows * 2 + kSmallWarps * kSmallBins * 4;

template <typename OutI>
__global__ void __launch_bounds__(kSmallThreads) sort_small_kernel(const int32_t* __restrict__ ro, int32_t m,
                                                                   OutI* __restrict__ out) {
    extern __shared__ __align__(16) unsigned char sm[];
    uint32_t* len = reinterpret_cast<uint32_t*>(sm);  // nnz of every row, by row id
    uint16_t* va = reinterpret_cast<uint16_t*>(len + kSmallSortRows);
    uint16_t* vb = va + kSmallSortRows;
    uint32_t(*wcnt)[kSmallBins] = reinterpret_cast<uint32_t(*)[kSmallBins]>(vb + kSmallSortRows);
    __shared__ int32_t red[2][kSmallWarps];
    __shared__ int32_t sh[32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t lt_mask = (1u << lane) - 1u;
    pdl_trigger();
    pdl_wait();

    int32_t mx = 0, mn = INT32_MAX;
    for (int32_t i = tid; i < m; i += kSmallThreads) {
        va[i] = (uint16_t)i;
        const int32_t c = ro[i + 1] - ro[i];
        len[i] = (uint32_t)c;
        mx = max(mx, c);
        mn = min(mn, c);
    }
    for (int o = 16; o; o >>= 1) {
        mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    }
    if (lane == 0) {
        red[0][warp] = mx;
        red[1][warp] = mn;
    }
    __syncthreads();
    mx = 0;
    mn = INT32_MAX;
    for (int w = 0; w < kSmallWarps; ++w) {
        mx = max(mx, red[0][w]);
        mn = min(mn, red[1][w]);
    }
    const uint32_t key_base = (uint32_t)mx;
    int bits = 0;
    while (bits < 32 && ((uint32_t)(mx - mn) >> bits) != 0) ++bits;
    const int32_t L = (m + kSmallWarps - 1) / kSmallWarps;
    const int32_t w0 = min(m, warp * L), w1 = min(m, w0 + L);
    for (int shift = 0; shift < bits; shift += kSmallBits) {
        const int db = min(kSmallBits, bits - shift);
        const uint32_t dmask = (1u << db) - 1u;
        const int nbins = 1 << db;
        auto digit = [&](uint32_t v) { return (int)(((key_base - len[v]) >> shift) & dmask); };
        for (int b = lane; b < nbins; b += 32) wcnt[warp][b] = 0;
        __syncwarp();
        // 1. counts per warp
        for (int32_t c0 = w0; c0 < w1; c0 += 32) {
            const int32_t i = c0 + lane;
            const bool valid = i < w1;
            const int d = valid ? digit(va[i]) : nbins + lane;  // invalid lanes never match a digit
            const uint32_t peers = __match_any_sync(0xffffffffu, d);
            if (valid && lane == __ffs(peers) - 1) wcnt[warp][d] += __popc(peers);
            __syncwarp();
        }
        __syncthreads();
        // 2. per digit: exclusive prefix over warps, then over digits
        int total = 0;
        if (tid < nbins) {
            for (int w = 0; w < kSmallWarps; ++w) {
                const uint32_t c = wcnt[w][tid];
                wcnt[w][tid] = (uint32_t)total;
                total += (int)c;
            }
        }
        {  // block exclusive scan of `total` over threads (digits)
            int x = total;
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += y;
            }
            if (lane == 31) sh[warp] = x;
            __syncthreads();
            if (warp == 0) {
                int y = sh[lane];
                for (int o = 1; o < 32; o <<= 1) {
                    const int z = __shfl_up_sync(0xffffffffu, y, o);
                    if (lane >= o) y += z;
                }
                sh[lane] = y;
            }
            __syncthreads();
            const int start = (warp ? sh[warp - 1] : 0) + x - total;
            if (tid < nbins)
                for (int w = 0; w < kSmallWarps; ++w) wcnt[w][tid] += (uint32_t)start;
        }
        __syncthreads();
        // 3. stable scatter
        for (int32_t c0 = w0; c0 < w1; c0 += 32) {
            const int32_t i = c0 + lane;
            const bool valid = i < w1;
            const uint16_t v = valid ? va[i] : 0;
            const int d = valid ? digit(v) : nbins + lane;
            const uint32_t peers = __match_any_sync(0xffffffffu, d);
            if (valid) vb[wcnt[warp][d] + __popc(peers & lt_mask)] = v;
            __syncwarp();
            if (valid && lane == __ffs(peers) - 1) wcnt[warp][d] += __popc(peers);
            __syncwarp();
        }
        __syncthreads();
        uint16_t* t = va;
        va = vb;
        vb = t;
    }
    for (int32_t i = tid; i < m; i += kSmallThreads) out[i] = static_cast<OutI>(va[i]);
}

template <typename OutI>
__global__ void iota_kernel(OutI* out, int32_t m) {
    for (int32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < m; i += gridDim.x * blockDim.x)
        out[i] = static_cast<OutI>(i);
}

__global__ void __launch_bounds__(1024) row_bins_kernel(const int32_t* __restrict__ ro, int32_t m, int32_t t_long,
                                                        int32_t* __restrict__ bins) {
    __shared__ int32_t red[2][32];
    int32_t nl = 0, ne = 0;
    for (int32_t i = threadIdx.x; i < m; i += blockDim.x) {
        const int32_t c = ro[i + 1] - ro[i];
        nl += c >= t_long;
        ne += c >= 1;
    }
    for (int off = 16; off; off >>= 1) {
        nl += __shfl_xor_sync(0xffffffffu, nl, off);
        ne += __shfl_xor_sync(0xffffffffu, ne, off);
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) {
        red[0][warp] = nl;
        red[1][warp] = ne;
    }
    __syncthreads();
    if (warp == 0) {
        nl = lane < (int)(blockDim.x >> 5) ? red[0][lane] : 0;
        ne = lane < (int)(blockDim.x >> 5) ? red[1][lane] : 0;
        for (int off = 16; off; off >>= 1) {
            nl += __shfl_xor_sync(0xffffffffu, nl, off);
            ne += __shfl_xor_sync(0xffffffffu, ne, off);
        }
        if (lane == 0) {
            bins[0] = 0;
            bins[1] = nl;
            bins[2] = ne;
            bins[3] = m;
        }
    }
}

// --------------------------------------------------------------- structure check

template <typename I>
__global__ void check_rows_kernel(const int32_t* __restrict__ ro, const I* __restrict__ col, int32_t m, int32_t n,
                                  int32_t nnz, int* err) {
    const int32_t stride = gridDim.x * blockDim.x;
    const int32_t tid = blockIdx.x * blockDim.x + threadIdx.x;
    if (tid == 0 && (ro[0] != 0 || ro[m] != nnz)) record_error(err, kDevErrRowOffsets);
    for (int32_t i = tid; i < m; i += stride) {
        const int32_t b = ro[i], e = ro[i + 1];
        if (b > e || b < 0 || e > nnz) {
            record_error(err, kDevErrRowOffsets);
            continue;
        }
        int prev = -1;
        for (int32_t k = b; k < e; ++k) {
            const int c = idx_of(col[k]);
            if (c < 0 || c >= n) record_error(err, kDevErrColRange);
            else if (c <= prev) record_error(err, kDevErrColOrder);
            prev = c;
        }
    }
}

__global__ void zero_words_kernel(uint32_t* p, int32_t words) {
    for (int32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < words; i += gridDim.x * blockDim.x) p[i] = 0;
}

template <typename I>
__global__ void check_perm_kernel(const I* __restrict__ row_idx, int32_t m, uint32_t* bits, int* err) {
    for (int32_t p = blockIdx.x * blockDim.x + threadIdx.x; p < m; p += gridDim.x * blockDim.x) {
        const int r = idx_of(row_idx[p]);
        if (r < 0 || r >= m) {
            record_error(err, kDevErrRowIdxPerm);
            continue;
        }
        const uint32_t bit = 1u << (r & 31);
        if (atomicOr(&bits[r >> 5], bit) & bit) record_error(err, kDevErrRowIdxPerm);
    }
}

int grid_for(int64_t items, int threads, int per_sm) {
    const int64_t g = (items + threads - 1) / threads;
    return (int)max64(1, min64(g, (int64_t)device_props().sm_count * per_sm));
}

}  // namespace

size_t sort_rows_workspace_bytes(int32_t m) {
    const size_t nb = (size_t)((m + kSortTile - 1) / kSortTile);
    const size_t arr = align_up((size_t)m * 4, 256);
    return 4 * arr + align_up(nb * kRadix * 4, 256);
}

cudaError_t launch_sort_rows(const int32_t* ro, int32_t m, int32_t nnz, void* row_idx_out, int it, void* ws,
                             cudaStream_t s) {
    if (m == 0) return cudaSuccess;
    if (m <= kRankSortRows) {
        cudaError_t e = it == kIdx16 ? launch_pdl(sort_rank_kernel<uint16_t>, 1, kRankSortRows, 0, s, ro, m,
                                                  (uint16_t*)row_idx_out)
                                     : launch_pdl(sort_rank_kernel<int32_t>, 1, kRankSortRows, 0, s, ro, m,
                                                  (int32_t*)row_idx_out);
        if (e != cudaSuccess) return e;
        count_launches(1);
        return cudaGetLastError();
    }
    if (m <= kSmallSortRows) {
        cudaError_t e = it == kIdx16
                            ? cudaFuncSetAttribute(sort_small_kernel<uint16_t>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmallSortSmem)
                            : cudaFuncSetAttribute(sort_small_kernel<int32_t>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmallSortSmem);
        if (e != cudaSuccess) return e;
        e = it == kIdx16 ? launch_pdl(sort_small_kernel<uint16_t>, 1, kSmallThreads, kSmallSortSmem, s, ro, m,
                                      (uint16_t*)row_idx_out)
                         : launch_pdl(sort_small_kernel<int32_t>, 1, kSmallThreads, kSmallSortSmem, s, ro, m,
                                      (int32_t*)row_idx_out);
        if (e != cudaSuccess) return e;
        count_launches(1);
        return cudaGetLastError();
    }
    int bits = 0;
    while (bits < 32 && ((uint64_t)nnz >> bits) != 0) ++bits;  // keys lie in [0, nnz]
    const int passes = (bits + 7) / 8;
    if (passes == 0) {
        if (it == kIdx16) iota_kernel<uint16_t><<<grid_for(m, 256, 4), 256, 0, s>>>((uint16_t*)row_idx_out, m);
        else iota_kernel<int32_t><<<grid_for(m, 256, 4), 256, 0, s>>>((int32_t*)row_idx_out, m);
        count_launches(1);
        return cudaGetLastError();
    }
    const int nb = (m + kSortTile - 1) / kSortTile;
    const size_t arr = align_up((size_t)m * 4, 256);
    char* w = static_cast<char*>(ws);
    uint32_t* keys[2] = {reinterpret_cast<uint32_t*>(w), reinterpret_cast<uint32_t*>(w + arr)};
    int32_t* vals[2] = {reinterpret_cast<int32_t*>(w + 2 * arr), reinterpret_cast<int32_t*>(w + 3 * arr)};
    uint32_t* hist = reinterpret_cast<uint32_t*>(w + 4 * arr);
    const uint32_t key_base = (uint32_t)nnz;
    for (int p = 0; p < passes; ++p) {
        const uint32_t* kin = p == 0 ? nullptr : keys[(p - 1) & 1];
        const int32_t* vin = p == 0 ? nullptr : vals[(p - 1) & 1];
        const bool last = p == passes - 1;
        radix_hist_kernel<<<nb, kSortThreads, 0, s>>>(ro, kin, m, key_base, 8 * p, hist);
        radix_scan_kernel<<<1, kScanThreads, 0, s>>>(hist, nb * kRadix);
        if (!last) {
            radix_scatter_kernel<int32_t><<<nb, kSortThreads, 0, s>>>(ro, kin, vin, m, key_base, 8 * p, hist,
                                                                       keys[p & 1], vals[p & 1]);
        } else if (it == kIdx16) {
            radix_scatter_kernel<uint16_t><<<nb, kSortThreads, 0, s>>>(ro, kin, vin, m, key_base, 8 * p, hist,
                                                                        nullptr, (uint16_t*)row_idx_out);
        } else {
            radix_scatter_kernel<int32_t><<<nb, kSortThreads, 0, s>>>(ro, kin, vin, m, key_base, 8 * p, hist,
                                                                       nullptr, (int32_t*)row_idx_out);
        }
    }
    count_launches(3 * passes);
    return cudaGetLastError();
}

cudaError_t launch_row_bins(const int32_t* ro, int32_t m, int32_t t_long, int32_t* bins, cudaStream_t s) {
    row_bins_kernel<<<1, 1024, 0, s>>>(ro, m, t_long, bins);
    count_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_check_csr(const int32_t* ro, const void* col, const void* row_idx, int it, int32_t m, int32_t n,
                             int32_t nnz, uint32_t* perm_bits, int* err, cudaStream_t s) {
    const int g = grid_for(m > 0 ? m : 1, 256, 8);
    if (it == kIdx16) check_rows_kernel<uint16_t><<<g, 256, 0, s>>>(ro, (const uint16_t*)col, m, n, nnz, err);
    else check_rows_kernel<int32_t><<<g, 256, 0, s>>>(ro, (const int32_t*)col, m, n, nnz, err);
    if (row_idx && perm_bits && m > 0) {
        const int32_t words = (m + 31) / 32;
        zero_words_kernel<<<grid_for(words, 256, 4), 256, 0, s>>>(perm_bits, words);
        if (it == kIdx16) check_perm_kernel<uint16_t><<<g, 256, 0, s>>>((const uint16_t*)row_idx, m, perm_bits, err);
        else check_perm_kernel<int32_t><<<g, 256, 0, s>>>((const int32_t*)row_idx, m, perm_bits, err);
        count_launches(2);
    }
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace spops
