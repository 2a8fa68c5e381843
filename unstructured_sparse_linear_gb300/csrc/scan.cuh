// Exclusive prefix sums of large uint32 counter arrays (radix-sort digit histograms) in two
// parallel steps instead of one serial block:
//   1. chunk_scan_kernel: every 1024-thread CTA scans kScanChunk consecutive counters in
//      place (coalesced 16-byte loads, a block scan) and writes the chunk's total;
//   2. chunk_sums_kernel: one CTA scans the chunk totals in place.
// The exclusive prefix of counter i is then counter[i] + sums[i / kScanChunk]; consumers add
// the second term when they read the first, so no third pass is needed.
#pragma once

#include <stdint.h>

namespace spops {
namespace {  // each including file gets its own copy of the kernels

constexpr int kScanThreads1k = 1024;
constexpr int kScanPer = 4;                                  // counters per thread
constexpr int kScanChunk = kScanThreads1k * kScanPer;        // counters per CTA

// Exclusive scan of one value per thread over a 1024-thread block; *total gets the sum.
__device__ __forceinline__ uint32_t block_scan_1k(uint32_t v, uint32_t* sh, uint32_t* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t x = v;
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sh[warp] = x;
    __syncthreads();
    if (warp == 0) {
        uint32_t w = sh[lane];
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        sh[lane] = w;
    }
    __syncthreads();
    const uint32_t before = (warp ? sh[warp - 1] : 0u) + x - v;
    *total = sh[31];
    __syncthreads();
    return before;
}

// counters: 16-byte aligned, `total` entries.
__global__ void __launch_bounds__(kScanThreads1k) chunk_scan_kernel(uint32_t* __restrict__ counters, int64_t total,
                                                                    uint32_t* __restrict__ sums) {
    __shared__ uint32_t sh[32];
    const int64_t base = (int64_t)blockIdx.x * kScanChunk + (int64_t)threadIdx.x * kScanPer;
    uint32_t c[kScanPer];
    if (base + kScanPer <= total) {
        const uint4 q = *reinterpret_cast<const uint4*>(counters + base);
        c[0] = q.x;
        c[1] = q.y;
        c[2] = q.z;
        c[3] = q.w;
    } else {
#pragma unroll
        for (int e = 0; e < kScanPer; ++e) c[e] = base + e < total ? counters[base + e] : 0u;
    }
    uint32_t s = 0;
#pragma unroll
    for (int e = 0; e < kScanPer; ++e) s += c[e];
    uint32_t tot;
    uint32_t run = block_scan_1k(s, sh, &tot);
#pragma unroll
    for (int e = 0; e < kScanPer; ++e) {
        if (base + e < total) counters[base + e] = run;
        run += c[e];
    }
    if (threadIdx.x == 0) sums[blockIdx.x] = tot;
}

// In-place exclusive scan of n chunk totals with one CTA.
__global__ void __launch_bounds__(kScanThreads1k) chunk_sums_kernel(uint32_t* __restrict__ sums, int32_t n) {
    __shared__ uint32_t sh[32];
    uint32_t carry = 0;
    for (int32_t b = 0; b < n; b += kScanThreads1k) {
        const int32_t i = b + threadIdx.x;
        const uint32_t v = i < n ? sums[i] : 0u;
        uint32_t tot;
        const uint32_t ex = block_scan_1k(v, sh, &tot);
        if (i < n) sums[i] = carry + ex;
        carry += tot;
    }
}

inline int64_t scan_chunks(int64_t total) { return (total + kScanChunk - 1) / kScanChunk; }

}  // namespace
}  // namespace spops
