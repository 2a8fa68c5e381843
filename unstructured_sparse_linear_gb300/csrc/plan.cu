// Mask plan: row bins and the dense-panel decomposition, from row_offsets / row_idx /
// col_idx alone.
//
// spops README ("Sparse Operations (spops)"): row_idx sorts rows by their number of
// non-zeros ("Usage"), and the structure-aware SDDMM exploits masks whose non-zeros
// cluster in few rows and columns ("Sampled Dense-Dense Matrix Multiplication"). The plan
// turns both into work lists:
//   * row bins per operator (long rows get a CTA each, short rows a lane group);
//   * panels = 128 consecutive positions of the plan's row order (row_idx, reordered for
//     masks of at most 16384 rows so that rows with one column pattern share panels when a
//     pattern recurs in separate runs; kernels 0a and 0b below). For each panel the union U
//     of its columns; a panel is dense when it has at least 16 non-empty rows and its
//     entries fill at least a quarter of (non-empty rows) x |U|. Dense panels run on the
//     tensor cores as 128 x |U| tiles (SDDMM when |U| <= 1024, SpMM when |U| <= 4096).
// After the order, two kernels; no counters to reset between builds:
//   1. a thread-block cluster of 8 CTAs per panel, 16 positions per CTA: row ids per
//      position, counts, and a column bitmap per CTA built with shared-memory atomics; after
//      a cluster barrier, rank 0 ORs the 8 bitmaps through distributed shared memory,
//      prefix-sums their popcounts, lists U and decides density (SDDMM tiles |U| <= 1024,
//      SpMM image |U| <= 4096) and whether the panel's CSR values are already in image
//      order (rows of one length |U| in two runs of 64 consecutive rows);
//   2. row groups of dense panels (8 rows per CTA): each entry's position in U and, per row,
//      the first entry of every 128-column tile of U and a bit mask of the U positions it
//      holds (not for panels whose rows each hold all of U in order: their consumers derive
//      all three from the row id and |U|); one extra CTA sums the panel counts into row
//      bins, lists dense panels and SDDMM tiles, and assigns SpMM image slots within the
//      image budget (in panel order).
// Index loads are batched (8 per lane) before their results are used, so a long row costs a
// few dependent load latencies, not one per 32 entries. Every count is an integer sum in a
// fixed order, so the plan is bit-identical on every build.
#include "common.cuh"
#include "plan.h"

namespace spops {
namespace {

constexpr int kPlanThreads = 256;

template <typename T>
T* at(char* b, size_t off) {
    return reinterpret_cast<T*>(b + off);
}

// Block-wide exclusive scan of one int per thread (blockDim.x a multiple of 32, <= 1024).
__device__ __forceinline__ int block_exclusive_scan(int v, int* sh, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int x = v;
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sh[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = lane < nw ? sh[lane] : 0;
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        sh[lane] = w;
    }
    __syncthreads();
    const int before = (warp ? sh[warp - 1] : 0) + x - v;
    *total = sh[nw - 1];
    __syncthreads();
    return before;
}

// Set bits x[j] (x >= 0; -1: nothing) of the shared bitmap bm, called by all 32 lanes with
// NB slices of entries. Lanes hold the entries of a row in U order, so lanes whose bits
// fall in one word form runs; a segmented OR over the run (shuffles at distance 1, 2, 4, 8,
// 16, taken while the lane at that distance has the same word) gathers the run's bits in its
// first lane, which does the one atomic. A lane at distance d with the same word but outside
// the run adds bits of that same word, which is harmless. The NB scans advance step by step
// together, so their shuffle latencies overlap.
template <int NB>
__device__ __forceinline__ void or_bits_aggregated(uint32_t* bm, const int (&x)[NB], int lane) {
    int w[NB];
    uint32_t bits[NB];
#pragma unroll
    for (int j = 0; j < NB; ++j) {
        w[j] = x[j] >= 0 ? x[j] >> 5 : -1;
        bits[j] = x[j] >= 0 ? 1u << (x[j] & 31) : 0u;
    }
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        uint32_t ob[NB];
        int ow[NB];
#pragma unroll
        for (int j = 0; j < NB; ++j) {
            ob[j] = __shfl_down_sync(0xffffffffu, bits[j], d);
            ow[j] = __shfl_down_sync(0xffffffffu, w[j], d);
        }
#pragma unroll
        for (int j = 0; j < NB; ++j)
            if (lane + d < 32 && ow[j] == w[j]) bits[j] |= ob[j];
    }
#pragma unroll
    for (int j = 0; j < NB; ++j) {
        const int pw = __shfl_up_sync(0xffffffffu, w[j], 1);
        if (w[j] >= 0 && (lane == 0 || pw != w[j])) atomicOr(&bm[w[j]], bits[j]);
    }
}

// Set bit x (x >= 0; -1: nothing) of the shared bitmap bm, called by all 32 lanes. When every
// lane's bit falls in one word (a 32-column slice of one row of a block-structured mask) the
// warp ORs them together and one lane does the atomic; otherwise every lane does its own
// (sparse rows rarely collide, and the hardware handles a few lanes on one word well).
__device__ __forceinline__ void or_bit_warp(uint32_t* bm, int x, int lane) {
    const int w = x >= 0 ? x >> 5 : -1;
    const uint32_t bit = x >= 0 ? 1u << (x & 31) : 0u;
    const int w0 = __shfl_sync(0xffffffffu, w, 0);
    if (__all_sync(0xffffffffu, w == w0 && w0 >= 0)) {
        const uint32_t b = __reduce_or_sync(0xffffffffu, bit);
        if (lane == 0) atomicOr(&bm[w0], b);
    } else if (x >= 0) {
        atomicOr(&bm[w], bit);
    }
}

// ---- 0. row order (masks of at most kOrderMaxRows rows): row_idx refined so that rows with
// the same column set become neighbours. Rows of a block-structured mask that share their
// blocks then fill the same panel, whose U is exactly their columns (the butterfly layer's
// 64-row block-rows r, r + 32, ... share four blocks). The positions of row_idx are sorted
// stably by (nnz descending, signature); the signature is a 16-bit hash of the row's first,
// middle and last column: rows with the same column set always agree on it, and rows that
// agree on it with different sets only share a panel (its U covers both), so no result
// depends on it. The sort runs only where it can merge panels: when two runs of row_idx
// (maximal stretches of positions whose non-empty rows have one key) of at least
// kOrdLongRun positions each have the same key, i.e. a column pattern recurs in separate
// places (the butterfly's block-rows r and r + 32). A random mask has no such runs; a
// clustered one keeps its repeated rows in one run already. Otherwise prow = row_idx and the
// panels are as without an order. Two kernels:
//   a. keys, one thread per position over the whole GPU (these are the gathers: the row's
//      offsets and three of its columns): prow = row_idx (-1 past m), the key of each
//      position, and per block of 32 positions the key of the long run that starts in it (or
//      none), so that the second kernel tests for a repeated key before loading anything;
//   b. one CTA: the repeated-key test; then coalesced loads of rows and keys into shared
//      memory and the runs, stably sorted by key with a bitonic network over (key, run)
//      pairs (at most 1024 runs), else a stable LSD radix sort of the positions with 8-bit
//      digits, skipping digits that are the same in every key.
constexpr int kKeyThreads = 256;
constexpr int kOrdThreads = 1024;
constexpr int kOrdWarps = kOrdThreads / 32;
constexpr int kOrdBins = 256;
constexpr int kOrdLongRun = 32;
constexpr int kOrdHash = 2 * kOrderMaxRows / kOrdLongRun;  // slots for the keys of the long runs
constexpr uint32_t kNoKey = 0xFFFFFFFFu;                    // no non-empty row has this key
constexpr size_t kOrdSmem = (size_t)kOrderMaxRows * 4      // keys, by row
                            + (size_t)kOrderMaxRows * 2 * 2  // rows, two buffers
                            + (size_t)kOrdWarps * kOrdBins * 4;  // digit counts, or the runs
static_assert((size_t)kOrdWarps * kOrdBins * 4 >= kOrdThreads * 8 + (2 * kOrdThreads + 2) * 4,
              "the run arrays fit in the digit counts");
static_assert(kOrderMaxRows / 32 <= kOrdThreads, "one word of break flags per thread");
static_assert(kOrderMaxRows % kOrdThreads == 0, "positions per thread");

__device__ __forceinline__ uint32_t mix_col(uint32_t c) {
    uint32_t h = c * 0x9E3779B1u;
    h ^= h >> 15;
    h *= 0x85EBCA77u;
    h ^= h >> 13;
    return h;
}

// 16-bit signature of a row from its first, middle and last column (an empty row: 0)
__device__ __forceinline__ uint32_t row_signature(uint32_t first, uint32_t mid, uint32_t last) {
    const uint32_t h = mix_col(first) + mix_col(mid ^ 0x55555555u) + mix_col(last ^ 0xAAAAAAAAu);
    return (h >> 16) ^ (h & 0xFFFFu);
}

// Sort key of a row with len entries: nnz descending (complemented, rows of 65535 entries or
// more tie), then the signature.
__device__ __forceinline__ uint32_t order_key(int32_t len, uint32_t sig) {
    return ((uint32_t)(0xFFFF - min(len, 0xFFFF)) << 16) | sig;
}

template <typename I>
__global__ void __launch_bounds__(kKeyThreads)
plan_keys_kernel(const int32_t* __restrict__ ro, const I* __restrict__ row_idx, const I* __restrict__ col,
                 PlanView v) {
    // keys of positions base - 1 .. base + kKeyThreads + kOrdLongRun - 1 (the run checks of
    // this CTA's positions read up to kOrdLongRun - 1 positions past its end)
    __shared__ uint32_t s_key[kKeyThreads + kOrdLongRun + 1];
    __shared__ uint32_t s_brk[kKeyThreads / 32 + 1];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int base = blockIdx.x * kKeyThreads;
    const int m = v.m;
    pdl_trigger();
    pdl_wait();
    // this thread's position p0, and for threads 0 .. kOrdLongRun a halo position p1 (past the
    // end, or base - 1); both keys are gathered together
    const int p0 = base + tid;
    const int p1 = tid < kOrdLongRun ? base + kKeyThreads + tid : (tid == kOrdLongRun ? base - 1 : -1);
    const int r0 = p0 < m ? idx_of(row_idx[p0]) : -1;
    const int r1 = p1 >= 0 && p1 < m ? idx_of(row_idx[p1]) : -1;
    const int32_t a0 = r0 >= 0 ? ro[r0] : 0, a1 = r1 >= 0 ? ro[r1] : 0;
    const int32_t l0 = r0 >= 0 ? ro[r0 + 1] - a0 : 0, l1 = r1 >= 0 ? ro[r1 + 1] - a1 : 0;
    uint32_t c[6] = {0, 0, 0, 0, 0, 0};
    if (l0 > 0) {
        c[0] = (uint32_t)idx_of(col[a0]);
        c[1] = (uint32_t)idx_of(col[a0 + l0 / 2]);
        c[2] = (uint32_t)idx_of(col[a0 + l0 - 1]);
    }
    if (l1 > 0) {
        c[3] = (uint32_t)idx_of(col[a1]);
        c[4] = (uint32_t)idx_of(col[a1 + l1 / 2]);
        c[5] = (uint32_t)idx_of(col[a1 + l1 - 1]);
    }
    const uint32_t k0 = r0 >= 0 ? order_key(l0, l0 > 0 ? row_signature(c[0], c[1], c[2]) : 0u) : kNoKey;
    const uint32_t k1 = r1 >= 0 ? order_key(l1, l1 > 0 ? row_signature(c[3], c[4], c[5]) : 0u) : kNoKey;
    if (p0 < v.P * kPM) v.prow[p0] = r0;
    if (p0 < m) v.okey[p0] = k0;
    s_key[1 + tid] = k0;
    if (tid < kOrdLongRun) s_key[1 + kKeyThreads + tid] = k1;
    if (tid == kOrdLongRun) s_key[0] = k1;
    __syncthreads();
    // breaks (a position whose key differs from the one before) at base + j, j < 256 + 32
    {
        const int j = tid;
        const bool b = base + j < m && (base + j == 0 || s_key[1 + j] != s_key[j]);
        const uint32_t word = __ballot_sync(0xffffffffu, b);
        if (lane == 0) s_brk[warp] = word;
        if (warp == 0) {
            const int jh = kKeyThreads + lane;
            const bool bh = base + jh < m && s_key[1 + jh] != s_key[jh];
            const uint32_t wh = __ballot_sync(0xffffffffu, bh);
            if (lane == 0) s_brk[kKeyThreads / 32] = wh;
        }
    }
    __syncthreads();
    // a long run of a non-empty key starts at p0: a break with no break in the next 31
    // positions; two such starts are 32 apart, so a block of 32 positions holds one at most
    static_assert(kOrdLongRun == 32, "one 32-bit window of break flags, one long run per 32 positions");
    uint32_t win = s_brk[warp] >> lane;
    if (lane) win |= s_brk[warp + 1] << (32 - lane);
    const bool lng = win == 1u && p0 + kOrdLongRun <= m && (k0 >> 16) != 0xFFFFu;
    const uint32_t lb = __ballot_sync(0xffffffffu, lng);
    const int blk = blockIdx.x * (kKeyThreads / 32) + warp;
    if (lane == 0 && blk < v.P * kPM / 32) {
        v.olong[blk] = lb ? s_key[1 + warp * 32 + __ffs(lb) - 1] : kNoKey;
        v.obrk[blk] = s_brk[warp];
    }
}

__global__ void __launch_bounds__(kOrdThreads, 1) plan_sort_kernel(PlanView v) {
    extern __shared__ __align__(16) uint8_t osm[];
    uint32_t* key = reinterpret_cast<uint32_t*>(osm);  // by row
    uint16_t* va = reinterpret_cast<uint16_t*>(key + kOrderMaxRows);
    uint16_t* vb = va + kOrderMaxRows;
    uint32_t(*wcnt)[kOrdBins] = reinterpret_cast<uint32_t(*)[kOrdBins]>(vb + kOrderMaxRows);
    __shared__ uint32_t s_var[kOrdWarps];
    __shared__ uint32_t brk[kOrderMaxRows / 32];
    __shared__ int wpre[kOrderMaxRows / 32];  // runs starting before each word of brk
    __shared__ uint32_t s_hash[kOrdHash];
    __shared__ int sh[32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int m = v.m;
    pdl_trigger();
    pdl_wait();
    // a repeated key among the long runs (at most one per 32 positions, so at most m / 32
    // keys in 2 m / 32 hash slots)
    for (int i = tid; i < kOrdHash; i += kOrdThreads) s_hash[i] = kNoKey;
    __syncthreads();
    int dup = 0;
    for (int b = tid; b < (m + 31) / 32; b += kOrdThreads) {
        const uint32_t k = v.olong[b];
        if (k == kNoKey) continue;
        uint32_t h = mix_col(k) & (kOrdHash - 1);
        for (int t = 0; t < kOrdHash; ++t) {
            const uint32_t old = atomicCAS(&s_hash[h], kNoKey, k);
            if (old == kNoKey) break;
            if (old == k) {
                dup = 1;
                break;
            }
            h = (h + 1) & (kOrdHash - 1);
        }
    }
    if (!__syncthreads_or(dup)) return;  // prow already holds row_idx
    // rows and keys (all of a thread's loads issued before any is used); the bits in which
    // some key differs from the first
    constexpr int kPer = kOrderMaxRows / kOrdThreads;
    const uint32_t k0 = v.okey[0];
    uint32_t var = 0;
    int rq[kPer];
    uint32_t kq[kPer];
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
        const int p = tid + q * kOrdThreads;
        rq[q] = p < m ? v.prow[p] : -1;
        kq[q] = p < m ? v.okey[p] : k0;
    }
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
        if (rq[q] < 0) continue;
        key[rq[q]] = kq[q];
        va[tid + q * kOrdThreads] = (uint16_t)rq[q];
        var |= kq[q] ^ k0;
    }
    // run breaks, from the keys kernel: bit p of brk is set when position p starts a
    // stretch of one key (p = 0 or its key differs from position p - 1)
    for (int w = tid; w < (m + 31) / 32; w += kOrdThreads) brk[w] = v.obrk[w];
    for (int o = 16; o; o >>= 1) var |= __shfl_xor_sync(0xffffffffu, var, o);
    if (lane == 0) s_var[warp] = var;
    __syncthreads();  // keys, rows and breaks are in place
    var = 0;
    for (int w = 0; w < kOrdWarps; ++w) var |= s_var[w];
    if (var == 0) return;  // one key: the order is row_idx
    __syncthreads();
    // The stretches of one key (runs) in row_idx order: a stable sort of the positions by key
    // keeps each run together and in place relative to the other runs of its key, so it is
    // the runs, stably sorted by key, laid end to end. With at most kOrdThreads runs they are
    // sorted as (key, run index) pairs by one bitonic network; more runs take the radix sort
    // of the positions below.
    const int nwords = (m + 31) / 32;
    int total_runs;
    {
        const int c = tid < nwords ? __popc(brk[tid]) : 0;
        const int before = block_exclusive_scan(c, sh, &total_runs);
        if (tid < nwords) wpre[tid] = before;
    }
    if (total_runs <= kOrdThreads) {
        const int R = total_runs;
        unsigned long long* sk = reinterpret_cast<unsigned long long*>(&wcnt[0][0]);  // [kOrdThreads]
        int32_t* rs = reinterpret_cast<int32_t*>(sk + kOrdThreads);                  // run starts
        int32_t* os = rs + kOrdThreads + 1;                                           // run destinations
        __syncthreads();  // wpre is complete
        if (tid < nwords) {
            uint32_t bits = brk[tid];
            int i = wpre[tid];
            while (bits) {
                const int p = tid * 32 + __ffs(bits) - 1;
                rs[i] = p;
                sk[i] = ((unsigned long long)key[va[p]] << 32) | (unsigned)i;
                ++i;
                bits &= bits - 1;
            }
        }
        if (tid >= R) sk[tid] = ~0ull;
        if (tid == 0) rs[R] = m;
        __syncthreads();
        // bitonic network over NP = the power of two >= max(R, 32) elements, one per thread
        // of the first NP / 32 warps: partners less than 32 apart exchange by shuffles, the
        // others through shared memory behind a named barrier of those warps
        int NP = 32;
        while (NP < R) NP <<= 1;
        if (tid < NP) {
            unsigned long long x = sk[tid];
            for (int kk = 2; kk <= NP; kk <<= 1) {
                for (int j = kk >> 1; j > 0; j >>= 1) {
                    unsigned long long y;
                    if (j >= 32) {
                        named_barrier(1, NP);  // the previous round's reads are done
                        sk[tid] = x;
                        named_barrier(1, NP);
                        y = sk[tid ^ j];
                    } else {
                        y = __shfl_xor_sync(0xffffffffu, x, j);
                    }
                    const bool up = (tid & kk) == 0, low = (tid & j) == 0;
                    x = (up == low) ? (x < y ? x : y) : (x < y ? y : x);
                }
            }
            named_barrier(1, NP);
            sk[tid] = x;
        }
        __syncthreads();
        // destinations: lengths summed in sorted order
        const int ri = tid < R ? (int)(unsigned)sk[tid] : 0;
        const int len = tid < R ? rs[ri + 1] - rs[ri] : 0;
        int tot;
        const int dst0 = block_exclusive_scan(len, sh, &tot);
        if (tid < R) os[ri] = dst0;
        __syncthreads();
#pragma unroll
        for (int q = 0; q < kPer; ++q) {
            const int p = tid + q * kOrdThreads;
            if (p >= m) break;
            const int w = p >> 5;
            const int i = wpre[w] + __popc(brk[w] & (0xFFFFFFFFu >> (31 - (p & 31)))) - 1;  // run of p
            v.prow[os[i] + (p - rs[i])] = va[p];
        }
        return;
    }
    // warp w owns positions [w L, (w + 1) L)
    const int L = (m + kOrdWarps - 1) / kOrdWarps;
    const int w0 = min(m, warp * L), w1 = min(m, w0 + L);
    const uint32_t lt_mask = (1u << lane) - 1u;
    uint16_t* src = va;
    uint16_t* dst = vb;
    for (int shift = 0; shift < 32; shift += 8) {
        if (((var >> shift) & (kOrdBins - 1)) == 0) continue;  // the same digit in every key
        auto digit = [&](uint16_t rr) { return (int)((key[rr] >> shift) & (kOrdBins - 1)); };
        for (int bn = lane; bn < kOrdBins; bn += 32) wcnt[warp][bn] = 0;
        __syncwarp();
        for (int c = w0; c < w1; c += 32) {
            const int i = c + lane;
            const bool valid = i < w1;
            const int d = valid ? digit(src[i]) : kOrdBins + lane;
            const uint32_t peers = __match_any_sync(0xffffffffu, d);
            if (valid && lane == __ffs(peers) - 1) wcnt[warp][d] += __popc(peers);
            __syncwarp();
        }
        __syncthreads();
        // digit tid (< 256): exclusive prefix over warps, then a scan over the digits
        int total = 0;
        if (tid < kOrdBins) {
            uint32_t acc = 0;
            for (int w = 0; w < kOrdWarps; ++w) {
                const uint32_t cn = wcnt[w][tid];
                wcnt[w][tid] = acc;
                acc += cn;
            }
            total = (int)acc;
        }
        int x = total;
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) sh[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int ws = lane < kOrdBins / 32 ? sh[lane] : 0;
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, ws, o);
                if (lane >= o) ws += y;
            }
            sh[lane] = ws;
        }
        __syncthreads();
        if (tid < kOrdBins) {
            const uint32_t before = (uint32_t)((warp ? sh[warp - 1] : 0) + x - total);
            for (int w = 0; w < kOrdWarps; ++w) wcnt[w][tid] += before;
        }
        __syncthreads();
        // stable scatter, each warp walking its positions in order
        for (int c = w0; c < w1; c += 32) {
            const int i = c + lane;
            const bool valid = i < w1;
            const uint16_t rr = valid ? src[i] : 0;
            const int d = valid ? digit(rr) : kOrdBins + lane;
            const uint32_t peers = __match_any_sync(0xffffffffu, d);
            const uint32_t rk = __popc(peers & lt_mask);
            if (valid) dst[wcnt[warp][d] + rk] = rr;
            __syncwarp();
            if (valid && lane == __ffs(peers) - 1) wcnt[warp][d] += __popc(peers);
            __syncwarp();
        }
        __syncthreads();
        uint16_t* t = src;
        src = dst;
        dst = t;
    }
    for (int p = tid; p < m; p += kOrdThreads) v.prow[p] = src[p];
}

constexpr int kRowsPerWarp = kCtaRows / (kPlanThreads / 32);  // positions per warp in the row step
constexpr int kLoadBatch = 8;                                  // index loads per lane in flight

__device__ void panel_work(const PlanView& v, const int32_t* __restrict__ ro, int p, uint32_t* sm, int nnz_p, int ne);

// ---- 1. row step: cluster of kPlanCluster CTAs per panel
template <typename I>
__global__ void __launch_bounds__(kPlanThreads)
plan_rows_kernel(const int32_t* __restrict__ ro, const I* __restrict__ row_idx, const I* __restrict__ col,
                 PlanView v, int ordered) {
    extern __shared__ uint32_t bitmap[];  // W words (2 W in rank 0, whose panel step reuses them)
    __shared__ int red[4][kPlanThreads / 32];
    __shared__ int s_cnt[4], s_tot[4];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int p = blockIdx.x / kPlanCluster;
    const int rank = (int)cluster_rank();
    pdl_trigger();
    if (v.panels)
        for (int w = tid; w < v.W; w += kPlanThreads) bitmap[w] = 0;
    pdl_wait();
    // the warp's positions: their rows, then the rows' offsets, each batch loaded together
    const int64_t pos0 = (int64_t)p * kPM + rank * kCtaRows + warp * kRowsPerWarp;
    int row[kRowsPerWarp];
    int32_t k0[kRowsPerWarp], len[kRowsPerWarp];
#pragma unroll
    for (int q = 0; q < kRowsPerWarp; ++q)
        row[q] = ordered ? v.prow[pos0 + q] : (pos0 + q < v.m ? idx_of(row_idx[pos0 + q]) : -1);
#pragma unroll
    for (int q = 0; q < kRowsPerWarp; ++q) {
        k0[q] = row[q] >= 0 ? ro[row[q]] : 0;
        len[q] = row[q] >= 0 ? ro[row[q] + 1] - k0[q] : 0;
    }
    int c_spmm = 0, c_sddmm = 0, c_ne = 0, c_ent = 0, total = 0;
#pragma unroll
    for (int q = 0; q < kRowsPerWarp; ++q) {
        if (v.panels && !ordered && lane == q) v.prow[pos0 + q] = row[q];  // pos0 + q < P * 128 always
        c_spmm += len[q] >= kSpmmLongRow;
        c_sddmm += len[q] >= kSddmmLongRow;
        c_ne += len[q] >= 1;
        c_ent += len[q];
        total += len[q];
    }
    if (v.panels) {
        static_assert(kRowsPerWarp == 2, "entry t of the warp's rows is in row 0 below len[0], else row 1");
        for (int t0 = 0; t0 < total; t0 += 32 * kLoadBatch) {
            int cc[kLoadBatch];
#pragma unroll
            for (int j = 0; j < kLoadBatch; ++j) {
                const int t = t0 + j * 32 + lane;
                const int32_t k = t < len[0] ? k0[0] + t : k0[1] + (t - len[0]);
                cc[j] = t < total ? idx_of(col[k]) : -1;
            }
#pragma unroll
            for (int j = 0; j < kLoadBatch; ++j) or_bit_warp(bitmap, cc[j], lane);
        }
    }
    if (lane == 0) {
        red[0][warp] = c_spmm;
        red[1][warp] = c_sddmm;
        red[2][warp] = c_ne;
        red[3][warp] = c_ent;
    }
    __syncthreads();
    if (tid < 4) {
        int x = 0;
#pragma unroll
        for (int w = 0; w < kPlanThreads / 32; ++w) x += red[tid][w];
        s_cnt[tid] = x;
    }
    cluster_sync();  // every CTA's bitmap and counts are final and visible to rank 0
    if (rank == 0) {
        if (v.panels)
            for (int w = tid; w < v.W; w += kPlanThreads) {
                const uint32_t a = smem_u32(&bitmap[w]);
                uint32_t x = bitmap[w];
#pragma unroll
                for (int r = 1; r < kPlanCluster; ++r) x |= ld_cluster_u32(cluster_map(a, r));
                bitmap[w] = x;
            }
        if (tid < 4) {
            int x = 0;
            for (int r = 0; r < kPlanCluster; ++r) x += (int)ld_cluster_u32(cluster_map(smem_u32(&s_cnt[tid]), r));
            v.pan_part[p * 4 + tid] = x;
            s_tot[tid] = x;
        }
    }
    cluster_sync();  // the other CTAs keep their shared memory until rank 0 has read it
    if (rank != 0 || !v.panels) return;
    panel_work(v, ro, p, bitmap, s_tot[3], s_tot[2]);
}

// ---- panel p (rank 0 of its cluster; sm holds the panel's OR-ed bitmap, W more words free)
__device__ void panel_work(const PlanView& v, const int32_t* __restrict__ ro, int p, uint32_t* sm, int nnz_p,
                           int ne) {
    uint32_t* bm = sm;  // bm[W], wbase[W]
    int* wb = reinterpret_cast<int*>(sm + v.W);
    __shared__ int sh[32];
    const int tid = threadIdx.x;
    const int per = (v.W + kPlanThreads - 1) / kPlanThreads;
    const int b = tid * per, e = min(v.W, b + per);
    int s = 0;
    for (int w = b; w < e; ++w) s += __popc(bm[w]);
    int U;
    int run = block_exclusive_scan(s, sh, &U);
    for (int w = b; w < e; ++w) {
        wb[w] = run;
        run += __popc(bm[w]);
    }
    __syncthreads();
    const bool filled = nnz_p > 0 && ne >= kMinDenseRows && (int64_t)nnz_p * 4 >= (int64_t)ne * U;
    const bool dense = filled && U <= kUCap;     // SDDMM tiles
    const bool dense_sp = filled && U <= kUList; // SpMM image
    // Values already in image order: every row of the mask has the same length L = nnz / m,
    // this panel's 128 rows are two runs of 64 consecutive rows and each of them holds all of
    // U (L == |U|). Then the panel's values are a 128 x |U| block of the m x L matrix the CSR
    // values form, in column order, and the SpMM pipeline can load its A chunks from them
    // directly instead of from a densified image.
    bool direct = false;
    if (dense_sp && v.m > 0 && v.nnz % v.m == 0 && (int64_t)v.nnz / v.m == U) {
        const int64_t L = (int64_t)v.nnz / v.m;
        bool ok = true;
        if (tid < kPM) {
            const int r = v.prow[(int64_t)p * kPM + tid];
            const int first = v.prow[(int64_t)p * kPM + (tid & ~63)];
            ok = r >= 0 && first >= 0 && r == first + (tid & 63) && (int64_t)ro[r] == (int64_t)r * L &&
                 (int64_t)ro[r + 1] == (int64_t)(r + 1) * L;
        }
        direct = __syncthreads_and(ok) != 0;
    }
    if (tid == 0) {
        v.desc[p] = make_int4((dense ? 1 : 0) | (dense_sp ? 2 : 0) | (direct ? 4 : 0), U, nnz_p, ne);
        v.dense[p] = dense ? 1 : 0;
    }
    if (!dense_sp) return;
    for (int w = tid; w < v.W; w += kPlanThreads) {
        v.bm[(size_t)p * v.W + w] = bm[w];
        v.wbase[(size_t)p * v.W + w] = wb[w];
        uint32_t bits = bm[w];
        int at = wb[w];
        while (bits) {
            const int bit = __ffs(bits) - 1;
            v.ulist[(size_t)p * kUList + at++] = w * 32 + bit;
            bits &= bits - 1;
        }
    }
}

// ---- bins and work lists (one CTA, after the row step)
__device__ void lists_work(const PlanView& v, int64_t img_budget) {
    __shared__ int sh[32];
    // row bins: fixed-order sums over the panels
    int a = 0, b = 0, c = 0;
    for (int i = threadIdx.x; i < v.P; i += blockDim.x) {
        a += v.pan_part[i * 4 + 0];
        b += v.pan_part[i * 4 + 1];
        c += v.pan_part[i * 4 + 2];
    }
    int ta, tb, tc;
    block_exclusive_scan(a, sh, &ta);
    block_exclusive_scan(b, sh, &tb);
    block_exclusive_scan(c, sh, &tc);
    if (threadIdx.x == 0) {
        int32_t* bs = v.bins_spmm();
        int32_t* bd = v.bins_sddmm();
        bs[0] = 0; bs[1] = ta; bs[2] = tc; bs[3] = v.m;
        bd[0] = 0; bd[1] = tb; bd[2] = tc; bd[3] = v.m;
    }
    if (!v.panels) {
        if (threadIdx.x < 8) v.counts()[threadIdx.x] = threadIdx.x == kCntPanels ? v.P : 0;
        return;
    }
    int cd = 0, ct = 0, cs = 0, cn = 0, cg = 0;
    int64_t ci = 0;
    for (int base = 0; base < v.P; base += blockDim.x) {
        const int p = base + threadIdx.x;
        const int4 d = p < v.P ? v.desc[p] : make_int4(0, 0, 0, 0);
        const int dn = d.x & 1;          // SDDMM tiles
        const int dsp = (d.x >> 1) & 1;  // SpMM image candidate
        const int tiles = dn ? (d.y + kTileN - 1) / kTileN : 0;
        const int groups = (tiles + kGroupTiles - 1) / kGroupTiles;
        const int img = dsp ? kPM * ((d.y + 63) / 64) * 64 : 0;
        int td, tt, ti, tn;
        const int ed = block_exclusive_scan(dn, sh, &td);
        const int et = block_exclusive_scan(tiles, sh, &tt);
        const int ei = block_exclusive_scan(img, sh, &ti);
        const int en = block_exclusive_scan(dn ? d.z : 0, sh, &tn);
        int tgr;
        const int egr = block_exclusive_scan(groups, sh, &tgr);
        (void)ed;
        (void)en;
        // image slots in panel order while they fit the budget
        const bool fits = dsp && ci + ei + img <= img_budget;
        int tf;
        const int ef = block_exclusive_scan(fits ? 1 : 0, sh, &tf);
        if (p < v.P) {
            v.img_slot[p] = fits ? (int)(ci + ei) : -1;
            v.sp_dense[p] = fits ? 1 : 0;
            if (fits) v.dlist_sp[cs + ef] = p;
            for (int j = 0; j < tiles; ++j) v.items[ct + et + j] = (p << 8) | j;
            for (int j = 0; j < groups; ++j) v.gitems[cg + egr + j] = (p << 8) | j;
        }
        cd += td;
        ct += tt;
        cs += tf;
        cn += tn;
        ci += ti;
        cg += tgr;
    }
    if (threadIdx.x == 0) {
        int32_t* cnt = v.counts();
        cnt[kCntDense] = cd;
        cnt[kCntTiles] = ct;
        cnt[kCntDenseSp] = cs;
        cnt[kCntDenseNnz] = cn;
        cnt[kCntImgElems] = (int32_t)min64(ci, img_budget);
        cnt[kCntPanels] = v.P;
        cnt[kCntGroups] = cg;
        cnt[7] = 0;
    }
}

// ---- 2. entry positions in U, tile starts and per-row column masks (dense panels), and
// the lists (the grid's last CTA)
template <typename I>
__global__ void __launch_bounds__(kPlanThreads)
plan_upos_kernel(const int32_t* __restrict__ ro, const I* __restrict__ col, PlanView v, int64_t img_budget) {
    extern __shared__ uint32_t sm[];
    constexpr int kMaskWords = kUCap / 32;
    static_assert(kMaskWords == 32, "one mask word per lane");
    static_assert(kGroupRows == kPlanThreads / 32, "one row per warp");
    __shared__ uint32_t rmask[kGroupRows][kMaskWords];
    pdl_trigger();
    pdl_wait();
    if (blockIdx.x == gridDim.x - 1) {
        lists_work(v, img_budget);
        return;
    }
    const int p = blockIdx.x / kGroups;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t pos = (int64_t)blockIdx.x * kGroupRows + warp;
    // the panel's dense bits and the warp's row are independent loads: issued together
    const int dbits = v.desc[p].x;
    const int row = v.prow[pos];
    // U positions for SpMM-dense panels, except the direct ones (bit 4: every row holds all
    // of U in order), whose consumers derive them from the row id and |U|
    if ((dbits & 6) != 2) return;
    const bool tiles = (dbits & 1) != 0;  // tile starts and masks for SDDMM-dense ones (U <= kUCap)
    uint32_t* bm = sm;
    int* wb = reinterpret_cast<int*>(sm + v.W);
    const int32_t k0 = row >= 0 ? ro[row] : 0, k1 = row >= 0 ? ro[row + 1] : 0;
    for (int w = tid; w < v.W; w += kPlanThreads) {
        bm[w] = v.bm[(size_t)p * v.W + w];
        wb[w] = v.wbase[(size_t)p * v.W + w];
    }
    rmask[warp][lane] = 0;
    __syncthreads();
    auto upos_of = [&](int c) { return wb[c >> 5] + __popc(bm[c >> 5] & ((1u << (c & 31)) - 1u)); };
    int32_t* ts = v.ts + pos * (kTiles + 1);
    uint32_t* tm = v.tmask + pos * kMaskWords;
    if (k0 == k1) {  // empty row or a position past m
        if (tiles) {
            if (lane <= kTiles) ts[lane] = k0;
            tm[lane] = 0;
        }
        return;
    }
    int carry = -1;  // U position of the entry before this batch (-1: none)
    for (int32_t kb = k0; kb < k1; kb += 32 * kLoadBatch) {
        int u[kLoadBatch];
#pragma unroll
        for (int j = 0; j < kLoadBatch; ++j) {
            const int32_t k = kb + j * 32 + lane;
            u[j] = k < k1 ? idx_of(col[k]) : 0;
        }
#pragma unroll
        for (int j = 0; j < kLoadBatch; ++j) u[j] = upos_of(u[j]);
#pragma unroll
        for (int j = 0; j < kLoadBatch; ++j) {
            const int32_t k = kb + j * 32 + lane;
            // U position of entry k - 1: the lane below, lane 31 of the slice before, or the carry
            const int up = __shfl_up_sync(0xffffffffu, u[j], 1);
            const int last_prev = __shfl_sync(0xffffffffu, j > 0 ? u[j > 0 ? j - 1 : 0] : carry, 31);
            const int u_prev = lane > 0 ? up : (j > 0 ? last_prev : carry);
            if (k >= k1) continue;
            v.upos[k] = (uint16_t)u[j];
            if (!tiles) continue;

            const int t_cur = u[j] / kTileN;
            const int t_prev = k > k0 ? u_prev / kTileN : -1;
            for (int t = t_prev + 1; t <= t_cur; ++t) ts[t] = k;  // tiles starting at entry k
            if (k == k1 - 1)
                for (int t = t_cur + 1; t <= kTiles; ++t) ts[t] = k1;
        }
        if (tiles) {
            int um[kLoadBatch];
#pragma unroll
            for (int j = 0; j < kLoadBatch; ++j) um[j] = kb + j * 32 + lane < k1 ? u[j] : -1;
            or_bits_aggregated<kLoadBatch>(rmask[warp], um, lane);  // U positions of a row are dense
        }
        carry = __shfl_sync(0xffffffffu, u[kLoadBatch - 1], 31);
    }
    __syncwarp();
    if (tiles) tm[lane] = rmask[warp][lane];
}

__global__ void plan_stats_kernel(PlanView v, int32_t* out) {
    if (threadIdx.x < 8) out[threadIdx.x] = v.counts()[threadIdx.x];
    if (threadIdx.x >= 8 && threadIdx.x < 16) out[threadIdx.x] = v.hdr[threadIdx.x - 8];  // bins
}

}  // namespace

bool plan_panels_enabled(int32_t m, int32_t n) { return m > 0 && n > 0 && n <= kMaxPanelCols; }

PlanLayout plan_layout(int32_t m, int32_t n, int32_t nnz) {
    PlanLayout L{};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t a = off;
        off = align_up(off + bytes, 1024);
        return a;
    };
    const size_t P = (size_t)(m + kPM - 1) / kPM;
    L.hdr = take(32 * 4);
    L.pan_part = take(P * 16);
    if (plan_panels_enabled(m, n)) {
        const size_t W = (size_t)(n + 31) / 32;
        L.bm = take(P * W * 4);
        L.wbase = take(P * W * 4);
        L.desc = take(P * 16);
        L.prow = take(P * kPM * 4);
        L.ulist = take(P * kUList * 4);
        L.upos = take((size_t)nnz * 2);
        L.ts = take(P * kPM * (kTiles + 1) * 4);
        L.tmask = take(P * kPM * (kUCap / 32) * 4);
        L.dense = take(P);
        L.sp_dense = take(P);
        L.items = take(P * kTiles * 4);
        L.gitems = take(P * (kTiles / kGroupTiles) * 4);
        L.dlist_sp = take(P * 4);
        L.img_slot = take(P * 4);
        if (m <= kOrderMaxRows) {
            L.okey = take(P * kPM * 4);
            L.olong = take(P * kPM / 32 * 4);
            L.obrk = take(P * kPM / 32 * 4);
        }
    }
    L.total = off;
    return L;
}

PlanView plan_view(void* base, int32_t m, int32_t n, int32_t nnz) {
    const PlanLayout L = plan_layout(m, n, nnz);
    char* b = static_cast<char*>(base);
    PlanView v{};
    v.m = m;
    v.n = n;
    v.nnz = nnz;
    v.panels = plan_panels_enabled(m, n);
    v.P = (m + kPM - 1) / kPM;
    v.W = v.panels ? (n + 31) / 32 : 0;
    v.hdr = at<int32_t>(b, L.hdr);
    v.pan_part = at<int32_t>(b, L.pan_part);
    if (v.panels) {
        v.bm = at<uint32_t>(b, L.bm);
        v.wbase = at<int32_t>(b, L.wbase);
        v.desc = at<int4>(b, L.desc);
        v.prow = at<int32_t>(b, L.prow);
        v.ulist = at<int32_t>(b, L.ulist);
        v.upos = at<uint16_t>(b, L.upos);
        v.ts = at<int32_t>(b, L.ts);
        v.tmask = at<uint32_t>(b, L.tmask);
        v.dense = at<uint8_t>(b, L.dense);
        v.sp_dense = at<uint8_t>(b, L.sp_dense);
        v.items = at<int32_t>(b, L.items);
        v.gitems = at<int32_t>(b, L.gitems);
        v.dlist_sp = at<int32_t>(b, L.dlist_sp);
        v.img_slot = at<int32_t>(b, L.img_slot);
        if (m <= kOrderMaxRows) {
            v.okey = at<uint32_t>(b, L.okey);
            v.olong = at<uint32_t>(b, L.olong);
            v.obrk = at<uint32_t>(b, L.obrk);
        }
    }
    return v;
}

size_t spmm_image_budget_elems(int32_t m, int32_t nnz) {
    // Dense panels satisfy entries >= |U| * rows / 4 with rows >= 16, so an image of
    // 128 x |U| elements needs at most 32 elements per entry; budget 8 per entry plus one
    // 128 x 64 chunk of padding per panel and give the rest to the general kernels.
    const size_t P = (size_t)(m + kPM - 1) / kPM;
    return (size_t)8 * nnz + P * kPM * 64;
}

// The order kernels. The keys kernel is launched stream-ordered (not as a programmatic
// dependent): it reads row_idx, row_offsets and col_idx, which the caller's previous
// operations on s (sort_rows, a transpose) have just written; the sort follows it as a
// programmatic dependent.
template <typename I>
cudaError_t launch_order(const int32_t* ro, const void* row_idx, const void* col, const PlanView& v, cudaStream_t s) {
    const unsigned grid = (unsigned)(((int64_t)v.P * kPM + kKeyThreads - 1) / kKeyThreads);
    plan_keys_kernel<I><<<grid, kKeyThreads, 0, s>>>(ro, static_cast<const I*>(row_idx), static_cast<const I*>(col),
                                                      v);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(plan_sort_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kOrdSmem);
    if (e != cudaSuccess) return e;
    return launch_pdl(plan_sort_kernel, 1, kOrdThreads, kOrdSmem, s, v);
}

cudaError_t launch_plan_build(int it, const int32_t* ro, const void* row_idx, const void* col, const PlanView& v,
                              int64_t img_budget, cudaStream_t s) {
    if (v.m <= 0) return cudaSuccess;
    // both kernels: the panel bitmap and its word prefix (2 W words) when panels are enabled
    const size_t smem = v.panels ? (size_t)v.W * 8 : 0;
    if (smem > 48 * 1024) {
        cudaError_t e = it == kIdx16 ? cudaFuncSetAttribute(plan_rows_kernel<uint16_t>,
                                                            cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)
                                     : cudaFuncSetAttribute(plan_rows_kernel<int32_t>,
                                                            cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        e = it == kIdx16 ? cudaFuncSetAttribute(plan_upos_kernel<uint16_t>,
                                                cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)
                         : cudaFuncSetAttribute(plan_upos_kernel<int32_t>,
                                                cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    // the column-pattern row order (panels, at most kOrderMaxRows rows)
    int ordered = 0;
    int nlaunch = 2;
    if (v.panels && v.m <= kOrderMaxRows) {
        cudaError_t e = it == kIdx16 ? launch_order<uint16_t>(ro, row_idx, col, v, s)
                                     : launch_order<int32_t>(ro, row_idx, col, v, s);
        if (e != cudaSuccess) return e;
        ordered = 1;
        nlaunch = 4;
    }
    const unsigned rows_grid = (unsigned)v.P * kPlanCluster;
    cudaError_t e = it == kIdx16
                        ? launch_pdl_cluster(plan_rows_kernel<uint16_t>, rows_grid, kPlanThreads, smem, kPlanCluster, s,
                                             ro, (const uint16_t*)row_idx, (const uint16_t*)col, v, ordered)
                        : launch_pdl_cluster(plan_rows_kernel<int32_t>, rows_grid, kPlanThreads, smem, kPlanCluster, s,
                                             ro, (const int32_t*)row_idx, (const int32_t*)col, v, ordered);
    if (e != cudaSuccess) return e;
    // U positions for every row group of every panel (only dense panels do work), plus the
    // lists CTA
    const unsigned upos_grid = (v.panels ? (unsigned)v.P * kGroups : 0u) + 1u;
    e = it == kIdx16 ? launch_pdl(plan_upos_kernel<uint16_t>, upos_grid, kPlanThreads, smem, s, ro,
                                  (const uint16_t*)col, v, img_budget)
                     : launch_pdl(plan_upos_kernel<int32_t>, upos_grid, kPlanThreads, smem, s, ro,
                                  (const int32_t*)col, v, img_budget);
    if (e != cudaSuccess) return e;
    count_launches(nlaunch);
    return cudaGetLastError();
}

cudaError_t launch_plan_stats(const PlanView& v, int32_t* out, cudaStream_t s) {
    plan_stats_kernel<<<1, 32, 0, s>>>(v, out);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace spops
