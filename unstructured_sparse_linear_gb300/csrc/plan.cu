// Mask plan: row bins and the dense-panel decomposition, from row_offsets / row_idx /
// col_idx alone.
//
// spops README ("Sparse Operations (spops)"): row_idx sorts rows by their number of
// non-zeros ("Usage"), and the structure-aware SDDMM exploits masks whose non-zeros
// cluster in few rows and columns ("Sampled Dense-Dense Matrix Multiplication"). The plan
// turns both into work lists:
//   * row bins per operator (long rows get a CTA each, short rows a lane group);
//   * panels = 128 consecutive row_idx positions. For each panel the union U of its
//     columns; a panel is dense when |U| <= 1024, it has at least 16 non-empty rows and its
//     entries fill at least a quarter of (non-empty rows) x |U|. Dense panels run on the
//     tensor cores as 128 x |U| tiles.
// Two kernels (after zeroing P + 1 completion counters), none with a serial per-thread loop
// over a panel:
//   1. row groups (8 rows per CTA): row ids per position, per-group counts, and a column
//      bitmap per 8-row group built with shared-memory atomics; then
//   2. the last group of a panel to finish: OR the group bitmaps, prefix-sum their
//      popcounts, list U, decide density (for SDDMM tiles |U| <= 1024, for a SpMM image
//      |U| <= 2048); then
//   3. the last panel to finish: sum the group counts into row bins, list dense panels and
//      SDDMM tiles, and assign SpMM image slots within the image budget (in panel order);
//   4. second kernel, row groups of dense panels: each entry's position in U and, per row,
//      the first entry of every 128-column tile of U and a bit mask of the U positions it
//      holds.
// Every count is an integer sum in a fixed order, so the plan is bit-identical on every
// build.
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

__device__ void panel_work(const PlanView& v, int p, uint32_t* sm);
__device__ void lists_work(const PlanView& v, int64_t img_budget);

// ---- 1. row groups
template <typename I>
__global__ void __launch_bounds__(kPlanThreads)
plan_rows_kernel(const int32_t* __restrict__ ro, const I* __restrict__ row_idx, const I* __restrict__ col,
                 PlanView v, int64_t img_budget) {
    extern __shared__ uint32_t bitmap[];  // 2 W words when panels are enabled (the panel step reuses them)
    __shared__ int red[4][8];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    pdl_trigger();
    pdl_wait();
    const int64_t p0 = (int64_t)blockIdx.x * kGroupRows;
    if (v.panels)
        for (int w = tid; w < v.W; w += kPlanThreads) bitmap[w] = 0;
    __syncthreads();
    int c_spmm = 0, c_sddmm = 0, c_ne = 0, c_ent = 0;
    for (int rr = 0; rr < kGroupRows / 8; ++rr) {
        const int64_t pos = p0 + warp * (kGroupRows / 8) + rr;
        int row = -1;
        if (pos < v.m) row = idx_of(row_idx[pos]);
        if (lane == 0 && v.panels) v.prow[pos] = row;  // pos < P * 128 always
        if (row < 0) continue;
        const int32_t k0 = ro[row], k1 = ro[row + 1];
        const int32_t c = k1 - k0;
        if (lane == 0) {
            c_spmm += c >= kSpmmLongRow;
            c_sddmm += c >= kSddmmLongRow;
            c_ne += c >= 1;
            c_ent += c;
        }
        if (v.panels) {
            for (int32_t k = k0 + lane; k < k1; k += 32) {
                const int cc = idx_of(col[k]);
                atomicOr(&bitmap[cc >> 5], 1u << (cc & 31));
            }
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
        int s = 0;
        for (int w = 0; w < 8; ++w) s += red[tid][w];
        v.cta_part[blockIdx.x * 4 + tid] = s;
    }
    if (v.panels) {
        uint32_t* dst = v.bm_part + (size_t)blockIdx.x * v.W;  // group g of panel p is CTA p*kGroups+g
        for (int w = tid; w < v.W; w += kPlanThreads) dst[w] = bitmap[w];
    }
    // The last row group of a panel to finish builds the panel; the last panel to finish
    // builds the bins and work lists. Each CTA publishes its writes (fence) before it counts
    // itself in; the one that completes a count fences again before reading the others'.
    __shared__ int s_last;
    const int p = blockIdx.x / kGroups;
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = atomicAdd(&v.done[p], 1) == kGroups - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    if (v.panels) panel_work(v, p, bitmap);
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = atomicAdd(&v.done[v.P], 1) == v.P - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    lists_work(v, img_budget);
}

// ---- 2. panel p (run by the last of its row-group CTAs to finish)
__device__ void panel_work(const PlanView& v, int p, uint32_t* sm) {
    uint32_t* bm = sm;  // bm[W], wbase[W]
    int* wb = reinterpret_cast<int*>(sm + v.W);
    __shared__ int sh[32];
    __shared__ int s_cnt[2];
    const int tid = threadIdx.x;
    for (int w = tid; w < v.W; w += kPlanThreads) {
        uint32_t x = 0;
#pragma unroll
        for (int g = 0; g < kGroups; ++g) x |= v.bm_part[((size_t)p * kGroups + g) * v.W + w];
        bm[w] = x;
    }
    if (tid < 2) {
        int s = 0;
        for (int g = 0; g < kGroups; ++g) {
            const int cta = p * kGroups + g;
            if (cta < v.ncta) s += v.cta_part[cta * 4 + (tid == 0 ? 3 : 2)];
        }
        s_cnt[tid] = s;  // [0] entries, [1] non-empty rows
    }
    __syncthreads();
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
    const int nnz_p = s_cnt[0], ne = s_cnt[1];
    const bool filled = nnz_p > 0 && ne >= kMinDenseRows && (int64_t)nnz_p * 4 >= (int64_t)ne * U;
    const bool dense = filled && U <= kUCap;     // SDDMM tiles
    const bool dense_sp = filled && U <= kUList; // SpMM image
    if (tid == 0) {
        v.desc[p] = make_int4((dense ? 1 : 0) | (dense_sp ? 2 : 0), U, nnz_p, ne);
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

// ---- 3. bins and work lists (run by the last panel to finish)
__device__ void lists_work(const PlanView& v, int64_t img_budget) {
    __shared__ int sh[32];
    // row bins: fixed-order sums over the group CTAs
    int a = 0, b = 0, c = 0;
    for (int i = threadIdx.x; i < v.ncta; i += blockDim.x) {
        a += v.cta_part[i * 4 + 0];
        b += v.cta_part[i * 4 + 1];
        c += v.cta_part[i * 4 + 2];
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
    int cd = 0, ct = 0, cs = 0, cn = 0;
    int64_t ci = 0;
    for (int base = 0; base < v.P; base += blockDim.x) {
        const int p = base + threadIdx.x;
        const int4 d = p < v.P ? v.desc[p] : make_int4(0, 0, 0, 0);
        const int dn = d.x & 1;          // SDDMM tiles
        const int dsp = (d.x >> 1) & 1;  // SpMM image candidate
        const int tiles = dn ? (d.y + kTileN - 1) / kTileN : 0;
        const int img = dsp ? kPM * ((d.y + 63) / 64) * 64 : 0;
        int td, tt, ti, tn;
        const int ed = block_exclusive_scan(dn, sh, &td);
        const int et = block_exclusive_scan(tiles, sh, &tt);
        const int ei = block_exclusive_scan(img, sh, &ti);
        const int en = block_exclusive_scan(dn ? d.z : 0, sh, &tn);
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
        }
        cd += td;
        ct += tt;
        cs += tf;
        cn += tn;
        ci += ti;
    }
    if (threadIdx.x == 0) {
        int32_t* cnt = v.counts();
        cnt[kCntDense] = cd;
        cnt[kCntTiles] = ct;
        cnt[kCntDenseSp] = cs;
        cnt[kCntDenseNnz] = cn;
        cnt[kCntImgElems] = (int32_t)min64(ci, img_budget);
        cnt[kCntPanels] = v.P;
        cnt[6] = 0;
        cnt[7] = 0;
    }
}

// ---- 4. entry positions in U, tile starts and per-row column masks (dense panels only)
template <typename I>
__global__ void __launch_bounds__(kPlanThreads)
plan_upos_kernel(const int32_t* __restrict__ ro, const I* __restrict__ col, PlanView v) {
    extern __shared__ uint32_t sm[];
    constexpr int kMaskWords = kUCap / 32;
    static_assert(kMaskWords == 32, "one mask word per lane");
    __shared__ uint32_t rmask[8][kMaskWords];  // one row per warp
    pdl_trigger();
    pdl_wait();
    const int p = blockIdx.x / kGroups;
    if (!(v.desc[p].x & 2)) return;  // U positions for SpMM-dense panels
    const bool tiles = v.dense[p];    // tile starts and masks for SDDMM-dense ones (U <= kUCap)
    uint32_t* bm = sm;
    int* wb = reinterpret_cast<int*>(sm + v.W);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int w = tid; w < v.W; w += kPlanThreads) {
        bm[w] = v.bm[(size_t)p * v.W + w];
        wb[w] = v.wbase[(size_t)p * v.W + w];
    }
    __syncthreads();
    auto upos_of = [&](int c) { return wb[c >> 5] + __popc(bm[c >> 5] & ((1u << (c & 31)) - 1u)); };
    const int64_t p0 = (int64_t)blockIdx.x * kGroupRows;
    for (int rr = 0; rr < kGroupRows / 8; ++rr) {
        const int64_t pos = p0 + warp * (kGroupRows / 8) + rr;
        const int row = v.prow[pos];
        int32_t* ts = v.ts + pos * (kTiles + 1);
        uint32_t* tm = v.tmask + pos * kMaskWords;
        rmask[warp][lane] = 0;  // kMaskWords == 32: one word per lane
        __syncwarp();
        if (row < 0) {
            if (tiles) {
                if (lane <= kTiles) ts[lane] = 0;
                tm[lane] = 0;
            }
            continue;
        }
        const int32_t k0 = ro[row], k1 = ro[row + 1];
        if (k0 == k1) {
            if (tiles) {
                if (lane <= kTiles) ts[lane] = k0;
                tm[lane] = 0;
            }
            continue;
        }
        for (int32_t k = k0 + lane; k < k1; k += 32) {
            const int u = upos_of(idx_of(col[k]));
            v.upos[k] = (uint16_t)u;
            if (!tiles) continue;
            atomicOr(&rmask[warp][u >> 5], 1u << (u & 31));
            const int t_cur = u / kTileN;
            const int t_prev = k > k0 ? upos_of(idx_of(col[k - 1])) / kTileN : -1;
            for (int t = t_prev + 1; t <= t_cur; ++t) ts[t] = k;  // tiles starting at entry k
            if (k == k1 - 1)
                for (int t = t_cur + 1; t <= kTiles; ++t) ts[t] = k1;
        }
        __syncwarp();
        if (tiles) tm[lane] = rmask[warp][lane];
    }
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
    // one row-group CTA per 16 positions of every panel, including the positions past m in
    // the last panel (they record row -1), so every panel position gets a row id
    const size_t nc = (size_t)((m + kPM - 1) / kPM) * kGroups;
    L.hdr = take(32 * 4);
    L.cta_part = take(nc * 16);
    L.done = take((size_t)((m + kPM - 1) / kPM + 1) * 4);
    if (plan_panels_enabled(m, n)) {
        const size_t P = (size_t)(m + kPM - 1) / kPM;
        const size_t W = (size_t)(n + 31) / 32;
        L.bm_part = take(P * kGroups * W * 4);
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
        L.dlist_sp = take(P * 4);
        L.img_slot = take(P * 4);
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
    v.ncta = v.P * kGroups;
    v.hdr = at<int32_t>(b, L.hdr);
    v.cta_part = at<int32_t>(b, L.cta_part);
    v.done = at<int32_t>(b, L.done);
    if (v.panels) {
        v.bm_part = at<uint32_t>(b, L.bm_part);
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
        v.dlist_sp = at<int32_t>(b, L.dlist_sp);
        v.img_slot = at<int32_t>(b, L.img_slot);
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

cudaError_t launch_plan_build(int it, const int32_t* ro, const void* row_idx, const void* col, const PlanView& v,
                              int64_t img_budget, cudaStream_t s) {
    if (v.m <= 0) return cudaSuccess;
    const size_t smem_rows = v.panels ? (size_t)v.W * 8 : 0;
    const size_t smem_pan = (size_t)v.W * 8;
    if (smem_pan > 48 * 1024) {
        cudaError_t e = it == kIdx16 ? cudaFuncSetAttribute(plan_rows_kernel<uint16_t>,
                                                            cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_rows)
                                     : cudaFuncSetAttribute(plan_rows_kernel<int32_t>,
                                                            cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_rows);
        if (e != cudaSuccess) return e;
        e = it == kIdx16 ? cudaFuncSetAttribute(plan_upos_kernel<uint16_t>,
                                                cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_pan)
                         : cudaFuncSetAttribute(plan_upos_kernel<int32_t>,
                                                cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_pan);
        if (e != cudaSuccess) return e;
    }
    cudaError_t e = cudaMemsetAsync(v.done, 0, (size_t)(v.P + 1) * sizeof(int32_t), s);
    if (e != cudaSuccess) return e;
    e = it == kIdx16 ? launch_pdl(plan_rows_kernel<uint16_t>, v.ncta, kPlanThreads, smem_rows, s, ro,
                                  (const uint16_t*)row_idx, (const uint16_t*)col, v, img_budget)
                     : launch_pdl(plan_rows_kernel<int32_t>, v.ncta, kPlanThreads, smem_rows, s, ro,
                                  (const int32_t*)row_idx, (const int32_t*)col, v, img_budget);
    if (e != cudaSuccess) return e;
    int launches = 1;
    if (v.panels) {
        e = it == kIdx16 ? launch_pdl(plan_upos_kernel<uint16_t>, v.P * kGroups, kPlanThreads, smem_pan, s, ro,
                                      (const uint16_t*)col, v)
                         : launch_pdl(plan_upos_kernel<int32_t>, v.P * kGroups, kPlanThreads, smem_pan, s, ro,
                                      (const int32_t*)col, v);
        if (e != cudaSuccess) return e;
        ++launches;
    }
    count_launches(launches);
    return cudaGetLastError();
}

cudaError_t launch_plan_stats(const PlanView& v, int32_t* out, cudaStream_t s) {
    plan_stats_kernel<<<1, 32, 0, s>>>(v, out);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace spops
