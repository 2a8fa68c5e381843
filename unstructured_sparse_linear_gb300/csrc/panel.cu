// Structure-aware path: dense panels of the CSR matrix on the tcgen05 tensor cores.
//
// spops README ("Sparse Operations (spops)"), section "Sampled Dense-Dense Matrix
// Multiplication (SDDMM)": besides the general kernel, SDDMM has a structure-aware kernel
// for the masks seen in RoSA, whose non-zeros cluster in a small subset of rows and
// columns. This file is that idea written for GB300:
//
// Plan (per call, from row_offsets / row_idx / col_idx only):
//   * panels: consecutive groups of 128 positions of row_idx (128 = UMMA M). Because
//     row_idx sorts rows by nnz, the clustered rows of a RoSA mask fill the first panels.
//   * for each panel, the union U of its columns (bitmap + popcount scan), the compact
//     position of every entry in U (upos), and a dense flag: |U| <= 1024 and the entries
//     fill at least a quarter of the 128 x |U| tile the tensor cores would compute.
//   * a work list of dense panels (and 128-column tiles of U for SDDMM).
// Execution:
//   * SDDMM: D = A[panel rows, :] * BT[U, :]^T per (panel, U tile, K split) on tcgen05
//     (fp16/bf16 in, fp32 accumulate in TMEM); the epilogue samples D at the panel's entries.
//     K is split across CTAs when there are fewer tiles than SMs; the fp32 partial sums are
//     added in split order by a finalize kernel, so results are deterministic.
//   * SpMM: the panel's values are scattered into a dense 128 x |U| image (already in the
//     UMMA 128-byte-swizzled K-major layout), and C[panel rows, N tile] = image * B[U, N tile]
//     on tcgen05, with B's rows gathered straight into an MN-major swizzled tile.
//   * rows of non-dense panels run through the general row kernels, which skip dense ones.
// Operands are gathered row by row with 16-byte cp.async copies into a 4-stage shared
// memory ring; one thread issues the MMAs and commits them to per-stage mbarriers, whose
// completion frees the stage for the next copy. Every mbarrier wait is bounded in time.
#include <type_traits>

#include "common.cuh"
#include "internal.h"
#include "panel.h"
#include "tc.cuh"

namespace spops {
namespace {

constexpr int kPM = 128;         // rows per panel (UMMA M)
constexpr int kUCap = 1024;      // most distinct columns a dense panel may have
constexpr int kKC = 64;          // K elements per pipeline chunk (128 bytes of 16-bit data)
constexpr int kStages = 4;
constexpr int kSdNT = 128;       // SDDMM: columns of U per tile (UMMA N)
constexpr int kSpNT = 256;       // SpMM: columns of C per tile (UMMA N)
constexpr int kMaxWords = 2048;  // column bitmap words: n <= 65536
constexpr int kMaxSplit = 16;
constexpr int kTileThreads = 128;
constexpr size_t kPartialBudget = 64ull << 20;  // bytes of fp32 split-K partial sums

constexpr uint32_t kSdStageBytes = 2 * kPM * kKC * 2;                  // A + BT tiles: 32 KB
constexpr uint32_t kSpStageA = kPM * kKC * 2;                          // 16 KB
constexpr uint32_t kSpStageB = kSpNT * kKC * 2;                        // 32 KB
constexpr uint32_t kSpStageBytes = kSpStageA + kSpStageB;              // 48 KB
constexpr uint32_t kSdSmem = kStages * kSdStageBytes + 1024;
constexpr uint32_t kSpSmem = kStages * kSpStageBytes + 1024;

struct PanelWs {
    int4* desc;        // [P] {dense, |U|, nnz of the panel, image offset in elements}
    int32_t* prow;     // [P * 128] row id at each panel position, -1 past m
    int32_t* ulist;    // [P * kUCap] sorted columns of U (dense panels)
    uint16_t* upos;    // [nnz] position of each entry's column in its panel's U
    uint8_t* dense;    // [P] dense flag
    int32_t* counts;   // [4] {#dense panels, #SDDMM tiles, image elements, 0}
    int32_t* dlist;    // [P] dense panel ids
    int32_t* items;    // [P * kUCap / kSdNT] (panel << 8) | tile
    float* partial;    // [max_split * nnz] SDDMM split-K partial sums
    void* img;         // SpMM dense images
};

struct Layout {
    size_t desc, prow, ulist, upos, dense, counts, dlist, items, partial, img, total;
};

Layout layout(int32_t m, int32_t nnz, bool sddmm, int max_split, bool spmm) {
    const size_t P = (size_t)(m + kPM - 1) / kPM;
    Layout L{};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = align_up(off + bytes, 1024);
        return at;
    };
    L.desc = take(P * 16);
    L.prow = take(P * kPM * 4);
    L.ulist = take(P * kUCap * 4);
    L.upos = take((size_t)nnz * 2);
    L.dense = take(P);
    L.counts = take(16);
    L.dlist = take(P * 4);
    L.items = take(P * (kUCap / kSdNT) * 4);
    L.partial = take(sddmm ? (size_t)max_split * nnz * 4 : 0);
    L.img = take(spmm ? ((size_t)4 * nnz + P * kPM * kKC) * 2 : 0);
    L.total = off + 1024;  // slack for aligning the base
    return L;
}

PanelWs carve(void* ws, const Layout& L) {
    char* b = reinterpret_cast<char*>(align_up(reinterpret_cast<uintptr_t>(ws), 1024));
    PanelWs w;
    w.desc = reinterpret_cast<int4*>(b + L.desc);
    w.prow = reinterpret_cast<int32_t*>(b + L.prow);
    w.ulist = reinterpret_cast<int32_t*>(b + L.ulist);
    w.upos = reinterpret_cast<uint16_t*>(b + L.upos);
    w.dense = reinterpret_cast<uint8_t*>(b + L.dense);
    w.counts = reinterpret_cast<int32_t*>(b + L.counts);
    w.dlist = reinterpret_cast<int32_t*>(b + L.dlist);
    w.items = reinterpret_cast<int32_t*>(b + L.items);
    w.partial = reinterpret_cast<float*>(b + L.partial);
    w.img = b + L.img;
    return w;
}

int sddmm_max_split(int32_t nnz, int32_t kd) {
    const int nkc = (kd + kKC - 1) / kKC;
    size_t by_mem = nnz > 0 ? kPartialBudget / ((size_t)nnz * 4) : kMaxSplit;
    int s = (int)min64((int64_t)kMaxSplit, (int64_t)by_mem);
    s = (int)min64(s, nkc);
    return s < 1 ? 1 : s;
}

bool panels_possible(int dt, int32_t m, int32_t ncols) {
    return (dt == kF16 || dt == kBF16) && m > 0 && ncols > 0 && ncols <= kMaxWords * 32;
}

// ------------------------------------------------------------------ plan kernels

__device__ __forceinline__ int warp_sum(int v) {
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

template <typename I>
__global__ void __launch_bounds__(256) plan_panels_kernel(const int32_t* __restrict__ ro, const I* __restrict__ row_idx,
                                                          const I* __restrict__ col, int32_t m, int32_t ncols,
                                                          PanelWs ws) {
    __shared__ uint32_t bitmap[kMaxWords];
    __shared__ uint32_t wbase[kMaxWords];
    __shared__ int32_t rows[kPM];
    __shared__ int32_t red[8];
    __shared__ int32_t scan[256];
    const int p = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int words = (ncols + 31) >> 5;
    if (tid < kPM) {
        const int64_t pos = (int64_t)p * kPM + tid;
        const int r = pos < m ? idx_of(row_idx[pos]) : -1;
        rows[tid] = r;
        ws.prow[p * kPM + tid] = r;
    }
    for (int w = tid; w < words; w += 256) bitmap[w] = 0;
    __syncthreads();
    int cnt = 0;
    for (int r = warp; r < kPM; r += 8) {
        const int i = rows[r];
        if (i < 0) continue;
        const int32_t k1 = ro[i + 1];
        for (int32_t k = ro[i] + lane; k < k1; k += 32) {
            const int c = idx_of(col[k]);
            atomicOr(&bitmap[c >> 5], 1u << (c & 31));
            ++cnt;
        }
    }
    cnt = warp_sum(cnt);
    if (lane == 0) red[warp] = cnt;
    __syncthreads();
    int nnz_p = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) nnz_p += red[w];
    // exclusive scan of the words' popcounts
    const int per = (words + 255) / 256;
    const int b = tid * per, e = min(words, b + per);
    int s = 0;
    for (int w = b; w < e; ++w) s += __popc(bitmap[w]);
    scan[tid] = s;
    __syncthreads();
    for (int off = 1; off < 256; off <<= 1) {
        const int v = tid >= off ? scan[tid - off] : 0;
        __syncthreads();
        scan[tid] += v;
        __syncthreads();
    }
    int run = tid ? scan[tid - 1] : 0;
    for (int w = b; w < e; ++w) {
        wbase[w] = run;
        run += __popc(bitmap[w]);
    }
    const int U = scan[255];
    __syncthreads();
    const bool dense = nnz_p > 0 && U <= kUCap && (int64_t)nnz_p * 4 >= (int64_t)kPM * U;
    if (tid == 0) {
        ws.desc[p] = make_int4(dense ? 1 : 0, U, nnz_p, 0);
        ws.dense[p] = dense ? 1 : 0;
    }
    if (!dense) return;
    for (int w = tid; w < words; w += 256) {
        uint32_t bits = bitmap[w];
        int at = wbase[w];
        while (bits) {
            const int bit = __ffs(bits) - 1;
            ws.ulist[p * kUCap + at++] = w * 32 + bit;
            bits &= bits - 1;
        }
    }
    for (int r = warp; r < kPM; r += 8) {
        const int i = rows[r];
        if (i < 0) continue;
        const int32_t k1 = ro[i + 1];
        for (int32_t k = ro[i] + lane; k < k1; k += 32) {
            const int c = idx_of(col[k]);
            ws.upos[k] = (uint16_t)(wbase[c >> 5] + __popc(bitmap[c >> 5] & ((1u << (c & 31)) - 1u)));
        }
    }
}

// Block-wide exclusive scan (1024 threads) of one int; returns the block total in *total.
__device__ __forceinline__ int block_scan_1024(int v, int* sh, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sh[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = sh[lane];
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        sh[lane] = w;
    }
    __syncthreads();
    const int before = (warp ? sh[warp - 1] : 0) + x - v;
    *total = sh[31];
    __syncthreads();
    return before;
}

__global__ void __launch_bounds__(1024) plan_worklist_kernel(int32_t P, PanelWs ws) {
    __shared__ int sh[32];
    int cd = 0, ct = 0, ci = 0;
    for (int base = 0; base < P; base += 1024) {
        const int p = base + threadIdx.x;
        int4 d = p < P ? ws.desc[p] : make_int4(0, 0, 0, 0);
        const int dn = d.x;
        const int tiles = dn ? (d.y + kSdNT - 1) / kSdNT : 0;
        const int img = dn ? kPM * ((d.y + kKC - 1) / kKC) * kKC : 0;
        int td, tt, ti;
        const int ed = block_scan_1024(dn, sh, &td);
        const int et = block_scan_1024(tiles, sh, &tt);
        const int ei = block_scan_1024(img, sh, &ti);
        if (dn) {
            ws.dlist[cd + ed] = p;
            for (int j = 0; j < tiles; ++j) ws.items[ct + et + j] = (p << 8) | j;
            ws.desc[p].w = ci + ei;
        }
        cd += td;
        ct += tt;
        ci += ti;
    }
    if (threadIdx.x == 0) {
        ws.counts[0] = cd;
        ws.counts[1] = ct;
        ws.counts[2] = ci;
        ws.counts[3] = 0;
    }
}

// ------------------------------------------------------------------ SDDMM dense panels

__device__ __forceinline__ int choose_split(int items, int grid, int max_split, int nkc) {
    int s = items > 0 ? grid / items : 1;
    s = s < 1 ? 1 : s;
    s = s > max_split ? max_split : s;
    s = s > nkc ? nkc : s;
    const int per = (nkc + s - 1) / s;
    return (nkc + per - 1) / per;  // splits actually used (each gets >= 1 chunk)
}

template <typename T>
__global__ void __launch_bounds__(kTileThreads, 1)
sddmm_panel_kernel(const int32_t* __restrict__ ro, const T* __restrict__ A, const T* __restrict__ BT,
                   T* __restrict__ out, int32_t kd, int32_t nnz, PanelWs ws, int max_split, uint32_t idesc,
                   int* err) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t mma_bar[kStages];
    __shared__ uint32_t tmem_base_sh;
    __shared__ int32_t s_rows[kPM];
    __shared__ int32_t s_u[kSdNT];
    uint8_t* smem = reinterpret_cast<uint8_t*>(align_up(reinterpret_cast<uintptr_t>(smem_raw), 1024));
    const uint32_t sbase = smem_u32(smem);
    const int tid = threadIdx.x, warp = tid >> 5;

    if (warp == 0) tc::tmem_alloc(smem_u32(&tmem_base_sh), kSdNT);
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(smem_u32(&mma_bar[s]), 1);
        fence_mbar_init();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = tmem_base_sh;

    const int nitems = ws.counts[1];
    const int nkc = (kd + kKC - 1) / kKC;
    const int S = choose_split(nitems, gridDim.x, max_split, nkc);
    const int kc_per = (nkc + S - 1) / S;
    const int64_t units = (int64_t)nitems * S;
    uint32_t g = 0;  // chunks consumed so far by this CTA: stage = g % kStages
    bool failed = false;

    for (int64_t unit = blockIdx.x; unit < units && !failed; unit += gridDim.x) {
        const int item = ws.items[unit / S];
        const int split = (int)(unit % S);
        const int p = item >> 8, t = item & 255;
        const int kc0 = split * kc_per;
        const int nk = min(nkc, kc0 + kc_per) - kc0;
        const int nU = ws.desc[p].y;
        const int u0 = t * kSdNT;
        const int ncols = min(kSdNT, nU - u0);
        __syncthreads();  // the previous unit's epilogue is done with s_rows / smem
        s_rows[tid] = ws.prow[p * kPM + tid];
        s_u[tid] = tid < ncols ? ws.ulist[p * kUCap + u0 + tid] : -1;
        __syncthreads();

        auto load = [&](int j, uint32_t gs) {
            const uint32_t st = sbase + (gs % kStages) * kSdStageBytes;
            const int k0 = (kc0 + j) * kKC;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int c = tid + kTileThreads * q;
                const int row = c >> 3, kch = c & 7;
                const int kk = k0 + kch * 8;
                const uint32_t off = tc::sw128_off(row, kch);
                const int r = s_rows[row];
                const bool oka = r >= 0 && kk < kd;
                tc::cp_async16(st + off, oka ? (const void*)(A + (int64_t)r * kd + kk) : (const void*)A, oka ? 16 : 0);
                const int cc = s_u[row];
                const bool okb = cc >= 0 && kk < kd;
                tc::cp_async16(st + kPM * kKC * 2 + off, okb ? (const void*)(BT + (int64_t)cc * kd + kk) : (const void*)BT,
                               okb ? 16 : 0);
            }
            tc::cp_async_commit();
        };

        for (int j = 0; j < kStages - 1; ++j) {
            if (j < nk) load(j, g + j);
            else tc::cp_async_commit();
        }
        for (int j = 0; j < nk; ++j) {
            const uint32_t gs = g + j;
            const uint32_t st = sbase + (gs % kStages) * kSdStageBytes;
            tc::cp_async_wait<kStages - 2>();
            fence_proxy_async_smem();
            __syncthreads();
            if (tid == 0) {
                tc::fence_after_sync();
#pragma unroll
                for (int kk = 0; kk < kKC / 16; ++kk) {
                    const uint64_t ad = tc::smem_desc_sw128(st + kk * 32, 16, 1024);
                    const uint64_t bd = tc::smem_desc_sw128(st + kPM * kKC * 2 + kk * 32, 16, 1024);
                    tc::mma_f16(tmem, ad, bd, idesc, (j > 0 || kk > 0) ? 1u : 0u);
                }
                tc::mma_commit(smem_u32(&mma_bar[gs % kStages]));
            }
            const int jn = j + kStages - 1;
            if (jn < nk) {
                if (j >= 1) {
                    const uint32_t gp = gs - 1;
                    if (!mbar_wait(smem_u32(&mma_bar[gp % kStages]), (gp / kStages) & 1u, err)) failed = true;
                }
                load(jn, gs + kStages - 1);
            } else {
                tc::cp_async_commit();
            }
        }
        {
            const uint32_t gl = g + nk - 1;
            if (!mbar_wait(smem_u32(&mma_bar[gl % kStages]), (gl / kStages) & 1u, err)) failed = true;
        }
        g += nk;
        tc::cp_async_wait<0>();
        if (__syncthreads_or(failed)) {
            failed = true;
            break;
        }
        tc::fence_after_sync();

        // epilogue: TMEM row tid -> padded shared scratch -> the row's entries in this tile
        float* scratch = reinterpret_cast<float*>(smem);
        const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16);
#pragma unroll 1
        for (int c = 0; c < kSdNT / 32; ++c) {
            float v[32];
            tc::tmem_ld32(lane_addr + c * 32, v);
#pragma unroll
            for (int x = 0; x < 32; ++x) scratch[tid * (kSdNT + 1) + c * 32 + x] = v[x];
        }
        tc::fence_before_sync();
        const int i = s_rows[tid];
        if (i >= 0) {
            int32_t lo = ro[i], hi = ro[i + 1];
            while (lo < hi) {  // first entry with upos >= u0
                const int32_t mid = (lo + hi) >> 1;
                if ((int)ws.upos[mid] < u0) lo = mid + 1;
                else hi = mid;
            }
            const int32_t k1 = ro[i + 1];
            for (int32_t k = lo; k < k1; ++k) {
                const int u = (int)ws.upos[k] - u0;
                if (u >= ncols) break;
                const float v = scratch[tid * (kSdNT + 1) + u];
                if (S == 1) out[k] = Elt<T>::from_f(v);
                else ws.partial[(int64_t)split * nnz + k] = v;
            }
        }
    }
    tc::cp_async_wait<0>();
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, kSdNT);
}

// out[k] = sum over splits, in split order, of the partial sums (dense panels only).
template <typename T>
__global__ void __launch_bounds__(256) sddmm_finalize_kernel(const int32_t* __restrict__ ro, T* __restrict__ out,
                                                             int32_t nnz, int32_t kd, PanelWs ws, int grid_tiles,
                                                             int max_split) {
    const int p = blockIdx.x;
    if (!ws.dense[p]) return;
    const int nkc = (kd + kKC - 1) / kKC;
    const int S = choose_split(ws.counts[1], grid_tiles, max_split, nkc);
    if (S == 1) return;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int r = warp; r < kPM; r += 8) {
        const int i = ws.prow[p * kPM + r];
        if (i < 0) continue;
        const int32_t k1 = ro[i + 1];
        for (int32_t k = ro[i] + lane; k < k1; k += 32) {
            float s = ws.partial[k];
            for (int sp = 1; sp < S; ++sp) s += ws.partial[(int64_t)sp * nnz + k];
            out[k] = Elt<T>::from_f(s);
        }
    }
}

// ------------------------------------------------------------------ SpMM dense panels

template <typename T>
__global__ void __launch_bounds__(256) densify_kernel(const T* __restrict__ vals, const int32_t* __restrict__ ro,
                                                      PanelWs ws) {
    const int p = blockIdx.x;
    if (!ws.dense[p]) return;
    const int4 d = ws.desc[p];
    const int upad = (d.y + kKC - 1) / kKC * kKC;
    T* img = static_cast<T*>(ws.img) + d.w;
    uint4* img4 = reinterpret_cast<uint4*>(img);
    const int n16 = kPM * upad * 2 / 16;
    for (int x = threadIdx.x; x < n16; x += 256) img4[x] = make_uint4(0, 0, 0, 0);
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int r = warp; r < kPM; r += 8) {
        const int i = ws.prow[p * kPM + r];
        if (i < 0) continue;
        const int32_t k1 = ro[i + 1];
        for (int32_t k = ro[i] + lane; k < k1; k += 32) {
            const int u = ws.upos[k];
            const int chunk = u / kKC, w = u % kKC;
            const uint32_t byte = tc::sw128_off(r, (w * 2) >> 4) + ((w * 2) & 15);
            img[(size_t)chunk * (kPM * kKC) + byte / 2] = vals[k];
        }
    }
}

template <typename T>
__global__ void __launch_bounds__(kTileThreads, 1)
spmm_panel_kernel(const T* __restrict__ B, T* __restrict__ C, int32_t N, PanelWs ws, uint32_t idesc, int* err) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t mma_bar[kStages];
    __shared__ uint32_t tmem_base_sh;
    __shared__ int32_t s_u[kUCap];
    uint8_t* smem = reinterpret_cast<uint8_t*>(align_up(reinterpret_cast<uintptr_t>(smem_raw), 1024));
    const uint32_t sbase = smem_u32(smem);
    const int tid = threadIdx.x, warp = tid >> 5;

    if (warp == 0) tc::tmem_alloc(smem_u32(&tmem_base_sh), kSpNT);
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(smem_u32(&mma_bar[s]), 1);
        fence_mbar_init();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = tmem_base_sh;

    const int D = ws.counts[0];
    const int ntn = (N + kSpNT - 1) / kSpNT;
    const int64_t units = (int64_t)D * ntn;
    uint32_t g = 0;
    bool failed = false;

    for (int64_t unit = blockIdx.x; unit < units && !failed; unit += gridDim.x) {
        const int p = ws.dlist[unit / ntn];
        const int n0 = (int)(unit % ntn) * kSpNT;
        const int4 d = ws.desc[p];
        const int nU = d.y;
        const int nk = (nU + kKC - 1) / kKC;
        const T* img = static_cast<const T*>(ws.img) + d.w;
        __syncthreads();
        for (int x = tid; x < nk * kKC; x += kTileThreads) s_u[x] = x < nU ? ws.ulist[p * kUCap + x] : -1;
        __syncthreads();

        auto load = [&](int j, uint32_t gs) {
            const uint32_t st = sbase + (gs % kStages) * kSpStageBytes;
            const char* src_a = reinterpret_cast<const char*>(img + (size_t)j * kPM * kKC);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int c = tid + kTileThreads * q;
                tc::cp_async16(st + c * 16, src_a + c * 16, 16);
            }
#pragma unroll
            for (int q = 0; q < 16; ++q) {
                const int c = tid + kTileThreads * q;
                const int kk = c >> 5, nch = c & 31;
                const int u = s_u[j * kKC + kk];
                const int ncol = n0 + nch * 8;
                const bool ok = u >= 0 && ncol < N;
                const uint32_t off = (uint32_t)(nch >> 3) * (kKC / 8 * 1024) + tc::sw128_off(kk, nch & 7);
                tc::cp_async16(st + kSpStageA + off, ok ? (const void*)(B + (int64_t)u * N + ncol) : (const void*)B,
                               ok ? 16 : 0);
            }
            tc::cp_async_commit();
        };

        for (int j = 0; j < kStages - 1; ++j) {
            if (j < nk) load(j, g + j);
            else tc::cp_async_commit();
        }
        for (int j = 0; j < nk; ++j) {
            const uint32_t gs = g + j;
            const uint32_t st = sbase + (gs % kStages) * kSpStageBytes;
            tc::cp_async_wait<kStages - 2>();
            fence_proxy_async_smem();
            __syncthreads();
            if (tid == 0) {
                tc::fence_after_sync();
#pragma unroll
                for (int kk = 0; kk < kKC / 16; ++kk) {
                    const uint64_t ad = tc::smem_desc_sw128(st + kk * 32, 16, 1024);
                    const uint64_t bd = tc::smem_desc_sw128(st + kSpStageA + kk * 2048, kKC / 8 * 1024, 1024);
                    tc::mma_f16(tmem, ad, bd, idesc, (j > 0 || kk > 0) ? 1u : 0u);
                }
                tc::mma_commit(smem_u32(&mma_bar[gs % kStages]));
            }
            const int jn = j + kStages - 1;
            if (jn < nk) {
                if (j >= 1) {
                    const uint32_t gp = gs - 1;
                    if (!mbar_wait(smem_u32(&mma_bar[gp % kStages]), (gp / kStages) & 1u, err)) failed = true;
                }
                load(jn, gs + kStages - 1);
            } else {
                tc::cp_async_commit();
            }
        }
        {
            const uint32_t gl = g + nk - 1;
            if (!mbar_wait(smem_u32(&mma_bar[gl % kStages]), (gl / kStages) & 1u, err)) failed = true;
        }
        g += nk;
        tc::cp_async_wait<0>();
        if (__syncthreads_or(failed)) {
            failed = true;
            break;
        }
        tc::fence_after_sync();

        // epilogue: TMEM row tid -> C[row, n0 .. n0 + 256)
        const int i = ws.prow[p * kPM + tid];
        const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16);
#pragma unroll 1
        for (int c = 0; c < kSpNT / 32; ++c) {
            float v[32];
            tc::tmem_ld32(lane_addr + c * 32, v);
            if (i >= 0) {
                T* dst = C + (int64_t)i * N + n0 + c * 32;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    if (n0 + c * 32 + q * 8 < N)
                        *reinterpret_cast<uint4*>(dst + q * 8) = Elt<T>::pack(v + q * 8);
                }
            }
        }
        tc::fence_before_sync();
    }
    tc::cp_async_wait<0>();
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, kSpNT);
}

// ------------------------------------------------------------------ host dispatch

template <typename I>
cudaError_t launch_plan(const int32_t* ro, const void* row_idx, const void* col, int32_t m, int32_t ncols,
                        const PanelWs& w, cudaStream_t s) {
    const int P = (m + kPM - 1) / kPM;
    plan_panels_kernel<I><<<P, 256, 0, s>>>(ro, static_cast<const I*>(row_idx), static_cast<const I*>(col), m, ncols,
                                            w);
    plan_worklist_kernel<<<1, 1024, 0, s>>>(P, w);
    count_launches(2);
    return cudaGetLastError();
}

template <typename T>
cudaError_t run_sddmm_panels(int it, const int32_t* ro, const void* row_idx, const void* col, int32_t m, int32_t n,
                             int32_t kd, int32_t nnz, const void* A, const void* BT, void* out, const PanelWs& w,
                             int max_split, cudaStream_t s) {
    cudaError_t e = it == kIdx16 ? launch_plan<uint16_t>(ro, row_idx, col, m, n, w, s)
                                 : launch_plan<int32_t>(ro, row_idx, col, m, n, w, s);
    if (e != cudaSuccess) return e;
    const int P = (m + kPM - 1) / kPM;
    const int max_items = P * (kUCap / kSdNT);
    const int grid = (int)min64((int64_t)device_props().sm_count, (int64_t)max_items * max_split);
    auto kern = sddmm_panel_kernel<T>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSdSmem);
    if (e != cudaSuccess) return e;
    const uint32_t idesc = tc::instr_desc_f16(std::is_same<T, __nv_bfloat16>::value ? 1u : 0u, 0, 0, kPM, kSdNT);
    kern<<<grid, kTileThreads, kSdSmem, s>>>(ro, static_cast<const T*>(A), static_cast<const T*>(BT),
                                             static_cast<T*>(out), kd, nnz, w, max_split, idesc,
                                             device_error_word());
    sddmm_finalize_kernel<T><<<P, 256, 0, s>>>(ro, static_cast<T*>(out), nnz, kd, w, grid, max_split);
    count_launches(2);
    return cudaGetLastError();
}

template <typename T>
cudaError_t run_spmm_panels(int it, const void* vals, const int32_t* ro, const void* row_idx, const void* col,
                            int32_t m, int32_t k, const void* B, int32_t N, void* C, const PanelWs& w,
                            cudaStream_t s) {
    cudaError_t e = it == kIdx16 ? launch_plan<uint16_t>(ro, row_idx, col, m, k, w, s)
                                 : launch_plan<int32_t>(ro, row_idx, col, m, k, w, s);
    if (e != cudaSuccess) return e;
    const int P = (m + kPM - 1) / kPM;
    densify_kernel<T><<<P, 256, 0, s>>>(static_cast<const T*>(vals), ro, w);
    const int ntn = (N + kSpNT - 1) / kSpNT;
    const int grid = (int)min64((int64_t)device_props().sm_count, (int64_t)P * ntn);
    auto kern = spmm_panel_kernel<T>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSpSmem);
    if (e != cudaSuccess) return e;
    const uint32_t idesc = tc::instr_desc_f16(std::is_same<T, __nv_bfloat16>::value ? 1u : 0u, 0, 1, kPM, kSpNT);
    kern<<<grid, kTileThreads, kSpSmem, s>>>(static_cast<const T*>(B), static_cast<T*>(C), N, w, idesc,
                                             device_error_word());
    count_launches(2);
    return cudaGetLastError();
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

__global__ void __launch_bounds__(1024) panel_stats_kernel(int32_t P, PanelWs ws, int32_t* out) {
    __shared__ int sh[32];
    int d = 0, e = 0;
    for (int p = threadIdx.x; p < P; p += 1024) {
        const int4 x = ws.desc[p];
        d += x.x;
        e += x.x ? x.z : 0;
    }
    int td, te;
    block_scan_1024(d, sh, &td);
    block_scan_1024(e, sh, &te);
    if (threadIdx.x == 0) {
        out[0] = td;
        out[1] = te;
        out[2] = ws.counts[1];
        out[3] = P;
    }
}

}  // namespace

size_t panel_plan_workspace_bytes(int32_t m, int32_t nnz) { return layout(m, nnz, false, 1, false).total; }

cudaError_t launch_panel_plan(int it, const int32_t* ro, const void* row_idx, const void* col, int32_t m, int32_t n,
                              int32_t nnz, int32_t* stats, void* ws, cudaStream_t s) {
    const Layout L = layout(m, nnz, false, 1, false);
    const PanelWs w = carve(ws, L);
    cudaError_t e = it == kIdx16 ? launch_plan<uint16_t>(ro, row_idx, col, m, n, w, s)
                                 : launch_plan<int32_t>(ro, row_idx, col, m, n, w, s);
    if (e != cudaSuccess) return e;
    panel_stats_kernel<<<1, 1024, 0, s>>>((m + kPM - 1) / kPM, w, stats);
    count_launches(1);
    return cudaGetLastError();
}

size_t panel_spmm_workspace_bytes(int32_t m, int32_t k, int32_t n, int32_t nnz, int dt, int it) {
    (void)it;
    (void)n;
    if (!panels_possible(dt, m, k)) return 0;
    return layout(m, nnz, false, 1, true).total;
}

size_t panel_sddmm_workspace_bytes(int32_t m, int32_t n, int32_t kd, int32_t nnz, int dt, int it) {
    (void)it;
    if (!panels_possible(dt, m, n) || kd <= 0) return 0;
    return layout(m, nnz, true, sddmm_max_split(nnz, kd), false).total;
}

cudaError_t launch_spmm(int dt, int it, const void* vals, const int32_t* ro, const void* row_idx, const void* col,
                        int32_t m, int32_t k, int32_t nnz, const void* B, int32_t n, void* C, const int32_t* bins,
                        void* ws, bool allow_panels, cudaStream_t s) {
    const bool panels = allow_panels && nnz > 0 && panels_possible(dt, m, k) && n % 8 == 0 && aligned16(B) &&
                        aligned16(C);
    if (!panels) return launch_spmm_general(dt, it, vals, ro, row_idx, col, m, k, B, n, C, bins, nullptr, s);
    const Layout L = layout(m, nnz, false, 1, true);
    const PanelWs w = carve(ws, L);
    cudaError_t e = dt == kF16 ? run_spmm_panels<__half>(it, vals, ro, row_idx, col, m, k, B, n, C, w, s)
                               : run_spmm_panels<__nv_bfloat16>(it, vals, ro, row_idx, col, m, k, B, n, C, w, s);
    if (e != cudaSuccess) return e;
    return launch_spmm_general(dt, it, vals, ro, row_idx, col, m, k, B, n, C, bins, w.dense, s);
}

cudaError_t launch_sddmm(int dt, int it, const int32_t* ro, const void* row_idx, const void* col, int32_t m,
                         int32_t n, int32_t kd, int32_t nnz, const void* A, const void* BT, void* out,
                         bool structure_aware, const int32_t* bins, void* ws, cudaStream_t s) {
    const bool panels = structure_aware && nnz > 0 && panels_possible(dt, m, n) && kd > 0 && kd % 8 == 0 &&
                        aligned16(A) && aligned16(BT);
    if (!panels) return launch_sddmm_general(dt, it, ro, row_idx, col, m, n, kd, A, BT, out, bins, nullptr, s);
    const int max_split = sddmm_max_split(nnz, kd);
    const Layout L = layout(m, nnz, true, max_split, false);
    const PanelWs w = carve(ws, L);
    cudaError_t e = dt == kF16
                        ? run_sddmm_panels<__half>(it, ro, row_idx, col, m, n, kd, nnz, A, BT, out, w, max_split, s)
                        : run_sddmm_panels<__nv_bfloat16>(it, ro, row_idx, col, m, n, kd, nnz, A, BT, out, w,
                                                          max_split, s);
    if (e != cudaSuccess) return e;
    return launch_sddmm_general(dt, it, ro, row_idx, col, m, n, kd, A, BT, out, bins, w.dense, s);
}

}  // namespace spops
