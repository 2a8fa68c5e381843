// Structure-aware path: dense panels of the CSR matrix on the tcgen05 tensor cores.
//
// spops README ("Sparse Operations (spops)"), section "Sampled Dense-Dense Matrix
// Multiplication (SDDMM)": besides the general kernel, SDDMM has a structure-aware kernel
// for the masks seen in RoSA, whose non-zeros cluster in a small subset of rows and
// columns. The mask plan (plan.cu) groups row_idx positions into panels of 128 rows and
// marks a panel dense when its entries fill its 128 x |U| tile well (U = the union of the
// panel's columns). Here:
//   * SDDMM: D = A[panel rows, :] * BT[U, :]^T per (panel, 128-column tile of U, K split)
//     on tcgen05 (fp16/bf16 operands, fp32 accumulators in tensor memory); the epilogue
//     reads each row's entries of the tile (contiguous, located by the plan's tile starts)
//     out of D. With fewer tiles than SMs, K is split in up to 16 parts whose fp32 partial
//     sums a finalize kernel adds in split order, so results are deterministic.
//   * SpMM: each dense panel's values are written into a 128 x |U| image already in the
//     UMMA K-major 128-byte-swizzled layout; C[panel rows, 128-column tile] =
//     image * B[U, tile] on tcgen05, with B's rows gathered into an MN-major swizzled tile.
//   * the other rows run through the general row kernels, which skip dense panels.
// Operands are gathered row by row with 16-byte cp.async copies into a 3-stage shared
// memory ring (two CTAs per SM, so two units' latency chains overlap); one thread issues
// the MMAs and commits them to per-stage mbarriers, whose completion frees the stage for
// the next copy. Every mbarrier wait is bounded in time.
#include <type_traits>

#include "common.cuh"
#include "internal.h"
#include "panel.h"
#include "plan.h"
#include "tc.cuh"

namespace spops {
namespace {

constexpr int kKC = 64;       // K elements per pipeline chunk (128 bytes of 16-bit data)
constexpr int kStages = 3;      // 3 x 32 KB ring: two CTAs per SM
constexpr int kSpNT = 128;    // SpMM: columns of C per tile (UMMA N)
constexpr int kMaxSplit = 16;
constexpr size_t kPartialBudget = 64ull << 20;  // bytes of fp32 split-K partial sums
constexpr int kTileThreads = 128;

constexpr uint32_t kSdStageA = kPM * kKC * 2;                 // 16 KB
constexpr uint32_t kSdStageBytes = kSdStageA + kTileN * kKC * 2;  // A + BT tiles: 32 KB
constexpr uint32_t kSpStageA = kPM * kKC * 2;                 // 16 KB
constexpr uint32_t kSpStageB = kSpNT * kKC * 2;               // 16 KB
constexpr uint32_t kSpStageBytes = kSpStageA + kSpStageB;     // 32 KB
constexpr uint32_t kSdSmem = kStages * kSdStageBytes + 1024;
constexpr uint32_t kSpSmem = kStages * kSpStageBytes + 1024;

bool dtype_ok(int dt) { return dt == kF16 || dt == kBF16; }

// Most K splits a call may use: bounded by the chunks of K and by the partial-sum budget.
int sddmm_max_split(int32_t kd, int32_t nnz) {
    const int64_t nkc = (kd + kKC - 1) / kKC;
    const int64_t by_mem = nnz > 0 ? (int64_t)(kPartialBudget / ((size_t)nnz * 4)) : kMaxSplit;
    const int64_t s = min64(min64(kMaxSplit, nkc), by_mem);
    return s < 1 ? 1 : (int)s;
}

// Number of K splits given the work items and the grid (identical on every CTA).
__host__ __device__ __forceinline__ int choose_split(int items, int grid, int max_split, int nkc) {
    int s = items > 0 ? grid / items : 1;
    s = s < 1 ? 1 : s;
    s = s > max_split ? max_split : s;
    s = s > nkc ? nkc : s;
    const int per = (nkc + s - 1) / s;
    return (nkc + per - 1) / per;  // every split gets at least one chunk
}

// ------------------------------------------------------------------ SDDMM dense panels

template <typename T>
__global__ void __launch_bounds__(kTileThreads, 2)
sddmm_panel_kernel(const T* __restrict__ A, const T* __restrict__ BT, T* __restrict__ out, float* __restrict__ partial,
                   int32_t kd, PlanView v, int max_split, uint32_t idesc, int* err) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t mma_bar[kStages];
    __shared__ uint32_t tmem_base_sh;
    __shared__ int32_t s_rows[kPM];
    __shared__ int32_t s_u[kTileN];
    __shared__ int32_t s_off[kPM], s_kb[kPM], s_cnt[kPM];
    __shared__ int32_t s_wsum[kTileThreads / 32];
    uint8_t* smem = reinterpret_cast<uint8_t*>(align_up(reinterpret_cast<uintptr_t>(smem_raw), 1024));
    const uint32_t sbase = smem_u32(smem);
    const int tid = threadIdx.x, warp = tid >> 5;

    if (warp == 0) tc::tmem_alloc(smem_u32(&tmem_base_sh), kTileN);
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(smem_u32(&mma_bar[s]), 1);
        fence_mbar_init();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = tmem_base_sh;

    const int nitems = v.counts()[kCntTiles];
    const int nkc = (kd + kKC - 1) / kKC;
    const int S = choose_split(nitems, gridDim.x, max_split, nkc);
    const int kc_per = (nkc + S - 1) / S;
    const int64_t units = (int64_t)nitems * S;
    uint32_t g = 0;  // chunks consumed so far by this CTA: stage = g % kStages
    bool failed = false;

    for (int64_t unit = blockIdx.x; unit < units && !failed; unit += gridDim.x) {
        const int item = v.items[unit / S];
        const int split = (int)(unit % S);
        const int p = item >> 8, t = item & 255;
        const int kc0 = split * kc_per;
        const int nk = min(nkc, kc0 + kc_per) - kc0;
        const int nU = v.desc[p].y;
        const int u0 = t * kTileN;
        const int ncols = min(kTileN, nU - u0);
        __syncthreads();  // the previous unit's epilogue is done with s_rows and the stages
        const int my_row = v.prow[p * kPM + tid];
        s_rows[tid] = my_row;
        s_u[tid] = tid < ncols ? v.ulist[(size_t)p * kUCap + u0 + tid] : -1;
        // The epilogue's per-row metadata (see below), loaded now so that its latency hides
        // behind the operand copies.
        int32_t kb = 0, cnt = 0;
        uint32_t mk[kTileN / 32];
#pragma unroll
        for (int c = 0; c < kTileN / 32; ++c) mk[c] = 0;
        if (my_row >= 0) {
            const size_t prow_at = (size_t)p * kPM + tid;
            const int32_t* ts = v.ts + prow_at * (kTiles + 1);
            kb = ts[t];
            cnt = ts[t + 1] - kb;
            const uint32_t* tm = v.tmask + prow_at * (kUCap / 32) + t * (kTileN / 32);
#pragma unroll
            for (int c = 0; c < kTileN / 32; ++c) mk[c] = tm[c];
        }
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
                tc::cp_async16(st + kSdStageA + off, okb ? (const void*)(BT + (int64_t)cc * kd + kk) : (const void*)BT,
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
                    const uint64_t bd = tc::smem_desc_sw128(st + kSdStageA + kk * 32, 16, 1024);
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

        // epilogue. Thread tid owns TMEM lane tid = panel row tid. The plan's mask says which
        // of the tile's 128 columns the row holds; its k-th set bit is the row's k-th entry
        // of the tile (entries and U are both in column order), starting at ts[t]. Each
        // thread packs its row's sampled values into a shared staging area (register index
        // fixed per bit, no loads of entry positions), then warps copy whole rows out with
        // coalesced stores.
        const int lane = tid & 31;
        int incl = cnt;  // exclusive scan of cnt over the 128 rows
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        if (lane == 31) s_wsum[warp] = incl;
        __syncthreads();
        int off = incl - cnt;
        for (int w = 0; w < warp; ++w) off += s_wsum[w];
        s_off[tid] = off;
        s_kb[tid] = kb;
        s_cnt[tid] = cnt;
        float* stage = reinterpret_cast<float*>(smem);
        const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16);
        int rank = off;
#pragma unroll
        for (int c = 0; c < kTileN / 32; ++c) {
            float x[32];
            tc::tmem_ld32(lane_addr + c * 32, x);
            const uint32_t word = mk[c];
#pragma unroll
            for (int q = 0; q < 32; ++q) {
                if ((word >> q) & 1u) stage[rank++] = x[q];
            }
        }
        tc::fence_before_sync();
        __syncthreads();
        for (int r = warp; r < kPM; r += kTileThreads / 32) {
            const int n_r = s_cnt[r];
            const float* src = stage + s_off[r];
            const int32_t kr = s_kb[r];
            for (int j = lane; j < n_r; j += 32) {
                if (S == 1) out[kr + j] = Elt<T>::from_f(src[j]);
                else partial[(int64_t)split * v.nnz + kr + j] = src[j];
            }
        }
    }
    tc::cp_async_wait<0>();
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, kTileN);
}

// out[k] = sum of the split partial sums in split order (dense panels, S > 1 only).
// One CTA per panel row, so even a few dense panels spread over many SMs.
constexpr int kFinalizeThreads = 128;

template <typename T>
__global__ void __launch_bounds__(kFinalizeThreads)
sddmm_finalize_kernel(const int32_t* __restrict__ ro, T* __restrict__ out, const float* __restrict__ partial,
                      int32_t kd, PlanView v, int grid_tiles, int max_split) {
    const int pos = blockIdx.x;
    if (!v.dense[pos / kPM]) return;
    const int i = v.prow[pos];
    if (i < 0) return;
    const int S = choose_split(v.counts()[kCntTiles], grid_tiles, max_split, (kd + kKC - 1) / kKC);
    if (S == 1) return;
    const int64_t nnz = v.nnz;
    const int32_t k1 = ro[i + 1];
    for (int32_t k = ro[i] + threadIdx.x; k < k1; k += kFinalizeThreads) {
        float x[kMaxSplit];
#pragma unroll
        for (int sp = 0; sp < kMaxSplit; ++sp) x[sp] = sp < S ? partial[sp * nnz + k] : 0.f;
        float s = x[0];
#pragma unroll
        for (int sp = 1; sp < kMaxSplit; ++sp)
            if (sp < S) s += x[sp];
        out[k] = Elt<T>::from_f(s);
    }
}

// ------------------------------------------------------------------ SpMM dense panels

// The 16 image rows of one row group: zeros, then the group's values at their U position,
// written out as whole 128-byte-swizzled K-major rows (16-byte stores).
template <typename T>
__global__ void __launch_bounds__(256) densify_kernel(const T* __restrict__ vals, const int32_t* __restrict__ ro,
                                                     T* __restrict__ img_base, PlanView v) {
    __shared__ __align__(16) T stage[kGroupRows][kUCap];
    const int p = blockIdx.x / kGroups, grp = blockIdx.x % kGroups;
    if (!v.sp_dense[p]) return;
    const int nU = v.desc[p].y;
    const int upad = (nU + kKC - 1) / kKC * kKC;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint4* st4 = reinterpret_cast<uint4*>(&stage[0][0]);
    const int row_vec = kUCap * (int)sizeof(T) / 16;
    for (int x = tid; x < kGroupRows * row_vec; x += 256) {
        if ((x % row_vec) * 16 < upad * (int)sizeof(T)) st4[x] = make_uint4(0, 0, 0, 0);
    }
    __syncthreads();
    for (int rr = 0; rr < kGroupRows / 8; ++rr) {
        const int lr = warp * (kGroupRows / 8) + rr;
        const int i = v.prow[p * kPM + grp * kGroupRows + lr];
        if (i < 0) continue;
        const int32_t k1 = ro[i + 1];
        for (int32_t k = ro[i] + lane; k < k1; k += 32) stage[lr][v.upos[k]] = vals[k];
    }
    __syncthreads();
    T* img = img_base + v.img_slot[p];
    const int chunks = upad / 8;  // 16-byte chunks per image row
    for (int x = tid; x < kGroupRows * chunks; x += 256) {
        const int lr = x / chunks, c = x % chunks;
        const int r = grp * kGroupRows + lr;           // panel row = image row
        const int kc = c / 8, w = c % 8;               // 64-column chunk, 16-byte piece in it
        uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<char*>(img + (size_t)kc * kPM * kKC) +
                                              tc::sw128_off(r, w));
        *dst = reinterpret_cast<const uint4*>(&stage[lr][0])[c];
    }
}

template <typename T>
__global__ void __launch_bounds__(kTileThreads, 2)
spmm_panel_kernel(const T* __restrict__ B, T* __restrict__ C, const T* __restrict__ img_base, int32_t N, PlanView v,
                  uint32_t idesc, int* err) {
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

    const int D = v.counts()[kCntDenseSp];
    const int ntn = (N + kSpNT - 1) / kSpNT;
    const int64_t units = (int64_t)D * ntn;
    uint32_t g = 0;
    bool failed = false;

    for (int64_t unit = blockIdx.x; unit < units && !failed; unit += gridDim.x) {
        const int p = v.dlist_sp[unit / ntn];
        const int n0 = (int)(unit % ntn) * kSpNT;
        const int nU = v.desc[p].y;
        const int nk = (nU + kKC - 1) / kKC;
        const T* img = img_base + v.img_slot[p];
        __syncthreads();
        for (int x = tid; x < nk * kKC; x += kTileThreads) s_u[x] = x < nU ? v.ulist[(size_t)p * kUCap + x] : -1;
        __syncthreads();

        auto load = [&](int j, uint32_t gs) {
            const uint32_t st = sbase + (gs % kStages) * kSpStageBytes;
            const char* src_a = reinterpret_cast<const char*>(img + (size_t)j * kPM * kKC);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int c = tid + kTileThreads * q;
                tc::cp_async16(st + c * 16, src_a + c * 16, 16);
            }
            // B[U rows j*64 .. +64, n0 .. n0 + kSpNT): kSpNT / 8 sixteen-byte pieces per row
            constexpr int kPieces = kSpNT / 8;
#pragma unroll
            for (int q = 0; q < kKC * kPieces / kTileThreads; ++q) {
                const int c = tid + kTileThreads * q;
                const int kk = c / kPieces, nch = c % kPieces;
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
        const int i = v.prow[p * kPM + tid];
        const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16);
#pragma unroll 1
        for (int c = 0; c < kSpNT / 32; ++c) {
            float x[32];
            tc::tmem_ld32(lane_addr + c * 32, x);
            if (i >= 0) {
                T* dst = C + (int64_t)i * N + n0 + c * 32;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    if (n0 + c * 32 + q * 8 < N) *reinterpret_cast<uint4*>(dst + q * 8) = Elt<T>::pack(x + q * 8);
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

template <typename T>
cudaError_t run_sddmm_panels(const int32_t* ro, const void* A, const void* BT, void* out, float* partial, int32_t kd,
                             const PlanView& v, cudaStream_t s) {
    const int max_split = sddmm_max_split(kd, v.nnz);
    const int max_items = v.P * kTiles;
    const int grid = (int)min64((int64_t)device_props().sm_count * 2, (int64_t)max_items * max_split);
    auto kern = sddmm_panel_kernel<T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSdSmem);
    if (e != cudaSuccess) return e;
    const uint32_t idesc = tc::instr_desc_f16(std::is_same<T, __nv_bfloat16>::value ? 1u : 0u, 0, 0, kPM, kTileN);
    kern<<<grid, kTileThreads, kSdSmem, s>>>(static_cast<const T*>(A), static_cast<const T*>(BT), static_cast<T*>(out),
                                             partial, kd, v, max_split, idesc, device_error_word());
    count_launches(1);
    if (max_split > 1) {
        sddmm_finalize_kernel<T><<<v.P * kPM, kFinalizeThreads, 0, s>>>(ro, static_cast<T*>(out), partial, kd, v,
                                                                        grid, max_split);
        count_launches(1);
    }
    return cudaGetLastError();
}

template <typename T>
cudaError_t run_spmm_panels(const void* vals, const int32_t* ro, const void* B, int32_t N, void* C, void* img,
                            const PlanView& v, cudaStream_t s) {
    densify_kernel<T><<<v.P * kGroups, 256, 0, s>>>(static_cast<const T*>(vals), ro, static_cast<T*>(img), v);
    const int ntn = (N + kSpNT - 1) / kSpNT;
    const int grid = (int)min64((int64_t)device_props().sm_count * 2, (int64_t)v.P * ntn);
    auto kern = spmm_panel_kernel<T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSpSmem);
    if (e != cudaSuccess) return e;
    const uint32_t idesc = tc::instr_desc_f16(std::is_same<T, __nv_bfloat16>::value ? 1u : 0u, 0, 1, kPM, kSpNT);
    kern<<<grid, kTileThreads, kSpSmem, s>>>(static_cast<const T*>(B), static_cast<T*>(C), static_cast<const T*>(img),
                                             N, v, idesc, device_error_word());
    count_launches(2);
    return cudaGetLastError();
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

size_t image_bytes(int dt, int32_t m, int32_t k, int32_t nnz) {
    if (!dtype_ok(dt) || !plan_panels_enabled(m, k)) return 0;
    return align_up(spmm_image_budget_elems(m, nnz) * 2, 1024);
}

size_t partial_bytes(int dt, int32_t m, int32_t n, int32_t kd, int32_t nnz) {
    if (!dtype_ok(dt) || !plan_panels_enabled(m, n) || kd <= 0) return 0;
    const int s = sddmm_max_split(kd, nnz);
    return s > 1 ? align_up((size_t)s * nnz * 4, 1024) : 0;
}

// The plan to use: the caller's, or one built now at the start of the workspace.
// Returns the view and advances *ws past the plan if it was built there.
cudaError_t resolve_plan(int it, const int32_t* ro, const void* row_idx, const void* col, int32_t m, int32_t n,
                         int32_t nnz, const void* plan, char** ws, PlanView* v, cudaStream_t s) {
    if (plan) {
        *v = plan_view(const_cast<void*>(plan), m, n, nnz);
        return cudaSuccess;
    }
    *v = plan_view(*ws, m, n, nnz);
    *ws += align_up(plan_bytes(m, n, nnz), 1024);
    return launch_plan_build(it, ro, row_idx, col, *v, (int64_t)spmm_image_budget_elems(m, nnz), s);
}

}  // namespace

size_t spmm_workspace_bytes(int32_t m, int32_t k, int32_t n, int32_t nnz, int dt) {
    (void)n;
    return 1024 + align_up(plan_bytes(m, k, nnz), 1024) + image_bytes(dt, m, k, nnz);
}

size_t sddmm_workspace_bytes(int32_t m, int32_t n, int32_t kd, int32_t nnz, int dt, bool structure_aware) {
    return 1024 + align_up(plan_bytes(m, n, nnz), 1024) + (structure_aware ? partial_bytes(dt, m, n, kd, nnz) : 0);
}

cudaError_t launch_spmm(int dt, int it, const void* vals, const int32_t* ro, const void* row_idx, const void* col,
                        int32_t m, int32_t k, int32_t nnz, const void* B, int32_t n, void* C, const void* plan,
                        void* ws, bool allow_panels, cudaStream_t s) {
    char* w = reinterpret_cast<char*>(align_up(reinterpret_cast<uintptr_t>(ws), 1024));
    PlanView v;
    cudaError_t e = resolve_plan(it, ro, row_idx, col, m, k, nnz, plan, &w, &v, s);
    if (e != cudaSuccess) return e;
    const bool panels = allow_panels && nnz > 0 && v.panels && dtype_ok(dt) && n % 8 == 0 && aligned16(B) &&
                        aligned16(C);
    if (panels) {
        e = dt == kF16 ? run_spmm_panels<__half>(vals, ro, B, n, C, w, v, s)
                       : run_spmm_panels<__nv_bfloat16>(vals, ro, B, n, C, w, v, s);
        if (e != cudaSuccess) return e;
    }
    return launch_spmm_general(dt, it, vals, ro, row_idx, col, m, k, B, n, C, v.bins_spmm(),
                               panels ? v.sp_dense : nullptr, s);
}

cudaError_t launch_sddmm(int dt, int it, const int32_t* ro, const void* row_idx, const void* col, int32_t m,
                         int32_t n, int32_t kd, int32_t nnz, const void* A, const void* BT, void* out,
                         bool structure_aware, const void* plan, void* ws, cudaStream_t s) {
    char* w = reinterpret_cast<char*>(align_up(reinterpret_cast<uintptr_t>(ws), 1024));
    PlanView v;
    cudaError_t e = resolve_plan(it, ro, row_idx, col, m, n, nnz, plan, &w, &v, s);
    if (e != cudaSuccess) return e;
    const bool panels = structure_aware && nnz > 0 && v.panels && dtype_ok(dt) && kd > 0 && kd % 8 == 0 &&
                        aligned16(A) && aligned16(BT);
    if (panels) {
        float* partial = reinterpret_cast<float*>(w);
        e = dt == kF16 ? run_sddmm_panels<__half>(ro, A, BT, out, partial, kd, v, s)
                       : run_sddmm_panels<__nv_bfloat16>(ro, A, BT, out, partial, kd, v, s);
        if (e != cudaSuccess) return e;
    }
    return launch_sddmm_general(dt, it, ro, row_idx, col, m, n, kd, A, BT, out, v.bins_sddmm(),
                                panels ? v.dense : nullptr, s);
}

}  // namespace spops
