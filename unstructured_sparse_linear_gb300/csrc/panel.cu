// Structure-aware path: dense panels of the CSR matrix on the tcgen05 tensor cores.
//
// spops README ("Sparse Operations (spops)"), section "Sampled Dense-Dense Matrix
// Multiplication (SDDMM)": besides the general kernel, SDDMM has a structure-aware kernel
// for the masks seen in RoSA, whose non-zeros cluster in a small subset of rows and
// columns. The mask plan (plan.cu) groups row_idx positions into panels of 128 rows and
// marks a panel dense when its entries fill its 128 x |U| tile well (U = the union of the
// panel's columns). Here:
//   * SDDMM: D = A[panel rows, :] * BT[U, :]^T per (panel, 128-column tile of U) on tcgen05
//     (fp16/bf16 operands, fp32 accumulators in tensor memory). K is split over the CTAs of
//     a thread-block cluster (up to 8); their fp32 partial tiles are added in rank order
//     through distributed shared memory, so results are deterministic and no partial sums
//     go to global memory. The epilogue reads each row's entries of the tile (contiguous,
//     located by the plan's tile starts) out of D.
//   * SpMM: each dense panel's values are written into a 128 x |U| image already in the
//     UMMA K-major 128-byte-swizzled layout; C[panel rows, 128-column tile] =
//     image * B[U, tile] on tcgen05, with B's rows gathered into an MN-major swizzled tile.
//   * the other rows run through the general row kernels, which skip dense panels.
// With few units, operands are gathered row by row with 16-byte cp.async copies into a
// 3-stage shared memory ring (two CTAs per SM, so two units' latency chains overlap); one
// thread issues the MMAs and commits them to per-stage mbarriers, whose completion frees the
// stage for the next copy. With many SpMM units, a warp-specialized kernel (one CTA per SM:
// producer warps with bulk and TMA tile copies, an MMA thread, epilogue warps on two TMEM
// accumulators) overlaps consecutive units. Every mbarrier wait is bounded in time.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>
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
constexpr int kMaxCluster = 8;  // SDDMM: CTAs (K splits) per tile, the portable cluster limit
constexpr int kNarrowMax = 16;  // SpMM with at most this many columns skips the panel path
constexpr int kTileThreads = 128;

constexpr uint32_t kSdStageA = kPM * kKC * 2;                 // 16 KB
constexpr uint32_t kSdStageBytes = kSdStageA + kTileN * kKC * 2;  // A + BT tiles: 32 KB
constexpr uint32_t kSpStageA = kPM * kKC * 2;                 // 16 KB
constexpr uint32_t kSpStageB = kSpNT * kKC * 2;               // 16 KB
constexpr uint32_t kSpStageBytes = kSpStageA + kSpStageB;     // 32 KB
constexpr uint32_t kSpCRowBytes = kSpNT * 2 + 16;              // staged C row (16-bit dtypes), padded
static_assert(kPM * kSpCRowBytes <= kStages * kSpStageBytes, "C tile must fit in the operand ring");
constexpr uint32_t kSdSmem = kStages * kSdStageBytes + 1024;
// Receive slots (C * ceil(128 / C) rows of 132 floats, largest at C = 7) and row words.
static_assert(133 * (kTileN + 4) * 4 + kPM * (kTileN / 4 + 1) * 4 <= kStages * kSdStageBytes,
              "SDDMM receive slots and row words must fit in the operand ring");
constexpr uint32_t kSpSmem = kStages * kSpStageBytes + 1024;

bool dtype_ok(int dt) { return dt == kF16 || dt == kBF16; }

// ------------------------------------------------------------------ SDDMM dense panels

// Epilogue data of tile t for one row of a panel whose rows each hold all of U in column
// order (the direct panels: rows of one length |U| = nU, row i starting at entry i * nU): the
// row's first entry of the tile, its entry count there and the mask of the U positions it
// holds, without the plan's per-entry tables.
__device__ __forceinline__ void direct_tile(int row, int nU, int t, int32_t& kb, int& cnt, uint4& mask) {
    kb = row * nU + t * kTileN;  // row * nU <= nnz < 2^31
    cnt = min(kTileN, nU - t * kTileN);
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int b = cnt - 32 * q;
        w[q] = b >= 32 ? 0xffffffffu : (b > 0 ? (1u << b) - 1u : 0u);
    }
    mask = make_uint4(w[0], w[1], w[2], w[3]);
}

// A cluster of C CTAs computes one tile (panel p, 128 columns t of U): CTA rank r multiplies
// K chunks [r * per, (r + 1) * per) into its tensor memory. Rows are split among the ranks
// (rank o finishes rows [o * 128 / C, ...)); after a cluster barrier (every ring is idle),
// each CTA stores its fp32 partial rows into a receive slot of the finishing rank through
// distributed shared memory; after a second barrier, each rank adds its rows' slots in rank
// order (so the result is deterministic) and writes the sampled entries. C = 1 is an
// ordinary launch.
template <typename T, int NT>
__global__ void __launch_bounds__(NT, 2)
sddmm_panel_kernel(const T* __restrict__ A, const T* __restrict__ BT, T* __restrict__ out, int32_t kd, PlanView v,
                   uint32_t idesc, int* err) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t mma_bar[kStages];
    __shared__ uint32_t tmem_base_sh;
    __shared__ int32_t s_rows[kPM];
    __shared__ int32_t s_u[kTileN];
    __shared__ int32_t s_kb[kPM], s_cnt[kPM];
    __shared__ uint4 s_mask[kPM];
    uint8_t* smem = reinterpret_cast<uint8_t*>(align_up(reinterpret_cast<uintptr_t>(smem_raw), 1024));
    const uint32_t sbase = smem_u32(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    pdl_trigger();

    if (warp == 0) tc::tmem_alloc(smem_u32(&tmem_base_sh), kTileN);
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(smem_u32(&mma_bar[s]), 1);
        fence_mbar_init();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = tmem_base_sh;
    pdl_wait();  // the plan and the operands come from earlier kernels

    // With at least one tile per two CTAs, K is not split: every CTA takes whole tiles on its
    // own and the cluster barriers become CTA barriers (the choice is the same on every CTA).
    const int nitems = v.counts()[kCntTiles];
    const bool split = (int)cluster_size() > 1 && 2 * nitems < (int)gridDim.x;
    const int C = split ? (int)cluster_size() : 1;
    const int crank = split ? (int)cluster_rank() : 0;
    const int cid = blockIdx.x / C, ncl = gridDim.x / C;
    const int nkc = (kd + kKC - 1) / kKC;
    const int per = (nkc + C - 1) / C;
    const int S = (nkc + per - 1) / per;  // ranks that own at least one chunk
    const int kc0 = crank * per;
    const int nk = crank < S ? min(nkc, kc0 + per) - kc0 : 0;
    const int rows_per = (kPM + C - 1) / C;
    const int r0 = min(kPM, crank * rows_per), r1 = min(kPM, r0 + rows_per);

    constexpr int kTS = kTileN + 4;      // receive slot row stride (floats)
    constexpr int kMS = kTileN / 4 + 1;  // per-row word stride
    float* recv = reinterpret_cast<float*>(smem);  // [C][rows_per][kTS] in the operand ring
    uint32_t* meta = reinterpret_cast<uint32_t*>(recv + (size_t)C * rows_per * kTS);
    uint32_t g = 0;  // chunks consumed so far by this CTA: stage = g % kStages
    bool failed = false;

    // The trip count is the same on every CTA of a cluster, and no CTA leaves the loop early
    // (a failed wait only skips work), so the cluster barriers always match.
    for (int it = cid; it < nitems; it += ncl) {
        const int item = v.items[it];
        const int p = item >> 8, t = item & 255;
        const int2 dsc = *reinterpret_cast<const int2*>(&v.desc[p]);  // dense bits, |U|
        const int nU = dsc.y;
        const bool direct = (dsc.x & 4) != 0;
        const int u0 = t * kTileN;
        const int ncols = min(kTileN, nU - u0);
        // One round of independent loads (all indexed by panel position, not by row): the
        // gather's row and column lists and the epilogue's per-row tile start, count and
        // column mask. Values of padding positions are loaded but never used.
        if (tid < kPM) {
            const size_t prow_at = (size_t)p * kPM + tid;
            const int my_row = v.prow[prow_at];
            const int u = v.ulist[(size_t)p * kUList + u0 + tid];
            int32_t kb;
            int cnt;
            uint4 mk;
            if (direct) {
                direct_tile(my_row, nU, t, kb, cnt, mk);
            } else {
                const int32_t* ts = v.ts + prow_at * (kTiles + 1);
                kb = ts[t];
                cnt = ts[t + 1] - kb;
                mk = *reinterpret_cast<const uint4*>(v.tmask + prow_at * (kUCap / 32) + t * (kTileN / 32));
            }
            s_rows[tid] = my_row;
            s_u[tid] = tid < ncols ? u : -1;
            s_kb[tid] = kb;
            s_cnt[tid] = my_row >= 0 ? cnt : 0;
            s_mask[tid] = mk;
        }
        __syncthreads();

        auto load = [&](int j, uint32_t gs) {
            const uint32_t st = sbase + (gs % kStages) * kSdStageBytes;
            const int k0 = (kc0 + j) * kKC;
#pragma unroll
            for (int q = 0; q < kPM * 8 / NT; ++q) {
                const int c = tid + NT * q;
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

        if (nk > 0 && !failed) {
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
            const uint32_t gl = g + nk - 1;
            if (!mbar_wait(smem_u32(&mma_bar[gl % kStages]), (gl / kStages) & 1u, err)) failed = true;
            g += nk;
        }
        tc::cp_async_wait<0>();
        failed = __syncthreads_or(failed);
        tc::fence_after_sync();

        // The ring is free on every CTA of the cluster once all have passed this barrier; the
        // receive slots below live in it.
        tc::fence_before_sync();
        if (split) cluster_sync();
        else __syncthreads();
        tc::fence_after_sync();

        // Partial tile: with NT / 128 threads per row, thread tid owns its share of TMEM lane
        // tid % 128 (panel row tid % 128; a warp reads the lane quarter it may access) and
        // sends those fp32 sums to the CTA that finishes the row (rank row / rows_per), into
        // the slot of this CTA's rank (row stride 132 floats: the 16-byte stores of eight
        // consecutive rows hit distinct banks).
        // (tcgen05.ld is warp-collective: the whole warp loads, only rows with entries send.)
        if (nk > 0 && !failed) {
            constexpr int kCols = kTileN * kPM / NT;  // TMEM columns per thread
            const int row = tid & (kPM - 1), half = tid / kPM;
            const int owner = row / rows_per;
            const bool send = s_cnt[row] > 0;
            const uint32_t dst =
                smem_u32(recv + ((size_t)crank * rows_per + (row - owner * rows_per)) * kTS + half * kCols);
            const uint32_t lane_addr = tmem + ((uint32_t)((warp & 3) * 32) << 16) + half * kCols;
            const uint32_t rdst = C == 1 ? dst : cluster_map(dst, owner);
#pragma unroll
            for (int c = 0; c < kCols / 32; ++c) {
                float x[32];
                tc::tmem_ld32(lane_addr + c * 32, x);
                if (send) {
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const float4 y = make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
                        if (C == 1) st_shared_f4(rdst + (c * 32 + q * 4) * 4, y);
                        else st_cluster_f4(rdst + (c * 32 + q * 4) * 4, y);
                    }
                }
            }
        }
        // For each group of 4 columns of row tid: the group's bits of the row's column mask
        // and the rank of its first entry among the row's entries of the tile (entries and U
        // are both in column order).
        if (tid < kPM && tid >= r0 && tid < r1) {
            const uint4 m = s_mask[tid];
            const uint32_t w[4] = {m.x, m.y, m.z, m.w};
            uint32_t run = 0;
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint32_t b = (w[c] >> (4 * j)) & 0xFu;
                    meta[(tid - r0) * kMS + c * 8 + j] = run | (b << 8);
                    run += __popc(b);
                }
        }
        tc::fence_before_sync();
        if (split) cluster_sync();  // every rank's rows have arrived
        else __syncthreads();

        // Rows [r0, r1): a warp per row; lane l adds columns 4l .. 4l+3 of the S slots in rank
        // order and writes the sampled values to ts[t] + rank.
        if (!failed) {
#pragma unroll 2
            for (int r = r0 + warp; r < r1; r += NT / 32) {
                if (s_cnt[r] == 0) continue;  // uniform across the warp
                const float4* slot = reinterpret_cast<const float4*>(recv + (size_t)(r - r0) * kTS) + lane;
                const size_t slot_step = (size_t)rows_per * kTS / 4;
                float4 x = slot[0];
                for (int q0 = 1; q0 < S; q0 += 4) {
                    float4 y[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        if (q0 + q < S) y[q] = slot[(q0 + q) * slot_step];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        if (q0 + q < S) {
                            x.x += y[q].x;
                            x.y += y[q].y;
                            x.z += y[q].z;
                            x.w += y[q].w;
                        }
                    }
                }
                const uint32_t mt = meta[(r - r0) * kMS + lane];
                const uint32_t bits = mt >> 8;
                T* o = out + (int64_t)s_kb[r] + (int)(mt & 0xFFu);
                const int k1 = bits & 1u, k2 = k1 + ((bits >> 1) & 1u), k3 = k2 + ((bits >> 2) & 1u);
                if (bits & 1u) o[0] = Elt<T>::from_f(x.x);
                if (bits & 2u) o[k1] = Elt<T>::from_f(x.y);
                if (bits & 4u) o[k2] = Elt<T>::from_f(x.z);
                if (bits & 8u) o[k3] = Elt<T>::from_f(x.w);
            }
        }
        __syncthreads();  // the shared arrays and the receive slots are rewritten by the next tile
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, kTileN);
}

// Grouped SDDMM for masks with many dense tiles: one item is a group of up to kGroupTiles
// consecutive 128-column tiles of one panel, all accumulated at once in tensor memory
// (kGroupTiles x 128 = 512 columns), so each 128 x 64 chunk of A rows is loaded once per
// group instead of once per tile. A stage holds the A chunk and the group's BT chunks
// (16 KB each); the ring takes as many stages (up to 4) as fit kGrpRing bytes.
// Roles: warp 0 lane 0 issues the MMAs and does nothing else (tile pairs as one N = 256
// MMA, so A is read from shared memory once per 256 columns; an odd last tile as N = 128).
// While the tensor core runs, shared-memory loads of other warps wait behind its operand
// reads, so the producers keep the chunk loop free of them. When each 64-row half of the
// panel is 64 consecutive rows of A and each 64-row half of a tile's U list 64 consecutive
// rows of BT, one thread per stage (lane 0 of warps 1 .. S) loads that stage's chunks as 2-D
// TMA boxes (128-byte swizzle, straight into the UMMA K-major layout) with one expect-tx
// arrive each, from box coordinates held in registers (several TMA issuers keep more loads
// in flight than one); otherwise warps 1 .. 7 gather every 16-byte piece with
// cp.async and each thread arrives once its pieces have landed (the stage barriers are
// re-armed per item for the producer count of its mode). The MMA issuer commits each stage
// to its empty barrier, which the producers wait on before refilling it, and the item's
// last MMAs to an accumulator barrier that every thread waits on before the epilogue. One
// CTA per SM. When the items fill less than the grid, K is split over the CTAs of a
// thread-block cluster and the partial tiles are added in rank order through distributed
// shared memory, one tile after the other, as in sddmm_panel_kernel.
constexpr int kGrpThreads = 256;
constexpr uint32_t kGrpChunk = kPM * kKC * 2;  // one 128 x 64 operand chunk: 16 KB
constexpr uint32_t kGrpRing = 12 * kGrpChunk;  // 192 KB of stages
constexpr int kGrpMaxStages = 4;
constexpr int kGrpProducers = kGrpThreads - 32;  // warps 1.. gather when a chunk is not all TMA boxes
constexpr uint32_t kGrpSmem = kGrpRing + 1024;
static_assert(2 * (kPM / 2) * (kTileN + 4) * 4 + (kPM / 2) * (kTileN / 4 + 1) * 4 <= kGrpRing,
              "grouped SDDMM receive slots (two ranks) fit in the ring");

__device__ __forceinline__ void cp_async_mbar_arrive(uint32_t bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// 2-D TMA tile load of the box at (x = column, y = row) into shared memory, completing on bar.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// L2 prefetch of the 2-D box at (x = column, y = row): no shared memory, no completion.
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* map, int x, int y) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y)
                 : "memory");
}

// 2-D TMA tile store of the box at (x = column, y = row) from shared memory, in the calling
// thread's bulk group (callers only store boxes that lie inside the tensor).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int x, int y, uint32_t src) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(src)
                 : "memory");
}

template <typename T>
__global__ void __launch_bounds__(kGrpThreads, 1)
sddmm_group_kernel(const T* __restrict__ A, const T* __restrict__ BT, T* __restrict__ out, int32_t kd, PlanView v,
                   uint32_t idesc, int* err, const __grid_constant__ CUtensorMap tmap_a,
                   const __grid_constant__ CUtensorMap tmap_bt, int use_tma) {
    constexpr int NT = kGrpThreads;
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kGrpMaxStages], empty_bar[kGrpMaxStages], acc_bar;
    __shared__ uint32_t tmem_base_sh;
    __shared__ int32_t s_rows[kPM];
    __shared__ int32_t s_u[kGroupTiles * kTileN];
    __shared__ int32_t s_kb[kPM], s_cnt[kPM];
    __shared__ uint4 s_mask[kPM];
    __shared__ int s_box[2 + 2 * kGroupTiles];  // first row of each 64-row TMA box of the item, -1: gather
    uint8_t* smem = reinterpret_cast<uint8_t*>(align_up(reinterpret_cast<uintptr_t>(smem_raw), 1024));
    const uint32_t sbase = smem_u32(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    pdl_trigger();

    if (warp == 0) tc::tmem_alloc(smem_u32(&tmem_base_sh), kGroupTiles * kTileN);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = tmem_base_sh;
    const uint32_t idesc_n256 = idesc + ((uint32_t)((2 * kTileN - kTileN) >> 3) << 17);  // the N field
    pdl_wait();  // the plan and the operands come from earlier kernels

    const int nitems = v.counts()[kCntGroups];
    const int csize = (int)cluster_size();
    const bool split = csize > 1 && nitems * csize <= (int)gridDim.x;  // the same on every CTA
    const int C = split ? csize : 1;
    const int crank = split ? (int)cluster_rank() : 0;
    const int cid = blockIdx.x / C, ncl = gridDim.x / C;
    const int nkc = (kd + kKC - 1) / kKC;
    const int per = (nkc + C - 1) / C;
    const int S_ranks = (nkc + per - 1) / per;  // ranks that own at least one chunk
    const int kc0 = crank * per;
    const int nk = crank < S_ranks ? min(nkc, kc0 + per) - kc0 : 0;
    const int rows_per = (kPM + C - 1) / C;
    const int r0 = min(kPM, crank * rows_per), r1 = min(kPM, r0 + rows_per);

    constexpr int kTS = kTileN + 4;      // receive slot row stride (floats)
    constexpr int kMS = kTileN / 4 + 1;  // per-row word stride
    float* recv = reinterpret_cast<float*>(smem);
    uint32_t* meta = reinterpret_cast<uint32_t*>(recv + (size_t)C * rows_per * kTS);
    bool failed = false;

    for (int it = cid; it < nitems; it += ncl) {
        const int item = v.gitems[it];
        const int p = item >> 8, grp = item & 255;
        const int2 dsc = *reinterpret_cast<const int2*>(&v.desc[p]);  // dense bits, |U|
        const int nU = dsc.y;
        const bool direct = (dsc.x & 4) != 0;
        const int t0 = grp * kGroupTiles;
        const int nt = min(kGroupTiles, (nU + kTileN - 1) / kTileN - t0);  // tiles in this group
        const uint32_t stage_bytes = (uint32_t)(1 + nt) * kGrpChunk;
        const int S = min(kGrpMaxStages, (int)(kGrpRing / stage_bytes));
        if (tid < kPM) s_rows[tid] = v.prow[(size_t)p * kPM + tid];
        for (int x = tid; x < nt * kTileN; x += NT) {
            const int u = t0 * kTileN + x;
            s_u[x] = u < nU ? v.ulist[(size_t)p * kUList + u] : -1;
        }
        __syncthreads();
        // 64-row TMA boxes: each half of the panel's A rows when its 64 rows are consecutive
        // rows of A; each 64-row half of a tile's BT rows when its 64 U columns are consecutive
        // (U is sorted and distinct)
        const bool a_lo = __syncthreads_and(tid >= kPM / 2 || s_rows[tid] == s_rows[0] + tid) != 0;
        const bool a_hi = __syncthreads_and(tid >= kPM / 2 || s_rows[kPM / 2 + tid] == s_rows[kPM / 2] + tid) != 0;
        if (tid < 2 + 2 * nt) {
            int first = -1;
            if (tid < 2) {
                const int r = s_rows[tid * (kPM / 2)];
                first = (tid == 0 ? a_lo : a_hi) && r >= 0 ? r : -1;
            } else {
                const int h = tid - 2;  // half h of the group's BT rows: positions 64 h .. 64 h + 63
                const int lo = s_u[h * 64], hi = s_u[h * 64 + 63];
                first = lo >= 0 && hi >= 0 && hi - lo == 63 ? lo : -1;
            }
            s_box[tid] = use_tma ? first : -1;
        }
        __syncthreads();

        // The whole chunk by TMA (every box a run) or the whole chunk by gathers; the stage
        // barriers are re-armed for the item's producer count (all of them are idle here).
        bool tma_all = true;
        for (int b = 0; b < 2 + 2 * nt; ++b) tma_all = tma_all && s_box[b] >= 0;
        if (tid == 0) {
            for (int st = 0; st < kGrpMaxStages; ++st) {
                mbar_inval(smem_u32(&full_bar[st]));
                mbar_inval(smem_u32(&empty_bar[st]));
                mbar_init(smem_u32(&full_bar[st]), tma_all ? 1 : kGrpProducers);
                mbar_init(smem_u32(&empty_bar[st]), 1);  // the MMA commit
            }
            mbar_inval(smem_u32(&acc_bar));
            mbar_init(smem_u32(&acc_bar), 1);
            fence_mbar_init();
        }
        __syncthreads();

        if (nk > 0 && !failed) {
            if (warp == 0) {
                // ---- MMA issuer (does nothing else, so the tensor pipe is fed without gaps):
                // tile pairs as one N = 256 MMA (A read once per 256 columns), an odd last
                // tile as N = 128
                if (lane == 0) {
                    uint32_t full_ph = 0;
                    for (int j = 0; j < nk; ++j) {
                        const int st = j % S;
                        if (!mbar_wait(smem_u32(&full_bar[st]), (full_ph >> st) & 1u, err)) {
                            failed = true;
                            break;
                        }
                        full_ph ^= 1u << st;
                        fence_proxy_async_smem();  // gathered data (generic proxy) before the tensor core reads it
                        tc::fence_after_sync();
                        const uint32_t sa = sbase + (uint32_t)st * stage_bytes;
                        for (int i = 0; i < nt; i += 2) {
                            const uint32_t id = i + 1 < nt ? idesc_n256 : idesc;
#pragma unroll
                            for (int kk = 0; kk < kKC / 16; ++kk) {
                                const uint64_t ad = tc::smem_desc_sw128(sa + kk * 32, 16, 1024);
                                const uint64_t bd =
                                    tc::smem_desc_sw128(sa + (uint32_t)(1 + i) * kGrpChunk + kk * 32, 16, 1024);
                                tc::mma_f16(tmem + (uint32_t)(i * kTileN), ad, bd, id, (j > 0 || kk > 0) ? 1u : 0u);
                            }
                        }
                        tc::mma_commit(smem_u32(&empty_bar[st]));
                    }
                    // The producers waited for the empty completions of chunks 0 .. nk - S - 1;
                    // wait here for the last ones (completion c of a stage's barrier is chunk
                    // st + c S), so that no arrive is pending on any barrier when the next item
                    // re-arms them. Then the accumulator barrier, which completes at once.
                    if (!failed)
                        for (int j = max(0, nk - S); j < nk; ++j)
                            if (!mbar_wait(smem_u32(&empty_bar[j % S]), (uint32_t)(j / S) & 1u, err)) failed = true;
                    tc::mma_commit(smem_u32(&acc_bar));
                }
                __syncwarp();
            } else if (tma_all) {
                // ---- one producer thread per stage (lane 0 of warps 1 .. S): chunk j is loaded
                // by the thread of stage j mod S, whole by TMA boxes with the coordinates in
                // registers; several issuers keep more of the SM's loads in flight, and each
                // waits only for the consumption of its own stage's previous chunk. With each
                // chunk's loads it asks L2 for the boxes of its next chunk (j + S), which that
                // chunk's loads then find closer: 61 -> 57 us on the butterfly layer.
                if (lane == 0 && warp >= 1 && warp <= S) {
                    const int st = warp - 1;
                    int by[2 + 2 * kGroupTiles];
#pragma unroll
                    for (int b = 0; b < 2 + 2 * kGroupTiles; ++b) by[b] = b < 2 + 2 * nt ? s_box[b] : 0;
                    const uint32_t sa = sbase + (uint32_t)st * stage_bytes;
                    const uint32_t fb = smem_u32(&full_bar[st]);
                    uint32_t empty_ph = 0;
                    for (int j = st; j < nk; j += S) {
                        if (j >= S) {  // the stage's previous chunk (j - S) has been consumed
                            if (!mbar_wait(smem_u32(&empty_bar[st]), empty_ph, err)) {
                                failed = true;
                                break;
                            }
                            empty_ph ^= 1u;
                        }
                        const int k0 = (kc0 + j) * kKC;
                        mbar_arrive_expect_tx(fb, stage_bytes);
                        tma_load_2d(sa, &tmap_a, k0, by[0], fb);
                        tma_load_2d(sa + kGrpChunk / 2, &tmap_a, k0, by[1], fb);
#pragma unroll
                        for (int h = 0; h < 2 * kGroupTiles; ++h)
                            if (h < 2 * nt)
                                tma_load_2d(sa + (uint32_t)(1 + (h >> 1)) * kGrpChunk + (uint32_t)(h & 1) * (kGrpChunk / 2),
                                            &tmap_bt, k0, by[2 + h], fb);
                        if (j + S < nk) {
                            const int kp = k0 + S * kKC;
                            tma_prefetch_2d(&tmap_a, kp, by[0]);
                            tma_prefetch_2d(&tmap_a, kp, by[1]);
#pragma unroll
                            for (int h = 0; h < 2 * kGroupTiles; ++h)
                                if (h < 2 * nt) tma_prefetch_2d(&tmap_bt, kp, by[2 + h]);
                        }
                    }
                }
            } else {
                // ---- producer warps 1..7: every 16-byte piece gathered with cp.async; each
                // thread arrives on the stage's full barrier once its pieces have landed
                const int pt = tid - 32;
                uint32_t empty_ph = 0;
                for (int j = 0; j < nk; ++j) {
                    const int st = j % S;
                    if (j >= S) {
                        if (!mbar_wait(smem_u32(&empty_bar[st]), (empty_ph >> st) & 1u, err)) {
                            failed = true;
                            break;
                        }
                        empty_ph ^= 1u << st;
                    }
                    const uint32_t sa = sbase + (uint32_t)st * stage_bytes;
                    const int k0 = (kc0 + j) * kKC;
                    for (int c = pt; c < (1 + nt) * kPM * 8; c += kGrpProducers) {
                        const int o = c / (kPM * 8), rc = c % (kPM * 8);
                        const int row = rc >> 3, kch = rc & 7;
                        const int kk = k0 + kch * 8;
                        const int r = o == 0 ? s_rows[row] : s_u[(o - 1) * kTileN + row];
                        const T* base = o == 0 ? A : BT;
                        const bool ok = r >= 0 && kk < kd;
                        tc::cp_async16(sa + (uint32_t)o * kGrpChunk + tc::sw128_off(row, kch),
                                       ok ? (const void*)(base + (int64_t)r * kd + kk) : (const void*)base, ok ? 16 : 0);
                    }
                    cp_async_mbar_arrive(smem_u32(&full_bar[st]));
                }
            }
            // the accumulator is final once the MMA issuer's last commit has arrived
            if (!mbar_wait(smem_u32(&acc_bar), 0, err)) failed = true;
        }
        tc::cp_async_commit();  // (gathers are tracked by their mbarrier arrives; none is left in flight)
        tc::cp_async_wait<0>();
        failed = __syncthreads_or(failed);
        tc::fence_after_sync();
        for (int i = 0; i < nt; ++i) {
            const int t = t0 + i;
            // the epilogue's per-row data for tile t
            if (tid < kPM) {
                const size_t prow_at = (size_t)p * kPM + tid;
                int32_t kb;
                int cnt;
                uint4 mk;
                if (direct) {
                    direct_tile(s_rows[tid], nU, t, kb, cnt, mk);
                } else {
                    const int32_t* ts = v.ts + prow_at * (kTiles + 1);
                    kb = ts[t];
                    cnt = ts[t + 1] - kb;
                    mk = *reinterpret_cast<const uint4*>(v.tmask + prow_at * (kUCap / 32) + t * (kTileN / 32));
                }
                s_kb[tid] = kb;
                s_cnt[tid] = s_rows[tid] >= 0 ? cnt : 0;
                s_mask[tid] = mk;
            }
            // the ring (and the previous tile's receive slots) is free on every CTA of the
            // cluster once all have passed this barrier
            tc::fence_before_sync();
            if (split) cluster_sync();
            else __syncthreads();
            tc::fence_after_sync();
            if (nk > 0 && !failed) {
                constexpr int kCols = kTileN * kPM / NT;  // TMEM columns per thread
                const int row = tid & (kPM - 1), half = tid / kPM;
                const int owner = row / rows_per;
                const bool send = s_cnt[row] > 0;
                const uint32_t dst =
                    smem_u32(recv + ((size_t)crank * rows_per + (row - owner * rows_per)) * kTS + half * kCols);
                const uint32_t lane_addr =
                    tmem + ((uint32_t)((warp & 3) * 32) << 16) + (uint32_t)(i * kTileN) + half * kCols;
                const uint32_t rdst = C == 1 ? dst : cluster_map(dst, owner);
#pragma unroll
                for (int c = 0; c < kCols / 32; ++c) {
                    float x[32];
                    tc::tmem_ld32(lane_addr + c * 32, x);
                    if (send) {
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            const float4 y = make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
                            if (C == 1) st_shared_f4(rdst + (c * 32 + q * 4) * 4, y);
                            else st_cluster_f4(rdst + (c * 32 + q * 4) * 4, y);
                        }
                    }
                }
            }
            if (tid < kPM && tid >= r0 && tid < r1) {
                const uint4 m = s_mask[tid];
                const uint32_t w[4] = {m.x, m.y, m.z, m.w};
                uint32_t run = 0;
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const uint32_t b = (w[c] >> (4 * j)) & 0xFu;
                        meta[(tid - r0) * kMS + c * 8 + j] = run | (b << 8);
                        run += __popc(b);
                    }
            }
            tc::fence_before_sync();
            if (split) cluster_sync();  // every rank's rows have arrived
            else __syncthreads();
            if (!failed) {
#pragma unroll 2
                for (int r = r0 + warp; r < r1; r += NT / 32) {
                    if (s_cnt[r] == 0) continue;  // uniform across the warp
                    const float4* slot = reinterpret_cast<const float4*>(recv + (size_t)(r - r0) * kTS) + lane;
                    const size_t slot_step = (size_t)rows_per * kTS / 4;
                    float4 x = slot[0];
                    for (int q = 1; q < S_ranks; ++q) {
                        const float4 y = slot[q * slot_step];
                        x.x += y.x;
                        x.y += y.y;
                        x.z += y.z;
                        x.w += y.w;
                    }
                    const uint32_t mt = meta[(r - r0) * kMS + lane];
                    const uint32_t bits = mt >> 8;
                    T* o = out + (int64_t)s_kb[r] + (int)(mt & 0xFFu);
                    const int k1 = bits & 1u, k2 = k1 + ((bits >> 1) & 1u), k3 = k2 + ((bits >> 2) & 1u);
                    if (bits & 1u) o[0] = Elt<T>::from_f(x.x);
                    if (bits & 2u) o[k1] = Elt<T>::from_f(x.y);
                    if (bits & 4u) o[k2] = Elt<T>::from_f(x.z);
                    if (bits & 8u) o[k3] = Elt<T>::from_f(x.w);
                }
            }
            __syncthreads();  // s_kb / s_cnt / s_mask and the slots are rewritten for the next tile
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, kGroupTiles * kTileN);
}

// ------------------------------------------------------------------ SpMM dense panels

// The 8 image rows of one row group: zeros, then the group's values at their U position,
// written out as whole 128-byte-swizzled K-major rows (16-byte stores). The staging rows are
// ucap = min(kUList, K rounded up to 64) values long (U is a set of the K columns), so that
// narrow matrices leave room for more CTAs per SM.
inline uint32_t densify_smem_bytes(int32_t K, size_t elt) {
    const int32_t ucap = (int32_t)min64(kUList, ((int64_t)K + kKC - 1) / kKC * kKC);
    return (uint32_t)(kGroupRows * (size_t)ucap * elt);
}

template <typename T>
__global__ void __launch_bounds__(256) densify_kernel(const T* __restrict__ vals, const int32_t* __restrict__ ro,
                                                     T* __restrict__ img_base, PlanView v, int ucap,
                                                     int skip_direct) {
    extern __shared__ __align__(16) uint8_t densify_smem[];
    T* stage = reinterpret_cast<T*>(densify_smem);  // [kGroupRows][ucap]
    pdl_trigger();
    pdl_wait();
    const int p = blockIdx.x / kGroups, grp = blockIdx.x % kGroups;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // the panel's image slot and size, and the warp's row, are independent loads: issued together
    const int slot = v.img_slot[p];
    const int2 d = *reinterpret_cast<const int2*>(&v.desc[p]);  // dense bits, |U|
    const int nU = d.y;
    const int i = v.prow[p * kPM + grp * kGroupRows + warp];
    if (slot < 0) return;                        // no image for this panel
    const bool direct = (d.x & 4) != 0;  // row i holds all of U in order: entry k sits at k - ro[i]
    if (skip_direct && direct) return;          // the SpMM pipeline reads these values directly
    const int upad = (nU + kKC - 1) / kKC * kKC;  // <= ucap
    uint4* st4 = reinterpret_cast<uint4*>(stage);
    const int row_vec = ucap * (int)sizeof(T) / 16;
    for (int x = tid; x < kGroupRows * row_vec; x += 256) {
        if ((x % row_vec) * 16 < upad * (int)sizeof(T)) st4[x] = make_uint4(0, 0, 0, 0);
    }
    __syncthreads();
    static_assert(kGroupRows == 8, "one row per warp");
    {
        const int lr = warp;
        const int32_t k0 = i >= 0 ? ro[i] : 0, k1 = i >= 0 ? ro[i + 1] : 0;
        // 8 (position, value) pairs per lane loaded before any is stored
        constexpr int kB = 8;
        for (int32_t kb = k0; kb < k1; kb += 32 * kB) {
            int u[kB];
            T x[kB];
#pragma unroll
            for (int j = 0; j < kB; ++j) {
                const int32_t k = kb + j * 32 + lane;
                u[j] = k < k1 ? (direct ? (int)(k - k0) : (int)v.upos[k]) : -1;
                x[j] = k < k1 ? vals[k] : T();
            }
#pragma unroll
            for (int j = 0; j < kB; ++j)
                if (u[j] >= 0) stage[lr * ucap + u[j]] = x[j];
        }
    }
    __syncthreads();
    T* img = img_base + slot;
    const int chunks = upad / 8;  // 16-byte chunks per image row
    for (int x = tid; x < kGroupRows * chunks; x += 256) {
        const int lr = x / chunks, c = x % chunks;
        const int r = grp * kGroupRows + lr;           // panel row = image row
        const int kc = c / 8, w = c % 8;               // 64-column chunk, 16-byte piece in it
        uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<char*>(img + (size_t)kc * kPM * kKC) +
                                              tc::sw128_off(r, w));
        *dst = reinterpret_cast<const uint4*>(stage + lr * ucap)[c];
    }
}

template <typename T, int NT>
__global__ void __launch_bounds__(NT, 2)
spmm_panel_kernel(const T* __restrict__ B, T* __restrict__ C, const T* __restrict__ img_base, int32_t N, PlanView v,
                  uint32_t idesc, int* err) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t mma_bar[kStages];
    __shared__ uint32_t tmem_base_sh;
    __shared__ uint16_t s_u[kUList];  // the panel's U list (columns < 65536); positions >= |U| unused
    uint8_t* smem = reinterpret_cast<uint8_t*>(align_up(reinterpret_cast<uintptr_t>(smem_raw), 1024));
    const uint32_t sbase = smem_u32(smem);
    const int tid = threadIdx.x, warp = tid >> 5;
    pdl_trigger();

    if (warp == 0) tc::tmem_alloc(smem_u32(&tmem_base_sh), kSpNT);
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(smem_u32(&mma_bar[s]), 1);
        fence_mbar_init();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = tmem_base_sh;
    pdl_wait();  // the plan and the operands come from earlier kernels

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
        for (int x = tid; x < nU; x += NT) s_u[x] = (uint16_t)v.ulist[(size_t)p * kUList + x];
        bulk_wait_read<0>();  // the previous unit's staged C row has been read out of shared memory
        __syncthreads();

        auto load = [&](int j, uint32_t gs) {
            const uint32_t st = sbase + (gs % kStages) * kSpStageBytes;
            const char* src_a = reinterpret_cast<const char*>(img + (size_t)j * kPM * kKC);
#pragma unroll
            for (int q = 0; q < kSpStageA / 16 / NT; ++q) {
                const int c = tid + NT * q;
                tc::cp_async16(st + c * 16, src_a + c * 16, 16);
            }
            // B[U rows j*64 .. +64, n0 .. n0 + kSpNT): kSpNT / 8 sixteen-byte pieces per row
            constexpr int kPieces = kSpNT / 8;
#pragma unroll
            for (int q = 0; q < kKC * kPieces / NT; ++q) {
                const int c = tid + NT * q;
                const int kk = c / kPieces, nch = c % kPieces;
                const int ncol = n0 + nch * 8;
                const bool ok = j * kKC + kk < nU && ncol < N;
                const int u = ok ? (int)s_u[j * kKC + kk] : 0;
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

        // epilogue: with NT / 128 threads per row, thread tid converts its share of TMEM
        // lane tid % 128 (panel row tid % 128; a warp reads the lane quarter it may access)
        // to the output dtype into a shared row (stride 272 bytes: the 16-byte stores of
        // eight consecutive rows hit distinct banks); then the row's first thread sends it to
        // C[row, n0 .. n0 + 128) with one bulk async copy, drained while the next unit's
        // operands are gathered.
        constexpr int kCols = kSpNT * kPM / NT;  // TMEM columns per thread
        const int r = tid & (kPM - 1), half = tid / kPM;
        const int i = v.prow[p * kPM + r];
        const uint32_t lane_addr = tmem + ((uint32_t)((warp & 3) * 32) << 16) + half * kCols;
        const uint32_t crow = sbase + (uint32_t)r * kSpCRowBytes;
#pragma unroll
        for (int c = 0; c < kCols / 32; ++c) {
            float x[32];
            tc::tmem_ld32(lane_addr + c * 32, x);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint4 w = Elt<T>::pack(x + q * 8);
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(crow + half * kCols * 2 + (c * 4 + q) * 16),
                             "r"(w.x), "r"(w.y), "r"(w.z), "r"(w.w)
                             : "memory");
            }
        }
        fence_proxy_async_smem();
        tc::fence_before_sync();
        __syncthreads();
        if (half == 0 && i >= 0) {
            bulk_s2g(C + (int64_t)i * N + n0, crow, (uint32_t)min(kSpNT, N - n0) * (uint32_t)sizeof(T));
            bulk_commit();
        }
    }
    bulk_wait<0>();
    tc::cp_async_wait<0>();
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, kSpNT);
}

// Warp-specialized SpMM panels for masks with many units (units = dense panels x column
// tiles well above the CTA count): one CTA per SM runs a persistent pipeline in which the
// operand loads, the MMAs and the epilogue of consecutive units overlap. Each CTA takes a
// contiguous range of units, so consecutive units mostly share their panel (its U list,
// image and rows are looked up once per panel, not once per unit).
//   warps 0-3   epilogue: thread r owns TMEM lane r (panel row r); it reads the finished
//               accumulator (256 columns, in four quarters), frees it and sends each quarter
//               to C: as 2-D TMA tile stores when the panel's rows are two runs of 64
//               consecutive rows of C, else one bulk async copy per row;
//   warps 4-7   producers, one per stage of a 4-stage ring of B tiles (32 KB each): per
//               64-wide K chunk the image chunk (16 KB, contiguous, already swizzled; a panel
//               of |U| <= 256 keeps its whole image in four slots, loaded with its first
//               unit in the CTA only) and the chunk's 64 rows of B (256 columns): when they
//               are 64 consecutive rows (block-structured masks), four TMA tile loads (64 x 64
//               boxes, 128-byte swizzle) straight into the MN-major operand layout;
//               otherwise a gather (cp.async, 16 bytes each) whose completion is signalled
//               on the stage's mbarrier. The panel's U list is read from global memory;
//   warp 8      TMEM owner and MMA issuer (one thread): 4 MMAs (M = 128, N = 256, K = 16)
//               per chunk, a commit that frees the stage, and a commit per unit that hands
//               the accumulator to the epilogue.
// A B tile takes about a microsecond from issue to arrival and the MMAs of a chunk about a
// quarter of that, so the ring holds four tiles (128 KB) in flight; the image slots, the
// ring and the C staging buffers fill the 227 KB of shared memory.
// Units are 256 columns wide, so every A chunk read by the tensor core serves 256 output
// columns (shared-memory bandwidth, not the tensor pipe, bounds 128-column tiles). Two
// accumulators of 256 columns (all of TMEM) alternate between units, so the MMAs of a unit
// run while the epilogue drains the previous one. Every wait is bounded in time; a role that gives up
// stops, and the others then give up on their next wait.
constexpr int kWsNT = 256;                                     // columns of C per unit (UMMA N)
constexpr uint32_t kWsStageB = kKC * kWsNT * 2;                // 32 KB
constexpr int kWsStages = 4;
// Image chunk slots: a panel of at most kWsASlots chunks (|U| <= 256) loads its image once
// per run of its units in a CTA and keeps it (slot j = chunk j); a larger panel streams its
// chunks through slots 0 .. kWsStages - 1 beside the B stages.
constexpr int kWsASlots = 4;
constexpr uint32_t kWsAReg = kWsASlots * kSpStageA;            // 64 KB
static_assert(kWsASlots >= kWsStages, "a streamed chunk uses the slot of its stage");
constexpr int kWsEpiWarps = 4;
// One producer warp per stage: chunk g goes to stage g mod 4 and warp g mod 4, so a warp only
// ever waits for the consumption of its own previous chunk (one barrier phase back; a parity
// wait cannot alias a phase two completions behind).
constexpr int kWsProdWarps = kWsStages;
constexpr int kWsThreads = (kWsEpiWarps + kWsProdWarps + 1) * 32;
constexpr uint32_t kWsQBuf = kPM * 128;             // one 64-column quarter of a unit, 128 rows
constexpr uint32_t kWsCStage = 2 * kWsQBuf;          // C staging: two quarter buffers
constexpr uint32_t kWsCRow = 64 * 2 + 16;            // a quarter row on the per-row path, padded
static_assert(kPM * kWsCRow <= kWsCStage, "per-row staging fits the quarter buffers");
constexpr uint32_t kWsSmem = kWsAReg + kWsStages * kWsStageB + kWsCStage + 1024;
static_assert(kWsSmem <= 227 * 1024, "warp-specialized SpMM shared memory");


template <typename T>
__global__ void __launch_bounds__(kWsThreads, 1)
spmm_panel_ws_kernel(const T* __restrict__ B, T* __restrict__ C, const T* __restrict__ img_base, int32_t N,
                     PlanView v, uint32_t idesc, int* err, const __grid_constant__ CUtensorMap tmap_b, int use_tma,
                     const __grid_constant__ CUtensorMap tmap_c, int use_tma_c,
                     const __grid_constant__ CUtensorMap tmap_v, int use_tma_v) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kWsStages], empty_bar[kWsStages], tfull_bar[2], tempty_bar[2], drain_bar;
    __shared__ int s_run[kWsEpiWarps];
    __shared__ uint32_t tmem_base_sh;
    uint8_t* smem = reinterpret_cast<uint8_t*>(align_up(reinterpret_cast<uintptr_t>(smem_raw), 1024));
    const uint32_t sbase = smem_u32(smem);                 // image slots
    const uint32_t bbase = sbase + kWsAReg;                 // B stages
    const uint32_t cstage = bbase + kWsStages * kWsStageB;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    pdl_trigger();

    if (warp == kWsEpiWarps + kWsProdWarps) tc::tmem_alloc(smem_u32(&tmem_base_sh), 2 * kWsNT);
    if (tid == 0) {
        for (int i = 0; i < kWsStages; ++i) {
            mbar_init(smem_u32(&full_bar[i]), 1);  // the owning producer warp's single arrive
            mbar_init(smem_u32(&empty_bar[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&tfull_bar[i]), 1);
            mbar_init(smem_u32(&tempty_bar[i]), kWsEpiWarps);
        }
        mbar_init(smem_u32(&drain_bar), 1);
        fence_mbar_init();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = tmem_base_sh;
    pdl_wait();  // the plan, the images and B come from earlier kernels

    const int D = v.counts()[kCntDenseSp];
    const int ntn = (N + kWsNT - 1) / kWsNT;
    const int64_t units = (int64_t)D * ntn;
    const int64_t per = (units + gridDim.x - 1) / gridDim.x;
    const int64_t u_begin = min64(units, (int64_t)blockIdx.x * per), u_end = min64(units, u_begin + per);

    if (warp < kWsEpiWarps) {
        // ---------------- epilogue
        // A unit leaves in 64-column quarters through the staging area, in one of two ways.
        // When the panel's rows are two runs of 64 consecutive rows of C and the unit lies
        // inside C: a 128-byte-swizzled 128 x 64 copy in one of two 16 KB buffers
        // (alternating, so a quarter is written while the previous one is stored) and two
        // 2-D TMA tile stores of 64 x 64 boxes issued by thread 0. Otherwise one shared row
        // per thread and one bulk copy per row. The epilogue warps meet at named barrier 1
        // before a buffer is rewritten and before the tile stores; every decision that leads
        // to a barrier is taken by all of them (a barrier-reduced AND for the accumulator waits).
        const int r = tid;  // panel row = TMEM lane
        constexpr int kEpi = kWsEpiWarps * 32;
        const uint32_t crow = cstage + (uint32_t)r * kWsCRow;
        uint32_t t = 0, qq = 0;
        int64_t cur = -1;
        int i = -1, y0 = 0, y1 = 0;
        bool tiles = false, prev_tile = false;
        for (int64_t unit = u_begin; unit < u_end; ++unit, ++t) {
            if (unit / ntn != cur) {
                cur = unit / ntn;
                const int base = v.dlist_sp[cur] * kPM;
                i = v.prow[base + r];
                const int first = v.prow[base + (r & ~63)];
                const bool run = __all_sync(0xffffffffu, use_tma_c && i >= 0 && first >= 0 && i == first + (r & 63));
                if (lane == 0) s_run[warp] = run;
                named_barrier(1, kEpi);
                tiles = s_run[0] && s_run[1] && s_run[2] && s_run[3];
                y0 = v.prow[base];
                y1 = v.prow[base + 64];
            }
            const int n0 = (int)(unit % ntn) * kWsNT;
            const bool tile_unit = tiles && n0 + kWsNT <= N;
            const uint32_t a = t & 1u;
            // the same outcome in every epilogue thread: the TMEM loads below are warp-collective
            // and the named barriers need all of them
            if (!named_barrier_and(1, kEpi, mbar_wait(smem_u32(&tfull_bar[a]), (t >> 1) & 1u, err))) break;
            tc::fence_after_sync();
            const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16) + a * kWsNT;
#pragma unroll
            for (int c = 0; c < kWsNT / 64; ++c) {
                uint4 packed[8];
#pragma unroll
                for (int hc = 0; hc < 2; ++hc) {
                    float x[32];
                    tc::tmem_ld32(lane_addr + c * 64 + hc * 32, x);
#pragma unroll
                    for (int q = 0; q < 4; ++q) packed[hc * 4 + q] = Elt<T>::pack(x + q * 8);
                }
                if (c == kWsNT / 64 - 1) {  // the whole accumulator row has been read
                    tc::fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&tempty_bar[a]));
                }
                if (tile_unit) {
                    // buffer qq & 1 was last read by the store of two quarters ago (thread 0's
                    // next-to-last group); after the row path every thread's copies must be read
                    if (c > 0 || prev_tile) {
                        if (tid == 0) bulk_wait_read<1>();
                    } else {
                        bulk_wait_read<0>();
                    }
                    named_barrier(1, kEpi);
                    const uint32_t buf = cstage + (qq & 1u) * kWsQBuf;
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(buf + tc::sw128_off(r, q)),
                                     "r"(packed[q].x), "r"(packed[q].y), "r"(packed[q].z), "r"(packed[q].w)
                                     : "memory");
                    fence_proxy_async_smem();
                    named_barrier(1, kEpi);
                    if (tid == 0) {
                        tma_store_2d(&tmap_c, n0 + c * 64, y0, buf);
                        tma_store_2d(&tmap_c, n0 + c * 64, y1, buf + kWsQBuf / 2);
                        bulk_commit();
                    }
                    ++qq;
                } else {
                    bulk_wait_read<0>();     // this thread's copies have read the staging area
                    named_barrier(1, kEpi);  // ... and every epilogue thread's
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(crow + q * 16),
                                     "r"(packed[q].x), "r"(packed[q].y), "r"(packed[q].z), "r"(packed[q].w)
                                     : "memory");
                    fence_proxy_async_smem();
                    const int nq = min(64, N - n0 - c * 64);  // columns of this quarter inside C
                    if (i >= 0 && nq > 0) {
                        bulk_s2g(C + (int64_t)i * N + n0 + c * 64, crow, (uint32_t)nq * (uint32_t)sizeof(T));
                        bulk_commit();
                    }
                }
            }
            prev_tile = tile_unit;
        }
        bulk_wait<0>();
    } else if (warp < kWsEpiWarps + kWsProdWarps) {
        // ---------------- producers: chunk g belongs to producer warp g mod 3, which loads
        // the whole stage: on the tile path (the chunk's 64 U rows are 64 consecutive rows
        // of B) lane 0 issues the image chunk and four B boxes with one expect-tx arrive; on
        // the gather path lane 0 issues the image chunk, the warp gathers B's 64 rows with
        // cp.async, waits for its own copies and lane 0 arrives. One arrival per chunk, and
        // the tile-path test is a per-panel bit mask in registers, so no shared-memory loads
        // sit in the tile path's loop (they are slow while the tensor core reads operands).
        const int pw = warp - kWsEpiWarps;
        const int32_t* ul = v.ulist;  // the current panel's U list (global, read through L1)
        constexpr int kPieces = kWsNT / 8;  // 16-byte pieces per B row of the tile
        uint32_t g = 0, t = 0;
        bool ok = true;
        int64_t cur = -1;
        int nU = 0, nk = 0;
        bool resident = false, load_a = true, direct = false;
        int ay0 = 0, ay1 = 0;    // direct panels: the first rows of the two 64-row runs
        uint64_t tile_mask = 0;  // bit j: chunk j of the panel loads B as tiles
        const T* img = img_base;
        for (int64_t unit = u_begin; unit < u_end && ok; ++unit, ++t) {
            if (unit / ntn != cur) {  // a new panel: its U list into this warp's shared copy
                cur = unit / ntn;
                const int p = v.dlist_sp[cur];
                const int2 d = *reinterpret_cast<const int2*>(&v.desc[p]);  // dense bits, |U|
                nU = d.y;
                nk = (nU + kKC - 1) / kKC;
                // A chunks straight from the CSR values (an m x L matrix) by two 64 x 64 boxes
                direct = use_tma_v && (d.x & 4);
                ay0 = direct ? v.prow[(int64_t)p * kPM] : 0;
                ay1 = direct ? v.prow[(int64_t)p * kPM + 64] : 0;
                const bool was_resident = resident;
                resident = nk <= kWsASlots;
                load_a = true;
                // Image slots change meaning: the previous unit's MMAs, which may still read
                // any slot, complete before this panel's chunks overwrite one. (The next
                // completion of that barrier needs this unit's chunks, so the wait cannot
                // alias a later phase.)
                if (t > 0 && (resident || was_resident)) {
                    const uint32_t tp = t - 1;
                    if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&tfull_bar[tp & 1u]), (tp >> 1) & 1u, err))) {
                        ok = false;
                        break;
                    }
                }
                img = img_base + v.img_slot[p];
                ul = v.ulist + (size_t)p * kUList;
                // U is sorted and distinct, so 64 positions spanning 63 columns are consecutive
                uint32_t lo = 0, hi = 0;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int j = lane + 32 * h;
                    const bool run = use_tma && j * kKC + kKC - 1 < nU && ul[j * kKC + kKC - 1] - ul[j * kKC] == kKC - 1;
                    const uint32_t bits = __ballot_sync(0xffffffffu, run);
                    if (h == 0) lo = bits;
                    else hi = bits;
                }
                static_assert(kUList / kKC <= 64, "one mask bit per chunk");
                tile_mask = ((uint64_t)hi << 32) | lo;
            } else if (resident) {
                load_a = false;  // the panel's image is already in its slots
            }
            const int n0 = (int)(unit % ntn) * kWsNT;  // the tile's first column
            for (int j = 0; j < nk; ++j, ++g) {
                if ((int)(g % kWsProdWarps) != pw) continue;
                const uint32_t st = g % kWsStages;  // = pw
                static_assert(kWsProdWarps == kWsStages, "stage g mod 4 is always loaded by warp g mod 4");
                // warp-uniform outcome
                if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&empty_bar[st]), ((g / kWsStages) + 1) & 1u, err))) {
                    ok = false;
                    break;
                }
                const uint32_t sb = bbase + st * kWsStageB;
                const uint32_t sa = sbase + (resident ? (uint32_t)j : st) * kSpStageA;
                const uint32_t abytes = load_a ? kSpStageA : 0u;
                const uint32_t fb = smem_u32(&full_bar[st]);
                const T* img_j = img + (size_t)j * kPM * kKC;
                if ((tile_mask >> j) & 1u) {
                    if (lane == 0) {
                        const int u0 = ul[j * kKC];
                        mbar_arrive_expect_tx(fb, abytes + kWsStageB);
                        if (load_a && direct) {
                            tma_load_2d(sa, &tmap_v, j * kKC, ay0, fb);
                            tma_load_2d(sa + kSpStageA / 2, &tmap_v, j * kKC, ay1, fb);
                        } else if (load_a) {
                            bulk_g2s(sa, img_j, kSpStageA, fb);
                        }
#pragma unroll
                        for (int bx = 0; bx < kWsNT / 64; ++bx)
                            tma_load_2d(sb + bx * (kKC / 8) * 1024, &tmap_b, n0 + 64 * bx, u0, fb);
                    }
                    continue;
                }
                if (lane == 0 && load_a) {
                    asm volatile("mbarrier.expect_tx.shared::cta.b64 [%0], %1;" ::"r"(fb), "r"(kSpStageA) : "memory");
                    if (direct) {
                        tma_load_2d(sa, &tmap_v, j * kKC, ay0, fb);
                        tma_load_2d(sa + kSpStageA / 2, &tmap_v, j * kKC, ay1, fb);
                    } else {
                        bulk_g2s(sa, img_j, kSpStageA, fb);
                    }
                }
                // B[U rows j*64 .. +64, n0 .. n0 + 256): 64 x 32 pieces, 64 per lane
                for (int c = lane; c < kKC * kPieces; c += 32) {
                    const int kk = c / kPieces, nch = c % kPieces;
                    const int ncol = n0 + nch * 8;
                    const bool in = j * kKC + kk < nU && ncol < N;
                    const int u = in ? ul[j * kKC + kk] : 0;
                    const uint32_t off = (uint32_t)(nch >> 3) * (kKC / 8 * 1024) + tc::sw128_off(kk, nch & 7);
                    tc::cp_async16(sb + off, in ? (const void*)(B + (int64_t)u * N + ncol) : (const void*)B,
                                   in ? 16 : 0);
                }
                tc::cp_async_commit();   // wait_group covers committed groups only
                tc::cp_async_wait<0>();  // this lane's pieces have landed
                __syncwarp();            // ... and every lane's, before lane 0 releases the stage
                if (lane == 0) mbar_arrive(fb);
            }
        }
        tc::cp_async_wait<0>();
    } else if (lane == 0) {
        // ---------------- MMA issuer
        // Descriptors of each stage's first K step; K step kk adds 32 B (A) or 2 KB (B) to
        // the 16-byte-unit start address in the low bits (no carry: shared addresses < 256 KB).
        uint64_t ad0[kWsASlots], bd0[kWsStages];
#pragma unroll
        for (int i = 0; i < kWsASlots; ++i) ad0[i] = tc::smem_desc_sw128(sbase + i * kSpStageA, 16, 1024);
#pragma unroll
        for (int i = 0; i < kWsStages; ++i) bd0[i] = tc::smem_desc_sw128(bbase + i * kWsStageB, kKC / 8 * 1024, 1024);
        uint32_t g = 0, t = 0, st = 0, ph = 0;  // chunk count, unit count, stage, stage parity
        bool ok = true;
        int64_t cur = -1;
        int nk = 0;
        bool resident = false;
        for (int64_t unit = u_begin; unit < u_end && ok; ++unit, ++t) {
            if (unit / ntn != cur) {
                cur = unit / ntn;
                nk = (v.desc[v.dlist_sp[cur]].y + kKC - 1) / kKC;
                resident = nk <= kWsASlots;
            }
            const uint32_t a = t & 1u;
            if (!mbar_wait(smem_u32(&tempty_bar[a]), ((t >> 1) + 1) & 1u, err)) break;
            tc::fence_after_sync();
            const uint32_t acc = tmem + a * kWsNT;
            for (int j = 0; j < nk; ++j, ++g) {
                if (!mbar_wait(smem_u32(&full_bar[st]), ph, err)) {
                    ok = false;
                    break;
                }
                fence_proxy_async_smem();  // cp.async data (generic proxy) before the tensor core reads it
                tc::fence_after_sync();
                const uint32_t slot = resident ? (uint32_t)j : st;  // j < kWsASlots when resident
                uint64_t ad = ad0[0], bd = bd0[0];
#pragma unroll
                for (int i = 1; i < kWsASlots; ++i)
                    if (slot == (uint32_t)i) ad = ad0[i];
#pragma unroll
                for (int i = 1; i < kWsStages; ++i)
                    if (st == (uint32_t)i) bd = bd0[i];
                tc::mma_f16(acc, ad, bd, idesc, j > 0 ? 1u : 0u);
#pragma unroll
                for (int kk = 1; kk < kKC / 16; ++kk)
                    tc::mma_f16(acc, ad + (uint64_t)(kk * 32 / 16), bd + (uint64_t)(kk * 2048 / 16), idesc, 1u);
                tc::mma_commit(smem_u32(&empty_bar[st]));
                if (++st == kWsStages) {
                    st = 0;
                    ph ^= 1u;
                }
            }
            if (ok) tc::mma_commit(smem_u32(&tfull_bar[a]));
        }
        // every MMA of this thread has completed before the accumulators are released
        tc::mma_commit(smem_u32(&drain_bar));
        mbar_wait(smem_u32(&drain_bar), 0, err);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == kWsEpiWarps + kWsProdWarps) tc::tmem_dealloc(tmem, 2 * kWsNT);
}

// ------------------------------------------------------------------ host dispatch

// Tensor map of a row-major rows x cols matrix of 16-bit elements for boxes of 64 columns x
// box_rows rows with the 128-byte swizzle (false if the driver entry point is unavailable or
// rejects it).
bool encode_rows_map(CUtensorMap* map, const void* base, int32_t rows, int32_t cols, int32_t box_rows, bool bf16) {
    static const PFN_cuTensorMapEncodeTiled_v12000 encode = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess) {
            cudaGetLastError();
            f = nullptr;
        }
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }();
    if (!encode || rows <= 0 || cols <= 0 || (reinterpret_cast<uintptr_t>(base) & 15) || ((int64_t)cols * 2) % 16)
        return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    const cuuint32_t elem[2] = {1, 1};
    return encode(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                  const_cast<void*>(base), dims, strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Cluster launch attributes for kern on `grid` CTAs in clusters of C (C = 1: none). Returns
// the cluster size that can be placed (1 when clusters of C do not fit).
template <typename K>
int fit_cluster(K kern, cudaLaunchConfig_t* cfg, cudaLaunchAttribute* attr, int C) {
    cfg->numAttrs = 1;
    if (C <= 1) return 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)C;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg->numAttrs = 2;
    int active = 0;
    if (cudaOccupancyMaxActiveClusters(&active, kern, cfg) != cudaSuccess || active <= 0) {
        cudaGetLastError();
        cfg->numAttrs = 1;
        return 1;
    }
    return C;
}

template <typename T>
cudaError_t run_sddmm_panels(const void* A, const void* BT, void* out, int32_t kd, const PlanView& v, cudaStream_t s) {
    const uint32_t idesc = tc::instr_desc_f16(std::is_same<T, __nv_bfloat16>::value ? 1u : 0u, 0, 0, kPM, kTileN);
    const int sms = device_props().sm_count;
    const int nkc = (kd + kKC - 1) / kKC;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.stream = s;
    // Many possible tiles (at least two per SM): the grouped kernel, one CTA per SM, each
    // gathering a panel's A rows once for up to four tiles; K split over pairs of CTAs when
    // the groups do not fill the SMs.
    if ((int64_t)v.P * kTiles >= (int64_t)sms * 2) {
        auto kern = sddmm_group_kernel<T>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kGrpSmem);
        if (e != cudaSuccess) return e;
        cfg.blockDim = dim3(kGrpThreads);
        cfg.dynamicSmemBytes = kGrpSmem;
        cfg.gridDim = dim3((unsigned)(sms / 2 * 2));
        const int C = fit_cluster(kern, &cfg, attr, nkc >= 2 ? 2 : 1);
        cfg.gridDim = dim3((unsigned)(sms / C * C));
        CUtensorMap tmap_a, tmap_bt;
        const bool bf16 = std::is_same<T, __nv_bfloat16>::value;
        const int use_tma = encode_rows_map(&tmap_a, A, v.m, kd, kKC, bf16) &&
                                    encode_rows_map(&tmap_bt, BT, v.n, kd, kKC, bf16)
                                ? 1
                                : 0;
        e = cudaLaunchKernelEx(&cfg, kern, static_cast<const T*>(A), static_cast<const T*>(BT), static_cast<T*>(out),
                               kd, v, idesc, device_error_word(), tmap_a, tmap_bt, use_tma);
        count_launches(1);
        if (e != cudaSuccess) return e;
        return cudaGetLastError();
    }
    // Few tiles: one tile per item, 4 warps, two CTAs per SM, K split over clusters of up to 8.
    auto kern = sddmm_panel_kernel<T, 128>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSdSmem);
    if (e != cudaSuccess) return e;
    // Largest shared-memory carveout, so that two CTAs fit on an SM (also when placing clusters).
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    const int64_t max_items = (int64_t)v.P * kTiles;
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = kSdSmem;
    cfg.gridDim = dim3((unsigned)((sms * 2) / min(nkc, kMaxCluster) * min(nkc, kMaxCluster)));
    const int C = fit_cluster(kern, &cfg, attr, nkc < kMaxCluster ? nkc : kMaxCluster);
    // Clusters beyond the co-resident count wait for a free slot; none waits on another.
    const int64_t nclusters = min64((int64_t)(sms * 2) / C, max_items);
    cfg.gridDim = dim3((unsigned)(nclusters * C));
    e = cudaLaunchKernelEx(&cfg, kern, static_cast<const T*>(A), static_cast<const T*>(BT), static_cast<T*>(out), kd, v,
                           idesc, device_error_word());
    count_launches(1);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <typename T>
cudaError_t run_spmm_panels(const void* vals, const int32_t* ro, const void* B, int32_t K, int32_t N, void* C,
                            void* img, const PlanView& v, cudaStream_t s) {
    const int ntn = (N + kSpNT - 1) / kSpNT;
    const bool bf = std::is_same<T, __nv_bfloat16>::value;
    // Many units per CTA: the warp-specialized pipeline, one CTA per SM. It reads the A chunks
    // of panels whose values are already in image order (plan bit 4) straight from the CSR
    // values, viewed as an m x L matrix when every row can have the same length L = nnz / m.
    const bool ws = (int64_t)v.P * ntn >= (int64_t)device_props().sm_count * 6;
    CUtensorMap tmap_v;
    int use_tma_v = 0;
    if (ws && v.m > 0 && v.nnz % v.m == 0) {
        const int64_t L = (int64_t)v.nnz / v.m;
        if (L >= kKC && L % 8 == 0 && L <= kUList && (uintptr_t)vals % 16 == 0)
            use_tma_v = encode_rows_map(&tmap_v, vals, v.m, (int32_t)L, 64, bf) ? 1 : 0;
    }
    const uint32_t dsmem = densify_smem_bytes(K, sizeof(T));
    cudaError_t e = cudaFuncSetAttribute(densify_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dsmem);
    if (e != cudaSuccess) return e;
    e = launch_pdl(densify_kernel<T>, v.P * kGroups, 256, dsmem, s, static_cast<const T*>(vals), ro,
                   static_cast<T*>(img), v, (int)(dsmem / (kGroupRows * sizeof(T))), use_tma_v);
    if (e != cudaSuccess) return e;
    const uint32_t idesc_ws = tc::instr_desc_f16(bf ? 1u : 0u, 0, 1, kPM, kWsNT);
    if (ws) {
        auto kws = spmm_panel_ws_kernel<T>;
        e = cudaFuncSetAttribute(kws, cudaFuncAttributeMaxDynamicSharedMemorySize, kWsSmem);
        if (e != cudaSuccess) return e;
        CUtensorMap tmap, tmap_c;
        const int use_tma = encode_rows_map(&tmap, B, K, N, 64, bf) ? 1 : 0;
        const int use_tma_c = encode_rows_map(&tmap_c, C, v.m, N, 64, bf) ? 1 : 0;  // 64 x 64 boxes of C
        if (!use_tma_v) std::memset(&tmap_v, 0, sizeof(tmap_v));
        e = launch_pdl(kws, device_props().sm_count, kWsThreads, kWsSmem, s, static_cast<const T*>(B),
                       static_cast<T*>(C), static_cast<const T*>(img), N, v, idesc_ws, device_error_word(), tmap,
                       use_tma, tmap_c, use_tma_c, tmap_v, use_tma_v);
        count_launches(2);
        if (e != cudaSuccess) return e;
        return cudaGetLastError();
    }
    const int grid = (int)min64((int64_t)device_props().sm_count * 2, (int64_t)v.P * ntn);
    // Few units (each CTA about one): 4 warps, which share the SMs better with concurrent
    // operators.
    auto kern = spmm_panel_kernel<T, kTileThreads>;
    const int threads = kTileThreads;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSpSmem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    const uint32_t idesc = tc::instr_desc_f16(std::is_same<T, __nv_bfloat16>::value ? 1u : 0u, 0, 1, kPM, kSpNT);
    e = launch_pdl(kern, grid, threads, kSpSmem, s, static_cast<const T*>(B), static_cast<T*>(C),
                   static_cast<const T*>(img), N, v, idesc, device_error_word());
    count_launches(2);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

size_t image_bytes(int dt, int32_t m, int32_t k, int32_t nnz) {
    if (!dtype_ok(dt) || !plan_panels_enabled(m, k)) return 0;
    return align_up(spmm_image_budget_elems(m, nnz) * 2, 1024);
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
    (void)kd;
    (void)dt;
    (void)structure_aware;
    return 1024 + align_up(plan_bytes(m, n, nnz), 1024);
}

cudaError_t launch_spmm(int dt, int it, const void* vals, const int32_t* ro, const void* row_idx, const void* col,
                        int32_t m, int32_t k, int32_t nnz, const void* B, int32_t n, void* C, const void* plan,
                        void* ws, bool allow_panels, cudaStream_t s) {
    char* w = reinterpret_cast<char*>(align_up(reinterpret_cast<uintptr_t>(ws), 1024));
    PlanView v;
    cudaError_t e = resolve_plan(it, ro, row_idx, col, m, k, nnz, plan, &w, &v, s);
    if (e != cudaSuccess) return e;
    // Narrow B (n <= 16) is bound by streaming A, not by products: no tensor-core tiles.
    const bool panels = allow_panels && nnz > 0 && v.panels && dtype_ok(dt) && n % 8 == 0 && n > kNarrowMax &&
                        aligned16(B) && aligned16(C);
    const int32_t* order = v.panels ? v.prow : nullptr;  // the plan's row order
    if (!panels)
        return launch_spmm_general(dt, it, vals, ro, row_idx, col, m, k, B, n, C, v.bins_spmm(), nullptr, order, s);
    // The general rows (outside the panels that get an image) and the panels write disjoint
    // rows of C: the row kernel runs on the side stream while the panels run on s. The panels
    // are queued first, so that their CTAs are placed before the row kernel fills the SMs.
    cudaStream_t side = side_fork(s);
    e = dt == kF16 ? run_spmm_panels<__half>(vals, ro, B, k, n, C, w, v, s)
                   : run_spmm_panels<__nv_bfloat16>(vals, ro, B, k, n, C, w, v, s);
    if (e == cudaSuccess)
        e = launch_spmm_general(dt, it, vals, ro, row_idx, col, m, k, B, n, C, v.bins_spmm(), v.sp_dense, order,
                                side ? side : s);
    // join on every path, so that s never runs ahead of work queued on the side stream
    const cudaError_t ej = side ? side_join(s) : cudaSuccess;
    return e != cudaSuccess ? e : ej;
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
    const int32_t* order = v.panels ? v.prow : nullptr;  // the plan's row order
    if (!panels)
        return launch_sddmm_general(dt, it, ro, row_idx, col, m, n, kd, A, BT, out, v.bins_sddmm(), nullptr, order, s);
    // The general rows and the dense panels write disjoint entries: side stream for the rows,
    // queued after the panels.
    cudaStream_t side = side_fork(s);
    e = dt == kF16 ? run_sddmm_panels<__half>(A, BT, out, kd, v, s)
                   : run_sddmm_panels<__nv_bfloat16>(A, BT, out, kd, v, s);
    if (e == cudaSuccess)
        e = launch_sddmm_general(dt, it, ro, row_idx, col, m, n, kd, A, BT, out, v.bins_sddmm(), v.dense, order,
                                 side ? side : s);
    const cudaError_t ej = side ? side_join(s) : cudaSuccess;
    return e != cudaSuccess ? e : ej;
}

}  // namespace spops
