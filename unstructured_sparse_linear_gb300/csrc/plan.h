// The mask plan: everything the operators derive from a CSR structure alone (row bins and
// the dense-panel decomposition), built once per mask and shared by spmm and sddmm.
//
// Layout in caller memory (all offsets 1024-byte aligned, computed by plan_layout):
//   hdr        int32[32]  bins_spmm[4], bins_sddmm[4], counts[8] (kCnt*), dims[4] {m, n, nnz, P}
//   pan_part   int32[P][4]    per panel: {#rows >= spmm long, #rows >= sddmm long,
//                             #non-empty rows, #entries}
// when panels are enabled (n <= 65536):
//   bm, wbase  [P][W]          column bitmap of a panel; exclusive prefix of its popcounts
//   desc       int4[P]         {dense bits, |U|, entries, non-empty rows}; dense bit 0: SDDMM
//                              tiles (|U| <= kUCap), bit 1: SpMM image (|U| <= kUList), bit 2:
//                              the CSR values already hold the image (rows of one length
//                              L = |U| in two runs of 64 consecutive rows)
//   prow       int32[P*128]    row id at each panel position (-1 past m)
//   ulist      int32[P][kUList] sorted columns of a dense panel
//   upos       uint16[nnz]     column position of each entry in its panel's U
//   ts         int32[P*128][kTiles + 1]  first entry of each 128-column tile of U, per row
//   tmask      uint32[P*128][kUCap / 32] bit u set when the row has an entry at U position u
//   dense      uint8[P]        panel runs on tensor cores (SDDMM)
//   sp_dense   uint8[P]        panel has a SpMM image slot (tensor cores for SpMM)
//   items      int32[P*kTiles] SDDMM work items (panel << 8 | tile)
//   gitems     int32[P*kTiles/kGroupTiles]  SDDMM work items of the grouped kernel
//                              (panel << 8 | group of kGroupTiles consecutive tiles)
//   dlist_sp   int32[P]        panels with an image slot
//   img_slot   int32[P]        image offset (elements) or -1
// when the rows are also ordered (m <= kOrderMaxRows):
//   okey       uint32[P*128]   sort key of each position of row_idx
//   olong      uint32[P*4]     per 32 positions: key of the run of >= 32 positions starting there, or ~0
//   obrk       uint32[P*4]     bit p: position p of row_idx starts a stretch of one key
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "internal.h"

namespace spops {

constexpr int kPM = kPanelRows;   // rows per panel (UMMA M)
constexpr int kUCap = 1024;       // most distinct columns of an SDDMM-dense panel (8 tiles of 128)
constexpr int kUList = 4096;      // most distinct columns of a SpMM-dense panel (the image's K)
constexpr int kTileN = 128;       // SDDMM tile width over U (UMMA N)
constexpr int kTiles = kUCap / kTileN;
constexpr int kGroupTiles = 4;    // tiles one CTA of the grouped SDDMM kernel keeps in tensor memory
constexpr int kGroupRows = 8;     // rows per CTA of the U-position and image kernels, one per warp
constexpr int kGroups = kPM / kGroupRows;
constexpr int kPlanCluster = 8;   // CTAs per panel (one thread-block cluster) in the row step
constexpr int kCtaRows = kPM / kPlanCluster;
constexpr int kMaxPanelCols = 65536;
constexpr int kMinDenseRows = 16;
constexpr int kOrderMaxRows = 16384;  // masks up to this many rows get the column-pattern row order

enum PlanCount {
    kCntDense = 0,      // dense panels (SDDMM)
    kCntTiles = 1,      // SDDMM items
    kCntDenseSp = 2,    // panels with a SpMM image
    kCntDenseNnz = 3,   // entries in dense panels
    kCntImgElems = 4,   // image elements assigned
    kCntPanels = 5,
    kCntGroups = 6,     // SDDMM items of the grouped kernel
};

struct PlanView {
    int32_t* hdr;
    int32_t* pan_part;
    uint32_t* bm;
    int32_t* wbase;
    int4* desc;
    int32_t* prow;
    int32_t* ulist;
    uint16_t* upos;
    int32_t* ts;
    uint32_t* tmask;
    uint8_t* dense;
    uint8_t* sp_dense;
    int32_t* items;
    int32_t* gitems;
    int32_t* dlist_sp;
    int32_t* img_slot;
    uint32_t* okey;
    uint32_t* olong;
    uint32_t* obrk;
    int32_t m, n, nnz, P, W;
    bool panels;
    __host__ __device__ int32_t* bins_spmm() const { return hdr; }
    __host__ __device__ int32_t* bins_sddmm() const { return hdr + 4; }
    __host__ __device__ int32_t* counts() const { return hdr + 8; }
};

struct PlanLayout {
    size_t hdr, pan_part, bm, wbase, desc, prow, ulist, upos, ts, tmask, dense, sp_dense, items, gitems, dlist_sp,
        img_slot, okey, olong, obrk;
    size_t total;
};

bool plan_panels_enabled(int32_t m, int32_t n);
PlanLayout plan_layout(int32_t m, int32_t n, int32_t nnz);
PlanView plan_view(void* base, int32_t m, int32_t n, int32_t nnz);
inline size_t plan_bytes(int32_t m, int32_t n, int32_t nnz) { return plan_layout(m, n, nnz).total; }

// Elements of SpMM image storage a workspace provides for this mask (images beyond this
// budget are not assigned and those panels run on the general kernels).
size_t spmm_image_budget_elems(int32_t m, int32_t nnz);

// Queue the plan kernels on s. img_budget: SpMM image elements available (0: none).
cudaError_t launch_plan_build(int it, const int32_t* ro, const void* row_idx, const void* col, const PlanView& v,
                              int64_t img_budget, cudaStream_t s);
cudaError_t launch_plan_stats(const PlanView& v, int32_t* out, cudaStream_t s);

}  // namespace spops
