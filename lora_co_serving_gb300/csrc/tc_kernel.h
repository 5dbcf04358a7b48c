// tc_kernel.h -- launch interface of the persistent tcgen05 kernel.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "common.h"
#include "lora_mixed.h"

namespace lora {

// Everything one launch needs.  Tensor maps live in the kernel's parameter space (__grid_constant__).
struct KParams {   // CUtensorMap members keep the 64-byte alignment the TMA unit needs
    CUtensorMap tm_x;      // x rows,  [T, K] bf16, box {64, 128}, 128B swizzle
    CUtensorMap tm_xg;     // gathered rows buffer, [G*128, K], box {64, 128}
    CUtensorMap tm_dy;     // dY rows, [T, N], box {64, 128}
    CUtensorMap tm_w;      // Wt [N, K]: forward box {64, 128} (K-major B half); backward box {64, 64} (MN-major)
    CUtensorMap tm_w3;     // backward, K a multiple of 64: Wt as [K/64][N][64] (64-column chunks outermost), box
                           //   {64, 64, 2}: both 64-column MN atoms of a CTA's B half in one load
    CUtensorMap tm_pa;     // A pool viewed as [rows, K], box {64, 8}
    CUtensorMap tm_pb;     // B pool viewed as [rows, N], box {64, 8}
    CUtensorMap tm_pa_h[3];  // A pool with boxes of 16, 32 and 64 rows (runs of 2, 4, 8 atoms)
    CUtensorMap tm_pb_h[3];  // B pool, same
    CUtensorMap tm_xat;    // xA^T  [128, P], box {64, 8}
    CUtensorMap tm_dybt;   // dYB^T [128, P], box {64, 8}
    CUtensorMap tm_out;    // main-pass output (y or dX) [rows, out_cols], ld out_ld, box {32, 32}, 64B swizzle
    CUtensorMap tm_z;      // Z blocks as [blocks*128, 64] bf16 rows of 128 B, box {64, 128}, no swizzle (the blocks
                           // already hold the swizzled shared-memory image)
    CUtensorMap tm_seg_dy[kMaxTrainSegs];   // dY rows of fine-tuning segment q, [len, N], box {64, 64}
    CUtensorMap tm_seg_x[kMaxTrainSegs];    // x rows of fine-tuning segment q,  [len, K], box {64, 64}

    const TileDesc* tiles;
    const Chunk* chunks;
    const int32_t* rowmap;
    const int32_t* rowchunk;
    const int32_t* rowaux;
    const GradGroup* groups;
    const TrainSeg* tsegs;
    const WorkItem* items;   // in CTA order: CTA (pair, in the main pass) c runs items [cta_off[c], cta_off[c + 1])
    const int32_t* cta_off;
    const int32_t* atoms_a;  // per tile, per 8 LoRA columns: A-pool row of the atom
    const int32_t* atoms_b;  // same for the B pool
    const int32_t* boxes_a;  // per atom: atoms in the TMA box that starts at it (0: covered by an earlier box)
    const int32_t* boxes_b;
    float* part;             // shrink items: fp32 partial sums, per 4 columns [128 rows][4]
    float* part_main;        // split main items: fp32 partial tiles, [slot][CTA][64 column groups][128 rows][4]
    const int32_t* seg_flags;  // backward with a per-segment flag table: snapshot, nonzero = saved xA is used
                               // (the segment's x A recompute items are skipped); null otherwise
    const ShrinkUnit* units; // shrink passes (splits of one pass share a unit)
    int32_t* counters;       // per unit and row quarter: splits finished (zeroed at the start of every call)

    const uint8_t* zin;     // Z blocks read by main items
    uint8_t* zout;          // Z blocks written by shrink items
    __nv_bfloat16* out;     // main items: y [T, N] or dX [T, K]
    __nv_bfloat16* xa_save; // forward shrink: saved xA of fine-tuning rows
    __nv_bfloat16* xat;     // backward shrink: xA^T  [128, P]
    __nv_bfloat16* dybt;    // backward shrink: dYB^T [128, P]
    float* dA;
    float* dB;
    int32_t* status;
    int32_t out_ld;         // row stride of `out` in elements
    int32_t out_cols;       // valid columns of `out`
    int32_t t_ld;           // P
    int32_t K, N;
    int32_t accumulate;
    int32_t w3;              // backward: tm_w3 is valid
    int32_t debug;           // LORA_DEBUG_CHECKS: check every store index against `db` (see common.h)
    DebugBounds db;
};

size_t tc_smem_bytes();
cudaError_t tc_launch(const KParams& P, int grid, cudaStream_t stream);      // shrink and grad items, 1 CTA each
size_t tc2_smem_bytes();
// Sums the partials of the split output tiles (device array of n_splits records) and writes their output rows.
cudaError_t main_reduce_launch(const SplitTile* splits, int32_t n_splits, const int32_t* rowmap, const float* part,
                               __nv_bfloat16* out, int32_t out_ld, int32_t out_cols, const KParams& P,
                               cudaStream_t stream);
cudaError_t tc2_launch(const KParams& P, int pairs, cudaStream_t stream);    // main items, clusters of 2 CTAs
cudaError_t selftest_timeout_launch(int32_t* status, cudaStream_t stream);
// The limit of every bounded wait of the library's kernels on the current device (synchronous copy).
cudaError_t set_wait_limit_ns(uint64_t ns);

}  // namespace lora
