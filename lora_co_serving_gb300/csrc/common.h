// common.h -- plan structures shared by the host planner and the sm_103a kernels.
//
// The layer is executed as lists of work items over 128-row tiles of tokens:
//   * a tile is a window of 128 consecutive rows of x (or dY), or 128 rows
//     copied out of x into a gathered buffer (short decode segments sorted by
//     adapter, so that one tile meets few adapters);
//   * each tile carries the list of adapters ("chunks") its rows use; chunk c
//     owns LoRA columns [zcol, zcol + roundup(r,16)) of the tile;
//   * the shrink x*A of every tile row is written, scaled and masked to its
//     own chunk, as the tile's "Z" matrix [128, sum of padded ranks]; the
//     expand (Z * stacked B) is then extra K-steps of the base GEMM, so the
//     LoRA term lands in the same accumulator and y is written once.
#pragma once
#include <stdint.h>

namespace lora {

constexpr int kTileM = 128;       // rows per tile (MMA M)
constexpr int kBN = 256;          // output columns per main work item (MMA N)
constexpr int kBK = 64;           // K elements per pipeline stage (one 128-byte swizzle row of bf16)
constexpr int kStages = 4;
constexpr int kZBlockBytes = kTileM * kBK * 2;   // one 128x64 bf16 Z block in its shared-memory image
constexpr int kMaxTrainSegs = 48;
constexpr int kPassCols = 256;    // LoRA columns per shrink pass (MMA N limit)

enum ItemKind : int32_t {
    kShrinkFwd = 0,   // Z <- s * mask(x A^T), xa_save <- x A^T           (A: x rows, B: A-pool rows, K-major)
    kMainFwd = 1,     // y <- x Wt^T + Z Bstack                             (B: Wt K-major; ext: B-pool MN-major)
    kShrinkDyb = 2,   // Z <- s * mask(dY B^T), dYB^T (transposed) <- dY B^T (A: dY rows, B: B-pool rows)
    kShrinkXa = 3,    // xA^T (transposed) <- x A^T                         (A: x rows, B: A-pool rows)
    kMainDx = 4,      // dX <- dY Wt + Z Astack                             (B: Wt MN-major; ext: A-pool MN-major)
    kGradDb = 5,      // dB^T[n, j] = s * sum_t dY[t,n] xA[t,j]             (A: dY^T MN-major, B: xA^T K-major)
    kGradDa = 6       // dA^T[k, j] = s * sum_t x[t,k] dYB[t,j]             (A: x^T MN-major, B: dYB^T K-major)
};

struct TileDesc {
    int32_t a_row0;   // first row of the window in the row source (x, dY or the gathered buffer)
    int32_t a_src;    // 0: x / dY window; 1: gathered buffer
    int32_t chunk0;   // first chunk (index into the chunk array)
    int32_t nchunk;
    int32_t ext_k;    // LoRA columns: sum over chunks of roundup(r,16)
    int32_t z_blk0;   // first Z block of this tile
    int32_t tpos0;    // backward tiles: column of tile row 0 in the transposed buffers; -1 otherwise
    int32_t atom0;    // first entry of this tile in the atom-row tables (one entry per 8 LoRA columns)
    int32_t sh_c0;    // LoRA columns [sh_c0, sh_c1) hold this tile's own adapters (the shrink computes only
    int32_t sh_c1;    //   these; the pair's other columns of this tile's Z stay zero)
    int32_t seg;      // backward tiles: fine-tuning segment (index in increasing start order); -1 otherwise
    int32_t zstride;  // sliced layers: LoRA-column stride between the slices' copies of a chunk (0: one slice).
                      //   A row keeps columns zcol + i*zstride + [0, r) of its chunk for every slice i.
};
// Tiles come in pairs (2p, 2p+1) that share one chunk list, ordered [adapters only in the first tile |
// adapters in both | adapters only in the second], so that the M = 256 main pass runs one pair per CTA pair
// and each tile's own adapters occupy one contiguous column range.
//
// Sliced layers (several projections of one input fused along N, e.g. q|k|v): slice i of adapter a has its own
// down factor (rows [i r, (i+1) r) of a's A block) and the up factor is a's B block restricted to the slice's
// output columns.  Forward tiles hold one region of LoRA columns per slice (stride zstride, a multiple of 64);
// the main items of slice i's output columns use a copy of the tile whose Z starts at region i.  Backward tiles
// (one adapter) hold the slices side by side, each padded to 16 columns.

struct Chunk {
    int32_t adapter;
    int32_t zcol;     // multiple of 16
    int32_t r;
    int32_t prow_a;   // first row of the adapter's block in the A pool viewed as [rows, K]
    int32_t prow_b;   // first row of the adapter's block in the B pool viewed as [rows, N]
    float scale;
    int32_t pad0, pad1;
};

struct WorkItem {
    int32_t kind;
    int32_t tile;     // tile index; for grad items: grad-group index
    int32_t n0;       // main: first output column; shrink: first LoRA column of the pass; grad: first row m0
    int32_t nk;       // main/shrink: k-blocks of the dense loop; grad: token blocks of this item (or split)
    int32_t mma_n;    // N of the MMA
    int32_t n_ext;    // main: LoRA k-blocks of this item (Z blocks it touches); shrink and split grad: its unit index
    int32_t kb0;      // shrink, split main and grad items: first k-block (token block) of this split
    int32_t part;     // shrink and split grad: column offset of this split's fp32 partial [mma_n, 128] in the
                      // partial buffer; main: first partial slot of the output tile (split s writes slot part + s)
    int32_t nsplit;   // main and grad: number of splits of the reduction (0 or 1 = no split)
    int32_t split;    // main and grad: index of this split
    int32_t ext_c0;   // main: LoRA columns [ext_c0, ext_c1) of the tile's Z that this item multiplies (16-aligned)
    int32_t ext_c1;
    int32_t j0;       // grad: first row of the transposed xA / dYB buffer this item reads (the slice's rows)
    int32_t pad0, pad1, pad2;
};

// An output tile of the main pass whose K loop is split: its splits write fp32 partials
// (slot part + s, each 2 CTAs x [256 columns][128 rows]) and a reduce launch sums them in split order.
struct SplitTile {
    int32_t tile;     // first tile of the pair (its rows)
    int32_t n0;       // first output column
    int32_t part;     // first partial slot
    int32_t nsplit;
    int32_t pad0, pad1, pad2, pad3;
};

// The shrink of the gathered decode rows on CUDA cores: each run of up to kBgmvRows consecutive gathered rows that
// share a chunk is one group; a work unit is one group and 8 of its LoRA columns.  The unit reads the rows from x
// and its adapter's 8 rows of A once, sums x . A_j in fp32 over K in a fixed order (so a row's value depends on its
// own x and A rows alone) and writes Z = bf16(s * xA) into the tile's Z image, where the main pass's K-extension
// reads it.  The unit of LoRA columns 0..7 also writes the run's rows into the gathered buffer (the main pass's row
// operand), so no separate gather launch runs; gathered rows without an adapter (and the empty rows that pad the
// last tile) form copy-only units (chunk -1).  Sliced forward layers: LoRA column j of the group (j < S * rank) is
// slice j / rank's column j % rank, in that slice's Z region.
struct BgmvGroup {
    int32_t g_row0;   // first row in the gathered buffer
    int32_t n_rows;   // rows of the run (at most kBgmvRows)
    int32_t chunk;    // the rows' chunk (adapter, Z column, rank, scale, first A row); -1: copy the rows only
    int32_t j0;       // first LoRA column of this work unit (multiple of 8, below S * rank)
    int32_t tile;     // tile of the rows
    int32_t row0;     // row of g_row0 in the tile
    int32_t pad0, pad1;
};
#ifndef LORA_BGMV_ROWS
#define LORA_BGMV_ROWS 4
#endif
constexpr int kBgmvRows = LORA_BGMV_ROWS;   // rows per CUDA-core shrink unit (4 or 8)
#ifndef LORA_BGMV_MAX_ROWS
#define LORA_BGMV_MAX_ROWS 1024
#endif
constexpr int kBgmvMaxRows = LORA_BGMV_MAX_ROWS;   // gathered rows (whole tiles) up to which the CUDA-core shrink runs

// One shrink pass of one tile, or one gradient item whose token range is split.  Its splits write fp32 partial
// sums; the last split to finish (counted per row quarter) sums them in split order and writes Z and the saved or
// transposed copies (a gradient item: its rows of dA or dB).
struct ShrinkUnit {
    int32_t kind;     // kShrinkFwd, kShrinkDyb or kShrinkXa; kGradDb or kGradDa for a split gradient item
                      // (then tile is its gradient group and n0 its first row)
    int32_t tile;
    int32_t n0;       // first LoRA column of the pass
    int32_t mma_n;
    int32_t nsplit;
    int32_t part0;    // column offset of split 0; split s sits at part0 + s * mma_n
    int32_t pad0, pad1;
};

// K-blocks per split of a shrink reduction.  Split boundaries depend on the batch size and K alone, so a row's
// xA is summed in the same order whatever the rest of its tile holds; small batches split finer so that their
// few tiles still spread over every SM.
inline int shrink_split_kb(int64_t T) { return T <= 1024 ? 8 : (T <= 4096 ? 16 : 32); }
// Forward shrink passes are kPassCols wide, narrowed (down to 64 columns) while a launch would have fewer items
// than about one per SM: a decode batch's few tiles carry many adapters' columns, and narrower passes spread them
// over more SMs and shrink each unit's partial sums.  A column's sum does not depend on the pass width.
constexpr int kShrinkTargetItems = 148;

// Main pass K-splits: when a launch has fewer output tiles than ~1.25 waves of CTA pairs, each tile's K loop is
// split, the splits write fp32 partials, and a reduce launch sums them in split order (96 measured best against 38,
// 57, 76, 114, 152 and 228 on decode batches of 64-1024 tokens: 256 tokens 59 -> 54 us replayed from a graph).  Forward tiles keep their
// LoRA K-steps out of the dense splits and cut them only at chunk boundaries, so every row's own adapter columns
// sit in one split: a row's sum is (dense splits, in K order) + (its LoRA term) + exact zeros, whatever the other
// rows of its tile, and stays independent of the segment and pool order.  Backward tiles hold one adapter; their
// LoRA K-steps go with the last dense split.
#ifndef LORA_MAIN_TARGET_ITEMS
#define LORA_MAIN_TARGET_ITEMS 96
#endif
constexpr int kMainTargetItems = LORA_MAIN_TARGET_ITEMS;
// CTA pairs the planner sizes waves for (76 on a 152-SM GB300; plans stay valid on any device).
constexpr int kPairsPlanned = 76;
constexpr int kMainPartialFloats = kBN * kTileM;   // one CTA's fp32 partial of a 128 x 256 output tile

// Extents of the buffers a launch writes, against which the kernels check every store index they derive from the
// plan when a call sets LORA_DEBUG_CHECKS (a failing check skips the store and records LORA_ERR_BOUNDS).
struct DebugBounds {
    int64_t out_rows;       // rows of y (forward) or dX (backward)
    int64_t z_blocks;       // Z blocks of the workspace
    int64_t xa_elems;       // elements of the saved-activation buffer
    int64_t t_elems;        // elements of each transposed buffer (xA^T, dYB^T)
    int64_t part_floats;    // floats of the shrink partials
    int64_t main_slots;     // split partial slots of the main pass
    int64_t grad_a, grad_b; // elements of dA and dB (the pools' extents)
    int64_t x_rows;         // rows of x
    int64_t g_rows;         // rows of the gathered buffer
};

struct GradGroup {    // one fine-tuning adapter of a backward call
    int32_t adapter;
    int32_t r;
    int32_t seg0;     // first entry in the train-segment arrays
    int32_t nseg;
    int32_t prow_a, prow_b;
    float scale;
    int32_t nslice;   // slices of the layer: the adapter's A block has nslice * r rows
};

struct TrainSeg {     // fine-tuning segment; grouped by adapter, increasing start within a group
    int32_t start;
    int32_t len;
    int32_t tpos0;    // first column in the transposed buffers (multiple of 128)
    int32_t group;
    int32_t xoff;     // element offset of the segment's [len, r] block in the saved-activation buffer
    int32_t r;        // width of that block (rank x slices)
    int32_t order;    // index among the fine-tuning segments in increasing start order
    int32_t pad1;
};

}  // namespace lora
