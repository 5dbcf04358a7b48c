// plan.h -- host-side validation and tile planning for the mixed-batch LoRA layer.
#pragma once
#include <stddef.h>
#include <stdint.h>

#include <string>
#include <vector>

#include "common.h"
#include "lora_mixed.h"

namespace lora {

// Segments shorter than this (and not fine-tuning) are decode-like: their rows are copied into a
// gathered buffer sorted by adapter, so that a tile meets as few adapters as possible.
constexpr int kShortSegment = 16;
// Tiles per L2 band: main items sweep all output columns of a band of tiles before the next band.
#ifndef LORA_BAND_TILES
#define LORA_BAND_TILES 16
#endif
constexpr int kBandTiles = LORA_BAND_TILES;


struct Problem {
    int32_t T = 0, K = 0, N = 0;
    lora_dtype_t dt = LORA_BF16;
    int32_t n_adapters = 0;
    const int64_t* a_off = nullptr;
    const int64_t* b_off = nullptr;
    const int32_t* rank = nullptr;
    const float* scale = nullptr;
    std::vector<lora_segment_t> segs;   // non-empty segments, increasing start
    int64_t rows_a = 0, rows_b = 0;     // row extents of the pools viewed as [rows, K] and [rows, N]
    int64_t xa_elems = 0;               // elements of the saved-activation buffer
    int32_t n_train = 0;
    int32_t S = 1;                      // slices of a fused layer; slice i = output columns [bounds[i], bounds[i+1])
    int32_t bounds[LORA_MAX_SLICES + 1] = {0, 0, 0, 0, 0};
    int32_t slice_of_col(int32_t n) const {
        int32_t i = 0;
        while (i + 1 < S && n >= bounds[i + 1]) ++i;
        return i;
    }
};

// Host validation of every argument that does not need the GPU.  Returns LORA_OK or a LORA_ERR_* code.
// slices may be NULL (one slice).
int validate(int32_t T, int32_t K, int32_t N, lora_dtype_t dt, const lora_pool_t* pool, const lora_segment_t* segs,
             int32_t n_segs, Problem* out, std::string* err, const lora_slices_t* slices = nullptr);

struct Plan {
    std::vector<TileDesc> tiles;
    std::vector<Chunk> chunks;
    std::vector<int32_t> rowmap;     // 128 per tile: token row or -1
    std::vector<int32_t> rowchunk;   // 128 per tile: chunk index or -1
    std::vector<int32_t> rowaux;     // 128 per tile: forward: xa_save element offset or -1; backward: -1
    std::vector<int32_t> atoms_a;    // per tile, per 8 LoRA columns: first A-pool row of that 8-row atom
    std::vector<int32_t> atoms_b;    // same for the B pool
    std::vector<int32_t> boxes_a;    // per atom: atoms loaded by one TMA box starting at it (1, 2, 4 or 8: a run of
    std::vector<int32_t> boxes_b;    //   consecutive pool rows inside one chunk and one 64-column block), 0 if an
                                     //   earlier atom's box covers it
    std::vector<WorkItem> items[3];  // shrink items (1-CTA kernel), main pair items (2-CTA kernel), grad items
    std::vector<ShrinkUnit> units;   // shrink passes (each finalized by its last K-split)
    std::vector<GradGroup> groups;
    std::vector<TrainSeg> tsegs;
    int32_t n_gtiles = 0;            // forward: tiles of the gathered buffer
    int32_t g_tile0 = 0;             // forward: index of the first gathered tile (they are consecutive)
    int64_t z_blocks = 0;
    int64_t tcols = 0;               // backward: columns of the transposed xA / dYB buffers
    int64_t part_cols = 0;           // columns (of 128 fp32 each) of the shrink partial-sum buffer
    int64_t main_slots = 0;          // K-split partial slots of the main pass (each 2 CTAs x 128 x 256 fp32)
    std::vector<SplitTile> splits;   // split output tiles of the main pass (summed by the reduce launch)
    std::vector<BgmvGroup> bgmv;     // CUDA-core shrink units of the gathered decode rows (few of them)
    int64_t T = 0;                   // tokens of the batch (sets the shrink split size)
};

void plan_forward(const Problem& p, Plan* out);
// recompute: x A of every fine-tuning tile is recomputed.  per_segment: the caller's device flag table decides
// per segment (recompute items exist for every tile and are skipped on the device for segments flagged saved).
void plan_backward(const Problem& p, bool want_dx, bool want_da, bool want_db, bool recompute, Plan* out,
                   bool per_segment = false);

// Host cross-check of a plan (LORA_DEBUG_CHECKS, lora_plan_check): every index the kernels derive from it -- rows
// of x and of the gathered buffer, pool rows of the adapter-row atoms and their boxes, Z blocks and columns, saved
// and transposed activation offsets, shrink and split partial slots, output columns, gradient rows -- lies inside
// the buffer it addresses.  Returns LORA_OK, or LORA_ERR_BOUNDS with the first violation in *err.
int check_plan(const Problem& p, const Plan& pl, bool backward, std::string* err);

// Greedy list scheduling of the items (in order) onto G persistent CTAs by estimated cost.
// off has G+1 entries; list holds item indices grouped by CTA, each CTA's in increasing order.
void assign_items(const std::vector<WorkItem>& items, const Plan& plan, int G, std::vector<int32_t>* off,
                  std::vector<int32_t>* list);
// The estimated cost (cycles) by which assign_items balances the CTAs.
int64_t item_cost_estimate(const WorkItem& w);

// Byte offsets of everything a call keeps in the workspace.
struct Layout {
    size_t status = 0;
    size_t counters = 0, zero_end = 0;   // [status, zero_end) is zeroed at the start of every call
    size_t tiles = 0, chunks = 0, rowmap = 0, rowchunk = 0, rowaux = 0, groups = 0, tsegs = 0;
    size_t atoms_a = 0, atoms_b = 0, boxes_a = 0, boxes_b = 0, units = 0, seg_flags = 0, splits = 0, bgmv = 0;
    size_t items[3] = {0, 0, 0}, cta_off[3] = {0, 0, 0};
    size_t plan_end = 0;
    size_t xg = 0, z = 0, xat = 0, dybt = 0, part = 0, part_main = 0;
    size_t simt = 0;                 // float32 path scratch
    size_t total = 0;
};

constexpr int kMaxCtas = 1024;
Layout layout_of(const Problem& p, const Plan& plan, bool backward);

// While alive, calls on this thread copy their plan straight from host memory (no pinned staging ring).
class DirectUpload {
  public:
    DirectUpload();
    ~DirectUpload();
  private:
    bool prev_;
};
void set_last_error(const char* msg);

// Bytes of workspace lora_mixed_forward needs for this call (its forward layout alone; the bf16 plan comes from the
// per-thread plan cache that the forward itself uses).  Returns LORA_OK or a validation error (message set).
int forward_scratch_bytes(int32_t T, int32_t K, int32_t N, lora_dtype_t dt, const lora_pool_t* pool,
                          const lora_segment_t* segs, int32_t n_segs, size_t* out);

// The float32 path keeps per-token adapter ids and an xA scratch of [T, 128] floats.
size_t simt_scratch_bytes(const Problem& p);

}  // namespace lora
