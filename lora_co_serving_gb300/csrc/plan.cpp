// plan.cpp -- host-side validation and tile planning (no CUDA calls).
#include "plan.h"

#include <algorithm>
#include <cstdint>
#include <functional>
#include <cstring>
#include <iterator>
#include <utility>

namespace lora {

static inline int32_t pad16(int32_t r) { return (r + 15) & ~15; }
static inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
static inline size_t align256(size_t v) { return (v + 255) & ~size_t(255); }
static int64_t item_cost(const WorkItem& w);

int validate(int32_t T, int32_t K, int32_t N, lora_dtype_t dt, const lora_pool_t* pool, const lora_segment_t* segs,
             int32_t n_segs, Problem* out, std::string* err, const lora_slices_t* slices) {
    if (dt != LORA_BF16 && dt != LORA_F32) { *err = "unknown dtype"; return LORA_ERR_DTYPE; }
    if (T < 0 || K <= 0 || N <= 0 || n_segs < 0) { *err = "T must be >= 0, K and N > 0, n_segs >= 0"; return LORA_ERR_INVALID_ARG; }
    if (dt == LORA_BF16 && ((K % 8) != 0 || (N % 8) != 0)) {
        *err = "bf16 layers need K and N to be multiples of 8 (16-byte rows)";
        return LORA_ERR_ALIGNMENT;
    }
    if (n_segs > 0 && segs == nullptr) { *err = "segs is NULL"; return LORA_ERR_INVALID_ARG; }
    if (pool == nullptr) { *err = "pool is NULL"; return LORA_ERR_INVALID_ARG; }
    if (pool->n_adapters < 0) { *err = "pool->n_adapters < 0"; return LORA_ERR_INVALID_ARG; }
    if (pool->n_adapters > 0 && (!pool->a_off || !pool->b_off || !pool->rank || !pool->scale)) {
        *err = "pool host arrays (a_off, b_off, rank, scale) must be non-NULL";
        return LORA_ERR_INVALID_ARG;
    }
    Problem& p = *out;
    p = Problem();
    p.T = T; p.K = K; p.N = N; p.dt = dt;
    p.bounds[0] = 0;
    p.bounds[1] = N;
    if (slices != nullptr) {
        const int32_t S = slices->n_slices;
        if (S < 1 || S > LORA_MAX_SLICES) { *err = "n_slices outside [1, 4]"; return LORA_ERR_INVALID_ARG; }
        if (!slices->col_bounds) { *err = "slices->col_bounds is NULL"; return LORA_ERR_INVALID_ARG; }
        const int32_t* b = slices->col_bounds;
        if (b[0] != 0 || b[S] != N) { *err = "slice bounds must start at 0 and end at N"; return LORA_ERR_INVALID_ARG; }
        for (int32_t i = 0; i < S; ++i) {
            if (b[i + 1] <= b[i]) { *err = "slice bounds must increase strictly"; return LORA_ERR_INVALID_ARG; }
            if (i > 0 && b[i] % kBN != 0) {
                *err = "interior slice bounds must be multiples of 256";
                return LORA_ERR_INVALID_ARG;
            }
        }
        if (S > 1 && dt != LORA_BF16) { *err = "sliced layers need the bf16 path"; return LORA_ERR_DTYPE; }
        p.S = S;
        for (int32_t i = 0; i <= S; ++i) p.bounds[i] = b[i];
    }
    p.n_adapters = pool->n_adapters;
    p.a_off = pool->a_off; p.b_off = pool->b_off; p.rank = pool->rank; p.scale = pool->scale;
    for (int32_t a = 0; a < pool->n_adapters; ++a) {
        int32_t r = pool->rank[a];
        if (r < 1 || r > LORA_MAX_RANK) { *err = "adapter " + std::to_string(a) + ": rank outside [1,128]"; return LORA_ERR_RANK; }
        int64_t ao = pool->a_off[a], bo = pool->b_off[a];
        if (ao < 0 || bo < 0 || ao % K != 0 || bo % N != 0) {
            *err = "adapter " + std::to_string(a) + ": a_off must be a non-negative multiple of K and b_off of N";
            return LORA_ERR_ADAPTER;
        }
        p.rows_a = std::max<int64_t>(p.rows_a, ao / K + (int64_t)p.S * r);
        p.rows_b = std::max<int64_t>(p.rows_b, bo / N + r);
        if (p.rows_a > INT32_MAX || p.rows_b > INT32_MAX) { *err = "pool too large"; return LORA_ERR_LIMIT; }
    }
    p.segs.reserve(n_segs);
    for (int32_t i = 0; i < n_segs; ++i) {
        const lora_segment_t& s = segs[i];
        if (s.len < 0 || s.start < 0 || (int64_t)s.start + s.len > T) {
            *err = "segment " + std::to_string(i) + " lies outside [0,T)";
            return LORA_ERR_SEGMENTS;
        }
        if (s.adapter_id < -1 || s.adapter_id >= pool->n_adapters) {
            *err = "segment " + std::to_string(i) + ": adapter id out of range";
            return LORA_ERR_ADAPTER;
        }
        if (s.is_train && s.adapter_id < 0) {
            *err = "segment " + std::to_string(i) + ": fine-tuning segment on adapter -1";
            return LORA_ERR_TRAIN_BASE;
        }
        if (s.len > 0) {
            lora_segment_t c = s;
            c.is_train = s.is_train ? 1 : 0;
            p.segs.push_back(c);
        }
    }
    std::stable_sort(p.segs.begin(), p.segs.end(),
                     [](const lora_segment_t& a, const lora_segment_t& b) { return a.start < b.start; });
    int64_t at = 0;
    for (const auto& s : p.segs) {
        if (s.start != at) {
            *err = s.start < at ? "segments overlap at token " + std::to_string(s.start)
                                : "tokens " + std::to_string(at) + ".." + std::to_string(s.start - 1) + " are in no segment";
            return LORA_ERR_SEGMENTS;
        }
        at = (int64_t)s.start + s.len;
    }
    if (at != T) { *err = "segments do not cover [0,T)"; return LORA_ERR_SEGMENTS; }
    for (const auto& s : p.segs) {
        if (s.is_train) {
            p.n_train++;
            p.xa_elems += (int64_t)s.len * p.S * p.rank[s.adapter_id];
        }
    }
    if (p.n_train > kMaxTrainSegs) { *err = "more than 48 fine-tuning segments in one call"; return LORA_ERR_LIMIT; }
    if (p.xa_elems > INT32_MAX) { *err = "saved-activation buffer exceeds 2^31 elements"; return LORA_ERR_LIMIT; }
    return LORA_OK;
}

// Append one pair of tiles.  rows / row_ad: 256 entries (token row and adapter per tile row, -1 = none);
// t0, t1: the two tiles' descriptors with a_row0 / a_src / tpos0 filled in.
//
// LoRA-column layouts (chunks 16-aligned, one 8-row pool atom per 8 columns):
//   one slice:           [chunk 0 | chunk 1 | ...]
//   sliced, forward:     S regions of stride W = roundup(chunk columns, 64), region i = the chunks' slice-i
//                        columns (down-factor rows of slice i; the up-factor rows are the same in every region)
//   sliced, backward:    one adapter; its slices side by side, slice i at [i rp, i rp + r), rp = roundup(r, 16)
static void add_pair(const Problem& p, Plan* pl, const int32_t* rows, const int32_t* row_ad, const int32_t* row_aux,
                     TileDesc t0, TileDesc t1, bool backward) {
    // rows come in runs of one adapter (consecutive tokens of a segment, or gathered rows sorted by adapter): an id
    // is collected once per run, then sorted and made unique
    std::vector<int32_t> A, B;
    for (int i = 0; i < kTileM; ++i) {
        if (row_ad[i] >= 0 && (A.empty() || A.back() != row_ad[i])) A.push_back(row_ad[i]);
        const int32_t b = row_ad[kTileM + i];
        if (b >= 0 && (B.empty() || B.back() != b)) B.push_back(b);
    }
    std::sort(A.begin(), A.end());
    A.erase(std::unique(A.begin(), A.end()), A.end());
    std::sort(B.begin(), B.end());
    B.erase(std::unique(B.begin(), B.end()), B.end());
    std::vector<int32_t> onlyA, both, onlyB;
    std::set_difference(A.begin(), A.end(), B.begin(), B.end(), std::back_inserter(onlyA));
    std::set_intersection(A.begin(), A.end(), B.begin(), B.end(), std::back_inserter(both));
    std::set_difference(B.begin(), B.end(), A.begin(), A.end(), std::back_inserter(onlyB));
    std::vector<int32_t> order;
    order.insert(order.end(), onlyA.begin(), onlyA.end());
    order.insert(order.end(), both.begin(), both.end());
    order.insert(order.end(), onlyB.begin(), onlyB.end());

    const int32_t S = p.S;
    const bool side_by_side = backward && S > 1;     // backward tiles hold one adapter
    const int32_t chunk0 = int32_t(pl->chunks.size());
    int32_t zcol = 0, end_a = 0, start_b = 0;
    for (size_t c = 0; c < order.size(); ++c) {
        if (c == onlyA.size()) start_b = zcol;
        const int32_t a = order[c];
        Chunk ch{};
        ch.adapter = a;
        ch.zcol = zcol;
        ch.r = p.rank[a];
        ch.prow_a = int32_t(p.a_off[a] / p.K);
        ch.prow_b = int32_t(p.b_off[a] / p.N);
        ch.scale = p.scale[a];
        pl->chunks.push_back(ch);
        zcol += side_by_side ? S * pad16(ch.r) : pad16(ch.r);
        if (c + 1 == onlyA.size() + both.size()) end_a = zcol;
    }
    if (onlyA.size() == order.size()) start_b = zcol;
    // pool row of every 8-column atom; the padding of a chunk to 16 repeats its last atom, so every loaded row
    // stays inside the adapter's own block (sliced: the slice's own rows or the next slice's)
    const int32_t atom0 = int32_t(pl->atoms_a.size());
    std::vector<uint8_t> brk;        // per atom: starts a region padding's columns (no box runs into padding)
    const int32_t n_reg = (S > 1 && !side_by_side) ? S : 1;
    const int32_t W = (n_reg > 1) ? int32_t(cdiv(zcol, kBK) * kBK) : zcol;
    for (int32_t reg = 0; reg < n_reg; ++reg) {
        for (size_t c = 0; c < order.size(); ++c) {
            const Chunk& ch = pl->chunks[chunk0 + c];
            const int32_t last = ((ch.r + 7) / 8 - 1) * 8;
            const int32_t nsl = side_by_side ? S : 1;
            for (int32_t i = 0; i < nsl; ++i) {
                const int32_t sl = side_by_side ? i : reg;      // slice whose down-factor rows these columns hold
                for (int32_t o = 0; o < pad16(ch.r); o += 8) {
                    pl->atoms_a.push_back(ch.prow_a + sl * ch.r + std::min(o, last));
                    pl->atoms_b.push_back(ch.prow_b + std::min(o, last));
                    brk.push_back(0);
                }
            }
        }
        for (int32_t o = zcol; o < W; o += 8) {     // region padding: any in-pool row (its columns are masked)
            pl->atoms_a.push_back(pl->atoms_a.back());
            pl->atoms_b.push_back(pl->atoms_b.back());
            brk.push_back(1);
        }
    }
    // TMA boxes: runs of atoms whose pool rows follow one another (across chunks too: adapters that are neighbours
    // in the pool, in the chunks' id order), cut at 64-column blocks (relative to the tile's first LoRA column) and
    // at region padding, split greedily into 8-, 4-, 2- and 1-atom boxes.  A loader takes a box whole only when it
    // lies inside the columns it loads, so boxes may straddle the LoRA splits of an item.
    auto boxes_of = [&](const std::vector<int32_t>& rows, std::vector<int32_t>* out) {
        const size_t n = brk.size();
        for (size_t i = 0; i < n;) {
            size_t j = i + 1;
            while (j < n && (j % 8) != 0 && !brk[j] && rows[atom0 + j] == rows[atom0 + j - 1] + 8) ++j;
            size_t k = i;
            while (k < j) {
                int32_t h = 8;
                while (size_t(h) > j - k) h >>= 1;
                out->push_back(h);
                for (int32_t t = 1; t < h; ++t) out->push_back(0);
                k += size_t(h);
            }
            i = j;
        }
    };
    boxes_of(pl->atoms_a, &pl->boxes_a);
    boxes_of(pl->atoms_b, &pl->boxes_b);
    const int32_t zstride = (S == 1) ? 0 : (side_by_side ? 0 : W);
    const int32_t z_cols = n_reg * W;
    TileDesc* td[2] = {&t0, &t1};
    for (int h = 0; h < 2; ++h) {
        td[h]->chunk0 = chunk0;
        td[h]->nchunk = int32_t(order.size());
        td[h]->ext_k = zcol;
        td[h]->atom0 = atom0;
        td[h]->z_blk0 = int32_t(pl->z_blocks);
        td[h]->zstride = zstride;
        pl->z_blocks += cdiv(z_cols, kBK);
    }
    if (side_by_side) {
        // the mask of a backward sliced tile: slice i of the chunk at columns [i rp, i rp + r)
        t0.zstride = t1.zstride = order.empty() ? 0 : pad16(pl->chunks[chunk0].r);
    }
    // the shrink columns of each tile (region 0's; a forward sliced tile repeats them in every region)
    t0.sh_c0 = 0;
    t0.sh_c1 = A.empty() ? 0 : end_a;
    t1.sh_c0 = B.empty() ? zcol : start_b;
    t1.sh_c1 = zcol;
    int32_t run_ad = -1, run_rc = -1;     // the chunk of the current run's adapter
    for (int i = 0; i < 2 * kTileM; ++i) {
        int32_t rc = -1;
        if (row_ad[i] >= 0) {
            if (row_ad[i] != run_ad) {
                run_ad = row_ad[i];
                run_rc = chunk0 + int32_t(std::find(order.begin(), order.end(), run_ad) - order.begin());
            }
            rc = run_rc;
        }
        pl->rowmap.push_back(rows[i]);
        pl->rowchunk.push_back(rc);
        pl->rowaux.push_back(row_aux ? row_aux[i] : -1);
    }
    pl->tiles.push_back(t0);
    pl->tiles.push_back(t1);
}

// Shrink items of one pass, split along the reduction at boundaries that depend on the k-block count alone.
// kb_first: first k-block of the reduction (a slice's output columns, for the backward shrink over N).
// nsplit: the number of splits (0: as many as the default split length for the call's token count gives).
static void add_shrink(Plan* pl, int32_t kind, int32_t tile, int32_t n0, int32_t mma_n, int32_t nk,
                       int32_t kb_first = 0, int32_t nsplit = 0) {
    if (nsplit <= 0) nsplit = std::max<int32_t>(1, int32_t(cdiv(nk, shrink_split_kb(pl->T))));
    ShrinkUnit u{};
    u.kind = kind; u.tile = tile; u.n0 = n0; u.mma_n = mma_n; u.nsplit = nsplit;
    u.part0 = int32_t(pl->part_cols);
    for (int32_t s = 0; s < nsplit; ++s) {
        WorkItem w{};
        w.kind = kind; w.tile = tile; w.n0 = n0; w.mma_n = mma_n;
        w.kb0 = int32_t((int64_t)s * nk / nsplit);
        w.nk = int32_t((int64_t)(s + 1) * nk / nsplit) - w.kb0;
        w.kb0 += kb_first;
        w.part = u.part0 + s * mma_n;
        w.n_ext = int32_t(pl->units.size());    // shrink items carry their unit index here
        pl->items[0].push_back(w);
    }
    pl->part_cols += (int64_t)nsplit * mma_n;
    pl->units.push_back(u);
}

// Main items of the M = 256 pass: one per (tile pair, 256 output columns), bands of kBandTiles tiles sweeping all
// output columns before the next band (L2 reuse of the band's rows).  tile_of(q, nt): first tile of the pair
// that output tile (pair q, column tile nt) reads (a sliced forward reads the copy of its slice).
//
// Few output tiles (less than ~1.5 waves of CTA pairs): the K loop of every output tile is split (see
// kMainTargetItems).  The number of dense splits is the same for every tile of the call; forward LoRA splits are
// cut at chunk boundaries and hold about as many k-blocks as a dense split.
// Dense K-splits of every output tile of a launch with tiles_out output tiles and nk k-blocks (1: no split).
static int32_t dense_splits(int64_t tiles_out, int32_t nk) {
    if (tiles_out <= 0 || tiles_out >= kMainTargetItems) return 1;
    return int32_t(std::max<int64_t>(1, std::min<int64_t>({cdiv(kMainTargetItems, tiles_out), nk / 4, 16})));
}

template <class TileOf>
static void add_main_items(Plan* pl, int32_t kind, int32_t n_nt, int32_t nk, size_t n_pairs, TileOf tile_of) {
    const size_t band = kBandTiles / 2;
    const int64_t tiles_out = (int64_t)n_pairs * n_nt;
    const int32_t nsb_all = dense_splits(tiles_out, nk);
    const int32_t nsb_fwd = nsb_all;
    const bool fwd = (kind == kMainFwd);
    const bool split_all = nsb_all > 1 || (fwd && tiles_out > 0 && tiles_out < kMainTargetItems);
    // dX: when the output tiles leave a last, partly filled wave of CTA pairs, the last ones in item order are
    // split so that the last wave runs short items (backward tiles follow the fine-tuning segments in start order,
    // so which rows are split does not depend on the segment or pool order)
    int64_t tail_from = tiles_out;
    int32_t nsb_tail = 1;
    if (!split_all && kind == kMainDx) {
        const int64_t rem = tiles_out % kPairsPlanned;
        if (rem > 0 && kPairsPlanned / rem >= 2) {
            nsb_tail = int32_t(std::min<int64_t>({kPairsPlanned / rem, nk / 4, 8}));
            if (nsb_tail > 1) tail_from = tiles_out - rem;
        }
    }
    // the order of the output tiles (pair q, column tile nt): bands of kBandTiles tile rows sweeping every column
    // tile before the next band (column bands, alternating sweep directions and bands of 8 or 32 tile rows measured
    // alike)
    pl->items[1].reserve(pl->items[1].size() + (size_t)tiles_out * (split_all ? nsb_all + 2 : 1));
    int64_t o = 0;                   // output tiles emitted so far
    std::vector<int32_t> cuts;       // LoRA split bounds (Z columns) of the current pair
    for (size_t b0 = 0; b0 < n_pairs; b0 += band) {
        const size_t b1 = std::min(n_pairs, b0 + band);
        for (int32_t nt = 0; nt < n_nt; ++nt)
            for (size_t q = b0; q < b1; ++q) {
                const int32_t tile = tile_of(q, nt);
                const TileDesc& td = pl->tiles[tile];
                const bool split = split_all || o >= tail_from;
                const int32_t nsb = split_all ? nsb_all : (o >= tail_from ? nsb_tail : 1);
                cuts.assign(1, 0);
                if (split && fwd && td.ext_k > 0) {
                    // chunk-aligned LoRA splits of about one dense split's k-blocks each
                    const int32_t target = std::max<int32_t>(kBK, int32_t(cdiv(nk, nsb_fwd)) * kBK);
                    for (int32_t c = 0; c < td.nchunk; ++c) {
                        const int32_t end = (c + 1 < td.nchunk) ? pl->chunks[td.chunk0 + c + 1].zcol : td.ext_k;
                        if (end - cuts.back() >= target || c + 1 == td.nchunk) cuts.push_back(end);
                    }
                }
                const int32_t n_lora = split && fwd ? int32_t(cuts.size()) - 1 : 0;
                const int32_t nsplit = split ? nsb + n_lora : 1;
                const int32_t slot0 = int32_t(pl->main_slots);
                for (int32_t sp = 0; sp < nsplit; ++sp) {
                    WorkItem w{};
                    w.kind = kind;
                    w.tile = tile;
                    w.n0 = nt * kBN;
                    w.mma_n = kBN;
                    w.nsplit = nsplit;
                    w.split = sp;
                    w.part = slot0;
                    if (sp < nsb) {                       // dense k-blocks [kb0, kb0 + nk)
                        w.kb0 = int32_t((int64_t)sp * nk / nsb);
                        w.nk = int32_t((int64_t)(sp + 1) * nk / nsb) - w.kb0;
                    }
                    if (!split || (!fwd && sp == nsb - 1)) {   // the whole LoRA range
                        w.ext_c0 = 0;
                        w.ext_c1 = td.ext_k;
                    } else if (sp >= nsb) {               // a forward LoRA split
                        w.ext_c0 = cuts[sp - nsb];
                        w.ext_c1 = cuts[sp - nsb + 1];
                    }
                    w.n_ext = (w.ext_c1 > w.ext_c0) ? int32_t(cdiv(w.ext_c1, kBK) - w.ext_c0 / kBK) : 0;
                    pl->items[1].push_back(w);
                }
                if (nsplit > 1) {
                    pl->splits.push_back(SplitTile{tile, nt * kBN, slot0, nsplit, 0, 0, 0, 0});
                    pl->main_slots += nsplit;
                }
                ++o;
            }
    }
}

void plan_forward(const Problem& p, Plan* out) {
    Plan& pl = *out;
    pl = Plan();
    pl.T = p.T;
    // xa_save offsets of fine-tuning segments (increasing start)
    std::vector<int64_t> seg_xoff(p.segs.size(), -1);
    int64_t xo = 0;
    for (size_t i = 0; i < p.segs.size(); ++i)
        if (p.segs[i].is_train) { seg_xoff[i] = xo; xo += (int64_t)p.segs[i].len * p.S * p.rank[p.segs[i].adapter_id]; }

    // classify rows: long (windowed) or short (gathered)
    std::vector<int32_t> row_seg(p.T);
    std::vector<uint8_t> is_long(p.T, 0);
    for (size_t i = 0; i < p.segs.size(); ++i) {
        const auto& s = p.segs[i];
        bool shortseg = s.len < kShortSegment && !s.is_train;
        for (int32_t t = s.start; t < s.start + s.len; ++t) {
            row_seg[t] = int32_t(i);
            if (!shortseg) is_long[t] = 1;
        }
    }
    // per pair: token rows, their adapters and saved-activation offsets
    int32_t rows[2 * kTileM], row_ad[2 * kTileM], row_aux[2 * kTileM];
    auto fill = [&](int i, int32_t t) {
        rows[i] = t;
        row_ad[i] = -1;
        row_aux[i] = -1;
        if (t >= 0) {
            const auto& s = p.segs[row_seg[t]];
            row_ad[i] = s.adapter_id;
            if (s.is_train)
                row_aux[i] = int32_t(seg_xoff[row_seg[t]] + (int64_t)(t - s.start) * p.S * p.rank[s.adapter_id]);
        }
    };
    // 256-row windows over the long rows
    for (int32_t t = 0; t < p.T;) {
        if (!is_long[t]) { ++t; continue; }
        const int32_t w0 = t;
        for (int i = 0; i < 2 * kTileM; ++i) {
            const int32_t r = w0 + i;
            fill(i, (r < p.T && is_long[r]) ? r : -1);
        }
        TileDesc t0{}, t1{};
        t0.a_row0 = w0; t1.a_row0 = w0 + kTileM;
        t0.tpos0 = t1.tpos0 = -1;
        t0.seg = t1.seg = -1;
        add_pair(p, &pl, rows, row_ad, row_aux, t0, t1, false);
        t = w0 + 2 * kTileM;
    }
    // gathered pairs: short rows sorted by (adapter, row) -- a counting sort by adapter (base-only rows first) of
    // the short rows taken in row order
    std::vector<int32_t> gathered;
    {
        std::vector<int64_t> at(p.n_adapters + 2, 0);
        for (int32_t t = 0; t < p.T; ++t)
            if (!is_long[t]) at[p.segs[row_seg[t]].adapter_id + 2]++;
        for (size_t a = 1; a < at.size(); ++a) at[a] += at[a - 1];
        gathered.resize(at.back());
        for (int32_t t = 0; t < p.T; ++t)
            if (!is_long[t]) gathered[at[p.segs[row_seg[t]].adapter_id + 1]++] = t;
    }
    pl.g_tile0 = int32_t(pl.tiles.size());
    for (size_t g0 = 0; g0 < gathered.size(); g0 += 2 * kTileM) {
        for (int i = 0; i < 2 * kTileM; ++i) fill(i, (g0 + i < gathered.size()) ? gathered[g0 + i] : -1);
        TileDesc t0{}, t1{};
        t0.a_src = t1.a_src = 1;
        t0.a_row0 = pl.n_gtiles * kTileM;
        t1.a_row0 = (pl.n_gtiles + 1) * kTileM;
        t0.tpos0 = t1.tpos0 = -1;
        t0.seg = t1.seg = -1;
        add_pair(p, &pl, rows, row_ad, row_aux, t0, t1, false);
        pl.n_gtiles += 2;
    }
    // items: shrink passes (per slice region), then main items banded for L2 reuse
    const int32_t nk = int32_t(cdiv(p.K, kBK));
    const size_t n_orig = pl.tiles.size();
    // the shrink of the gathered decode rows runs on CUDA cores (BgmvGroup) when they are few: per group of rows
    // sharing an adapter it reads the adapter's rows of A once, where a tensor-core pass runs over the whole tile
    const bool bgmv = pl.n_gtiles > 0 && pl.n_gtiles * kTileM <= kBgmvMaxRows;
    if (bgmv) {
        const int32_t n_g = pl.n_gtiles * kTileM;
        for (int32_t g = 0; g < n_g;) {
            const int32_t idx = pl.g_tile0 * kTileM + g;
            const int32_t c = pl.rowmap[idx] < 0 ? -1 : pl.rowchunk[idx];
            int32_t n = 1;     // a run stays inside one tile; rows without an adapter (or token) form copy-only runs
            auto chunk_at = [&](int32_t i) { return pl.rowmap[i] < 0 ? -1 : pl.rowchunk[i]; };
            while (n < kBgmvRows && (g + n) % kTileM != 0 && chunk_at(idx + n) == c) ++n;
            if (c < 0) {
                pl.bgmv.push_back(BgmvGroup{g, n, -1, 0, pl.g_tile0 + g / kTileM, g % kTileM, 0, 0});
            } else {
                for (int32_t j0 = 0; j0 < p.S * pl.chunks[c].r; j0 += 8)
                    pl.bgmv.push_back(BgmvGroup{g, n, c, j0, pl.g_tile0 + g / kTileM, g % kTileM, 0, 0});
            }
            g += n;
        }
    }
    const int64_t nsplit = std::max<int64_t>(1, cdiv(nk, shrink_split_kb(p.T)));
    auto shrink_items = [&](int32_t width) {
        int64_t n = 0;
        for (size_t ti = 0; ti < n_orig; ++ti)
            if (!(bgmv && int32_t(ti) >= pl.g_tile0))
                n += p.S * cdiv(std::max(0, pl.tiles[ti].sh_c1 - pl.tiles[ti].sh_c0), width);
        return n * nsplit;
    };
    int32_t width = kPassCols;
    while (width > 64 && shrink_items(width) < kShrinkTargetItems) width /= 2;
    for (size_t ti = 0; ti < n_orig; ++ti) {
        if (bgmv && int32_t(ti) >= pl.g_tile0) continue;     // computed on CUDA cores
        const TileDesc& td = pl.tiles[ti];
        for (int32_t reg = 0; reg < p.S; ++reg) {
            const int32_t base = reg * td.zstride;
            for (int32_t c0 = base + td.sh_c0; c0 < base + td.sh_c1; c0 += width)
                add_shrink(&pl, kShrinkFwd, int32_t(ti), c0, std::min(width, base + td.sh_c1 - c0), nk);
        }
    }
    // sliced: one copy of every tile per further slice, its Z starting at that slice's region
    for (int32_t reg = 1; reg < p.S; ++reg)
        for (size_t ti = 0; ti < n_orig; ++ti) {
            TileDesc c = pl.tiles[ti];
            c.z_blk0 += reg * (c.zstride / kBK);
            c.sh_c0 = c.sh_c1 = 0;
            pl.tiles.push_back(c);
            for (int i = 0; i < kTileM; ++i) {
                pl.rowmap.push_back(pl.rowmap[ti * kTileM + i]);
                pl.rowchunk.push_back(pl.rowchunk[ti * kTileM + i]);
                pl.rowaux.push_back(pl.rowaux[ti * kTileM + i]);
            }
        }
    add_main_items(&pl, kMainFwd, int32_t(cdiv(p.N, kBN)), nk, n_orig / 2, [&](size_t q, int32_t nt) {
        const int32_t reg = p.slice_of_col(nt * kBN);
        return int32_t(reg * n_orig + 2 * q);
    });
}

// Gradient items: when they fill less of the last wave of CTAs than a split of their token ranges would, every
// item is split the same number of ways (at most 8, at least 8 token blocks a split) so that the waves fill; the
// splits' fp32 partials are summed in split order by the last split to finish.  The number of ways depends on the
// number of items and their shortest token range alone, so it does not change with the segment or pool order.
static void split_grad_items(Plan* pl) {
    std::vector<WorkItem>& items = pl->items[2];
    if (items.empty()) return;
    const int64_t G = 2 * kPairsPlanned;              // CTAs of the gradient launch
    const int64_t n = int64_t(items.size());
    int32_t min_nk = items[0].nk;
    for (const WorkItem& w : items) min_nk = std::min(min_nk, w.nk);
    int32_t ways = 1;
    double best = double(cdiv(n, G));                 // waves of whole items
    for (int32_t s = 2; s <= 8 && min_nk / s >= 8; ++s) {
        const double waves = double(cdiv(n * s, G)) / s;
        if (waves < 0.8 * best) {
            best = waves;
            ways = s;
        }
    }
    if (ways == 1) return;
    std::vector<WorkItem> out;
    out.reserve(items.size() * ways);
    for (const WorkItem& w : items) {
        ShrinkUnit u{};
        u.kind = w.kind; u.tile = w.tile; u.n0 = w.n0; u.mma_n = w.mma_n; u.nsplit = ways;
        u.part0 = int32_t(pl->part_cols);
        for (int32_t sp = 0; sp < ways; ++sp) {
            WorkItem v = w;
            v.kb0 = int32_t((int64_t)sp * w.nk / ways);
            v.nk = int32_t((int64_t)(sp + 1) * w.nk / ways) - v.kb0;
            v.nsplit = ways;
            v.split = sp;
            v.part = u.part0 + sp * w.mma_n;
            v.n_ext = int32_t(pl->units.size());     // split items carry their unit index here
            out.push_back(v);
        }
        pl->part_cols += (int64_t)ways * w.mma_n;
        pl->units.push_back(u);
    }
    items.swap(out);
}

void plan_backward(const Problem& p, bool want_dx, bool want_da, bool want_db, bool recompute, Plan* out,
                   bool per_segment) {
    Plan& pl = *out;
    pl = Plan();
    pl.T = p.T;
    // fine-tuning segments in increasing start order, grouped by adapter
    std::vector<int32_t> group_of_adapter(p.n_adapters, -1);
    std::vector<std::vector<int32_t>> members;
    std::vector<lora_segment_t> tr;
    for (const auto& s : p.segs)
        if (s.is_train) tr.push_back(s);
    for (size_t i = 0; i < tr.size(); ++i) {
        int32_t a = tr[i].adapter_id;
        if (group_of_adapter[a] < 0) {
            group_of_adapter[a] = int32_t(members.size());
            members.emplace_back();
        }
        members[group_of_adapter[a]].push_back(int32_t(i));
    }
    // train-segment records ordered by group, then start (the fixed summation order of dA/dB)
    int64_t tpos = 0, xo = 0;
    std::vector<int32_t> tpos_of(tr.size()), xoff_of(tr.size());
    for (size_t i = 0; i < tr.size(); ++i) {
        tpos_of[i] = int32_t(tpos);
        tpos += cdiv(tr[i].len, 2 * kTileM) * 2 * kTileM;
        xoff_of[i] = int32_t(xo);
        xo += (int64_t)tr[i].len * p.S * p.rank[tr[i].adapter_id];
    }
    pl.tcols = tpos;
    for (size_t g = 0; g < members.size(); ++g) {
        GradGroup gg{};
        int32_t a = tr[members[g][0]].adapter_id;
        gg.adapter = a;
        gg.r = p.rank[a];
        gg.seg0 = int32_t(pl.tsegs.size());
        gg.nseg = int32_t(members[g].size());
        gg.prow_a = int32_t(p.a_off[a] / p.K);
        gg.prow_b = int32_t(p.b_off[a] / p.N);
        gg.scale = p.scale[a];
        gg.nslice = p.S;
        for (int32_t i : members[g])
            pl.tsegs.push_back(TrainSeg{tr[i].start, tr[i].len, tpos_of[i], int32_t(g), xoff_of[i], p.S * gg.r, i, 0});
        pl.groups.push_back(gg);
    }
    // one pair of tiles per 256 rows of each fine-tuning segment
    for (size_t i = 0; i < tr.size(); ++i) {
        for (int32_t b = 0; b < tr[i].len; b += 2 * kTileM) {
            int32_t rows[2 * kTileM], row_ad[2 * kTileM];
            for (int k = 0; k < 2 * kTileM; ++k) {
                const bool v = b + k < tr[i].len;
                rows[k] = v ? tr[i].start + b + k : -1;
                row_ad[k] = v ? tr[i].adapter_id : -1;
            }
            TileDesc t0{}, t1{};
            t0.a_row0 = tr[i].start + b;
            t1.a_row0 = tr[i].start + b + kTileM;
            t0.tpos0 = tpos_of[i] + b;
            t1.tpos0 = tpos_of[i] + b + kTileM;
            t0.seg = t1.seg = int32_t(i);
            add_pair(p, &pl, rows, row_ad, nullptr, t0, t1, true);
        }
    }
    const bool need_dyb = want_dx || want_da;
    const bool need_xa = want_db && (recompute || per_segment);
    // The backward shrink passes in launch order: per tile its dY B^T passes (one per slice), then its x A passes.
    struct Pass {
        int32_t kind, tile, n0, mma_n, nk, kb_first;
    };
    std::vector<Pass> passes;
    for (size_t ti = 0; ti < pl.tiles.size(); ++ti) {
        const TileDesc& td = pl.tiles[ti];
        if (td.sh_c1 <= td.sh_c0) continue;      // the empty second tile of a short segment's pair
        if (need_dyb) {
            if (p.S == 1) {
                passes.push_back({kShrinkDyb, int32_t(ti), td.sh_c0, td.sh_c1 - td.sh_c0, int32_t(cdiv(p.N, kBK)), 0});
            } else {
                // slice i: dY's slice-i columns against the up factor's slice-i columns, into LoRA columns
                // [i rp, (i+1) rp)
                for (int32_t i = 0; i < p.S; ++i) {
                    const int32_t kb_a = p.bounds[i] / kBK, kb_b = int32_t(cdiv(p.bounds[i + 1], kBK));
                    passes.push_back({kShrinkDyb, int32_t(ti), i * td.zstride, td.zstride, kb_b - kb_a, kb_a});
                }
            }
        }
        if (need_xa)
            for (int32_t c0 = td.sh_c0; c0 < td.sh_c1; c0 += kPassCols)
                passes.push_back({kShrinkXa, int32_t(ti), c0, std::min(kPassCols, td.sh_c1 - c0),
                                  int32_t(cdiv(p.K, kBK)), 0});
    }
    // The x A passes keep the forward's splits, so that a recomputed xA equals the saved one bit for bit.  The
    // dY B^T passes of an unsliced layer (all of one length) may take another split count, from half to twice
    // the default, when the default's items fill at least one wave of 2 x kPairsPlanned CTAs and leave the last
    // one less than half full (320 items of 16 k-blocks on 152 CTAs end after 48 k-blocks; 288, with the dY B^T
    // passes in 20-k-block pieces, after 40): the count whose greedy list schedule of the whole launch by the
    // items' estimated costs ends first, if it ends before the default's.  It depends on the passes' shapes
    // alone, not on the segment or pool order.
    const int32_t kb_default = shrink_split_kb(p.T);
    const int64_t G = 2 * kPairsPlanned;
    auto default_splits = [&](int32_t nk) { return std::max<int32_t>(1, int32_t(cdiv(nk, kb_default))); };
    auto n_items = [&](int32_t dyb_splits) {
        int64_t n = 0;
        for (const Pass& ps : passes) n += (ps.kind == kShrinkDyb) ? dyb_splits : default_splits(ps.nk);
        return n;
    };
    // the end of the greedy schedule, or `bound` as soon as a CTA's load reaches it
    std::vector<int64_t> load(G);
    auto schedule_end = [&](int32_t dyb_splits, int64_t bound) {
        std::fill(load.begin(), load.end(), 0);     // a min-heap of CTA loads
        for (const Pass& ps : passes) {
            const int32_t ns = (ps.kind == kShrinkDyb) ? dyb_splits : default_splits(ps.nk);
            for (int32_t sp = 0; sp < ns; ++sp) {
                WorkItem w{};
                w.kind = ps.kind; w.mma_n = ps.mma_n;
                w.nk = int32_t((int64_t)(sp + 1) * ps.nk / ns - (int64_t)sp * ps.nk / ns);
                std::pop_heap(load.begin(), load.end(), std::greater<int64_t>());
                load.back() += item_cost(w);
                if (load.back() >= bound) return bound;
                std::push_heap(load.begin(), load.end(), std::greater<int64_t>());
            }
        }
        return *std::max_element(load.begin(), load.end());
    };
    int32_t dyb_splits = 0;                  // 0: the default
    if (need_dyb && p.S == 1 && !passes.empty()) {
        const int32_t nk = int32_t(cdiv(p.N, kBK)), s0 = default_splits(nk);
        // searched only when the default fills a wave and leaves the last one less than half full, among the
        // two counts whose last waves are fullest (the fewer items first on a tie)
        auto fill = [&](int32_t ns) { const int64_t r = n_items(ns) % G; return r == 0 ? G : r; };
        if (n_items(s0) >= G && 2 * fill(s0) < G) {
            std::vector<std::pair<int64_t, int32_t>> cand;     // (-fill, count)
            for (int32_t ns = std::max(1, s0 / 2); ns <= std::min(2 * s0, std::max(1, nk / 4)); ++ns)
                if (ns != s0) cand.push_back({-fill(ns), ns});
            std::sort(cand.begin(), cand.end());
            int64_t best = schedule_end(s0, INT64_MAX);
            for (size_t i = 0; i < cand.size() && i < 2; ++i) {
                const int64_t e = schedule_end(cand[i].second, best);
                if (e < best) { best = e; dyb_splits = cand[i].second; }
            }
        }
    }
    for (const Pass& ps : passes)
        add_shrink(&pl, ps.kind, ps.tile, ps.n0, ps.mma_n, ps.nk, ps.kb_first, ps.kind == kShrinkDyb ? dyb_splits : 0);
    if (want_dx)
        add_main_items(&pl, kMainDx, int32_t(cdiv(p.K, kBN)), int32_t(cdiv(p.N, kBK)), pl.tiles.size() / 2,
                       [](size_t q, int32_t) { return int32_t(2 * q); });
    for (size_t g = 0; g < pl.groups.size(); ++g) {
        const GradGroup& gg = pl.groups[g];
        int32_t kb = 0;
        for (int32_t q = 0; q < gg.nseg; ++q) kb += int32_t(cdiv(pl.tsegs[gg.seg0 + q].len, kBK));
        if (want_db)
            for (int32_t i = 0; i < p.S; ++i)              // slice i's columns of dB read slice i's rows of xA^T
                for (int32_t m0 = p.bounds[i]; m0 < p.bounds[i + 1]; m0 += kTileM) {
                    WorkItem w{};
                    w.kind = kGradDb; w.tile = int32_t(g); w.n0 = m0; w.nk = kb; w.mma_n = pad16(gg.r);
                    w.j0 = i * gg.r;
                    pl.items[2].push_back(w);
                }
        if (want_da)
            for (int32_t m0 = 0; m0 < p.K; m0 += kTileM)
                for (int32_t j0 = 0; j0 < p.S * gg.r; j0 += kPassCols) {   // all slices' rows of the A block
                    WorkItem w{};
                    w.kind = kGradDa; w.tile = int32_t(g); w.n0 = m0; w.nk = kb;
                    w.mma_n = std::min(kPassCols, pad16(p.S * gg.r - j0));
                    w.j0 = j0;
                    pl.items[2].push_back(w);
                }
    }
    split_grad_items(&pl);
}

int check_plan(const Problem& p, const Plan& pl, bool backward, std::string* err) {
    const int64_t nt = int64_t(pl.tiles.size());
    const int64_t n_chunks = int64_t(pl.chunks.size());
    const int64_t n_atoms = int64_t(pl.atoms_a.size());
    const int64_t g_rows = int64_t(pl.n_gtiles) * kTileM;
    const int64_t out_cols = backward ? p.K : p.N;
    const int64_t kb_main = cdiv(backward ? p.N : p.K, kBK);
    auto bad = [&](const std::string& what) {
        *err = "plan check: " + what;
        return LORA_ERR_BOUNDS;
    };
    if (int64_t(pl.rowmap.size()) != nt * kTileM || int64_t(pl.rowchunk.size()) != nt * kTileM ||
        int64_t(pl.rowaux.size()) != nt * kTileM || pl.atoms_b.size() != pl.atoms_a.size() ||
        pl.boxes_a.size() != pl.atoms_a.size() || pl.boxes_b.size() != pl.atoms_a.size())
        return bad("per-row or per-atom tables of the wrong length");
    // LoRA columns of a tile's Z (all slice regions of a forward sliced tile)
    auto z_cols = [&](const TileDesc& td) -> int64_t {
        return (!backward && p.S > 1) ? int64_t(p.S) * td.zstride : td.ext_k;
    };
    for (int64_t i = 0; i < nt; ++i) {
        const TileDesc& td = pl.tiles[i];
        auto at = [&] { return "tile " + std::to_string(i) + ": "; };   // built only for a report
        // a window's second tile may start past the last row (its rows then read as zero)
        if (td.a_src == 0 ? (td.a_row0 < 0 || td.a_row0 >= p.T + kTileM) : (td.a_row0 < 0 || td.a_row0 + kTileM > g_rows))
            return bad(at() + "row window outside its source");
        if (td.chunk0 < 0 || td.nchunk < 0 || td.chunk0 + td.nchunk > n_chunks) return bad(at() + "chunk range");
        if (td.ext_k < 0 || td.ext_k % 16 != 0) return bad(at() + "LoRA columns not a multiple of 16");
        if (td.atom0 < 0 || td.atom0 + cdiv(z_cols(td), 8) > n_atoms) return bad(at() + "atom range");
        if (td.z_blk0 < 0 || td.z_blk0 + cdiv(td.ext_k, kBK) > pl.z_blocks) return bad(at() + "Z blocks");
        if (td.sh_c0 < 0 || td.sh_c0 > td.sh_c1 || td.sh_c1 > td.ext_k) return bad(at() + "shrink columns");
        if (backward && (td.tpos0 < 0 || td.tpos0 + kTileM > pl.tcols || td.seg < 0 ||
                         td.seg >= int32_t(pl.tsegs.size())))
            return bad(at() + "transposed-buffer columns or segment");
        for (int r = 0; r < kTileM; ++r) {
            const int64_t k = i * kTileM + r;
            const int32_t t = pl.rowmap[k], c = pl.rowchunk[k], aux = pl.rowaux[k];
            if (t < -1 || t >= p.T) return bad(at() + "row " + std::to_string(r) + " maps outside [0, T)");
            if (c != -1 && (c < td.chunk0 || c >= td.chunk0 + td.nchunk)) return bad(at() + "row chunk outside the tile");
            if (aux != -1) {
                if (c < 0) return bad(at() + "saved-activation offset on a row without an adapter");
                if (aux < 0 || aux + int64_t(p.S) * pl.chunks[c].r > p.xa_elems) return bad(at() + "saved-activation offset");
            }
        }
    }
    // an atom is loaded as an 8-row TMA box (or the first of a taller box's runs of consecutive atoms); a rank that
    // is not a multiple of 8 rounds the last atom up, and rows past the pool's end read as zero, so what must hold
    // is that every atom starts inside the pool and a box's atoms follow one another
    for (int64_t i = 0; i < n_atoms; ++i) {
        const int32_t ra = pl.atoms_a[i], rb = pl.atoms_b[i];
        if (ra < 0 || ra >= p.rows_a || rb < 0 || rb >= p.rows_b)
            return bad("atom " + std::to_string(i) + ": starts outside the pool");
        for (int pass = 0; pass < 2; ++pass) {
            const std::vector<int32_t>& rows = pass ? pl.atoms_b : pl.atoms_a;
            const int32_t box = (pass ? pl.boxes_b : pl.boxes_a)[i];
            if (box < 0 || box > 8 || i + box > n_atoms) return bad("atom " + std::to_string(i) + ": box size");
            for (int32_t k = 1; k < box; ++k)
                if (rows[i + k] != rows[i] + 8 * k) return bad("atom " + std::to_string(i) + ": box of unrelated rows");
        }
    }
    for (int64_t c = 0; c < n_chunks; ++c) {
        const Chunk& ch = pl.chunks[c];
        if (ch.adapter < 0 || ch.adapter >= p.n_adapters || ch.r != p.rank[ch.adapter] || ch.zcol % 16 != 0 ||
            ch.prow_a < 0 || ch.prow_a + int64_t(p.S) * ch.r > p.rows_a || ch.prow_b < 0 || ch.prow_b + ch.r > p.rows_b)
            return bad("chunk " + std::to_string(c));
    }
    for (size_t u = 0; u < pl.units.size(); ++u) {
        const ShrinkUnit& su = pl.units[u];
        const bool grad = su.kind == kGradDb || su.kind == kGradDa;
        const int64_t n_tiles = grad ? int64_t(pl.groups.size()) : nt;    // a gradient unit's tile is its group
        if (su.tile < 0 || su.tile >= n_tiles || su.nsplit < 1 || su.part0 < 0 ||
            su.part0 + int64_t(su.nsplit) * su.mma_n > pl.part_cols)
            return bad("shrink unit " + std::to_string(u));
    }
    for (int k = 0; k < 3; ++k) {
        for (size_t j = 0; j < pl.items[k].size(); ++j) {
            const WorkItem& w = pl.items[k][j];
            auto at = [&] { return "item " + std::to_string(k) + "." + std::to_string(j) + ": "; };
            if (w.mma_n < 16 || w.mma_n > kPassCols || w.mma_n % 16 != 0) return bad(at() + "MMA N");
            if (w.kind == kMainFwd || w.kind == kMainDx) {
                if (w.tile < 0 || w.tile + 1 >= nt) return bad(at() + "tile pair");
                if (w.n0 < 0 || w.n0 >= out_cols) return bad(at() + "output columns");
                if (w.kb0 < 0 || w.nk < 0 || w.kb0 + w.nk > kb_main) return bad(at() + "k-blocks");
                const int32_t ek = pl.tiles[w.tile].ext_k;
                if (w.ext_c0 < 0 || w.ext_c0 > w.ext_c1 || w.ext_c1 > ek) return bad(at() + "LoRA columns");
                if (w.ext_c0 / kBK + w.n_ext > cdiv(ek, kBK)) return bad(at() + "LoRA k-blocks");
                if (w.nsplit > 1 && (w.part < 0 || w.part + w.split >= pl.main_slots)) return bad(at() + "split slot");
            } else if (w.kind == kGradDb || w.kind == kGradDa) {
                if (w.tile < 0 || w.tile >= int32_t(pl.groups.size())) return bad(at() + "gradient group");
                const GradGroup& g = pl.groups[w.tile];
                if (w.n0 < 0 || w.n0 >= (w.kind == kGradDb ? p.N : p.K)) return bad(at() + "gradient rows");
                if (w.j0 < 0 || w.j0 + w.mma_n > int64_t(p.S) * LORA_MAX_RANK) return bad(at() + "transposed rows");
                if (w.kind == kGradDa && w.j0 >= int64_t(g.nslice) * g.r) return bad(at() + "down-factor rows");
                if (g.seg0 < 0 || g.nseg < 1 || g.seg0 + g.nseg > int32_t(pl.tsegs.size()))
                    return bad(at() + "gradient group segments");
                int64_t blocks = 0;                  // token blocks of the group's segments
                for (int32_t q = 0; q < g.nseg; ++q) blocks += cdiv(pl.tsegs[g.seg0 + q].len, kBK);
                if (w.kb0 < 0 || w.nk < 1 || w.kb0 + w.nk > blocks) return bad(at() + "token blocks");
                if (w.nsplit > 1) {
                    if (w.n_ext < 0 || w.n_ext >= int32_t(pl.units.size()) || pl.units[w.n_ext].kind != w.kind ||
                        pl.units[w.n_ext].tile != w.tile || pl.units[w.n_ext].nsplit != w.nsplit ||
                        w.split < 0 || w.split >= w.nsplit)
                        return bad(at() + "split unit");
                    const ShrinkUnit& su = pl.units[w.n_ext];
                    if (su.mma_n != w.mma_n || w.part != su.part0 + w.split * w.mma_n)
                        return bad(at() + "partial columns");
                }
            } else {
                if (w.tile < 0 || w.tile >= nt) return bad(at() + "tile");
                if (w.n_ext < 0 || w.n_ext >= int32_t(pl.units.size()) || pl.units[w.n_ext].tile != w.tile)
                    return bad(at() + "shrink unit");
                const TileDesc& td = pl.tiles[w.tile];
                const int64_t kb_all = cdiv(w.kind == kShrinkDyb ? p.N : p.K, kBK);
                if (w.kb0 < 0 || w.nk < 1 || w.kb0 + w.nk > kb_all) return bad(at() + "k-blocks");
                if (w.n0 < 0 || w.n0 + w.mma_n > cdiv(z_cols(td), 16) * 16 || td.atom0 + (w.n0 + w.mma_n) / 8 > n_atoms)
                    return bad(at() + "LoRA columns");
                if (w.part < 0 || w.part + w.mma_n > pl.part_cols) return bad(at() + "partial columns");
                if (w.kind != kShrinkXa && td.z_blk0 + cdiv(w.n0 + w.mma_n, kBK) > pl.z_blocks) return bad(at() + "Z blocks");
            }
        }
    }
    for (size_t i = 0; i < pl.splits.size(); ++i) {
        const SplitTile& st = pl.splits[i];
        if (st.tile < 0 || st.tile + 1 >= nt || st.n0 < 0 || st.n0 >= out_cols || st.part < 0 ||
            st.part + st.nsplit > pl.main_slots)
            return bad("split tile " + std::to_string(i));
    }
    for (size_t i = 0; i < pl.bgmv.size(); ++i) {
        const BgmvGroup& g = pl.bgmv[i];
        auto at = [&] { return "decode-shrink unit " + std::to_string(i) + ": "; };
        if (g.g_row0 < 0 || g.n_rows < 1 || g.n_rows > kBgmvRows || g.g_row0 + g.n_rows > g_rows) return bad(at() + "rows");
        if (g.tile < pl.g_tile0 || g.tile >= nt || g.row0 < 0 || g.row0 + g.n_rows > kTileM) return bad(at() + "tile rows");
        if (g.chunk >= 0) {
            if (g.chunk >= n_chunks) return bad(at() + "chunk");
            const Chunk& ch = pl.chunks[g.chunk];
            if (g.j0 < 0 || g.j0 >= int64_t(p.S) * ch.r) return bad(at() + "LoRA columns");
            const TileDesc& td = pl.tiles[g.tile];
            const int64_t last = int64_t(p.S - 1) * td.zstride + ch.zcol + ch.r;   // one past the last Z column
            if (last > cdiv(z_cols(td), kBK) * kBK) return bad(at() + "Z columns");
        }
    }
    for (size_t q = 0; q < pl.tsegs.size(); ++q) {
        const TrainSeg& s = pl.tsegs[q];
        if (s.start < 0 || s.start + s.len > p.T || s.tpos0 < 0 || s.tpos0 + cdiv(s.len, 2 * kTileM) * 2 * kTileM > pl.tcols ||
            s.xoff < 0 || s.xoff + int64_t(s.len) * s.r > p.xa_elems || s.group < 0 || s.group >= int32_t(pl.groups.size()))
            return bad("fine-tuning segment " + std::to_string(q));
    }
    for (size_t g = 0; g < pl.groups.size(); ++g) {
        const GradGroup& gg = pl.groups[g];
        if (gg.seg0 < 0 || gg.seg0 + gg.nseg > int32_t(pl.tsegs.size()) || gg.prow_a < 0 ||
            gg.prow_a + int64_t(gg.nslice) * gg.r > p.rows_a || gg.prow_b < 0 || gg.prow_b + gg.r > p.rows_b)
            return bad("gradient group " + std::to_string(g));
    }
    return LORA_OK;
}

static int64_t item_cost(const WorkItem& w) {
    // rough cycles per k-block: the larger of its TMA bytes at ~64 B/cycle and its MMA time (~2.7 cycles per N
    // column for M = 128, K = 64)
    int64_t bytes = 0;
    switch (w.kind) {
        case kMainFwd:
        case kMainDx: bytes = kTileM * kBK * 2 + kBN * kBK * 2; break;
        default: bytes = kTileM * kBK * 2 + (int64_t)w.mma_n * kBK * 2; break;
    }
    const int64_t per = std::max<int64_t>(bytes / 64, (27 * (int64_t)w.mma_n) / 10);
    int64_t c = (int64_t)w.nk * per;
    if (w.kind == kMainFwd || w.kind == kMainDx) c += (int64_t)w.n_ext * per;   // (shrink items: n_ext = unit)
    return c + 2000;
}

int64_t item_cost_estimate(const WorkItem& w) { return item_cost(w); }

void assign_items(const std::vector<WorkItem>& items, const Plan&, int G, std::vector<int32_t>* off,
                  std::vector<int32_t>* list) {
    // each item goes to the least-loaded CTA (ties: lowest index), found in a tournament tree over the CTAs: a node
    // holds the CTA with the least (load, index) below it, and an assignment replays only the grown leaf's path
    int P2 = 1;
    while (P2 < G) P2 <<= 1;
    std::vector<int64_t> load(G, 0);
    std::vector<int32_t> win(2 * (size_t)P2, -1);      // -1: no CTA below
    auto better = [&](int32_t a, int32_t b) {
        if (a < 0) return b;
        if (b < 0) return a;
        return (load[b] < load[a] || (load[b] == load[a] && b < a)) ? b : a;
    };
    for (int c = 0; c < G; ++c) win[P2 + c] = c;
    for (int n = P2 - 1; n >= 1; --n) win[n] = better(win[2 * n], win[2 * n + 1]);
    std::vector<int32_t> owner(items.size());
    std::vector<int32_t> count(G + 1, 0);
    for (size_t i = 0; i < items.size(); ++i) {
        const int32_t c = win[1];
        owner[i] = c;
        count[c + 1]++;
        load[c] += item_cost(items[i]);
        for (int n = (P2 + c) >> 1; n >= 1; n >>= 1) win[n] = better(win[2 * n], win[2 * n + 1]);
    }
    off->assign(G + 1, 0);
    for (int c = 0; c < G; ++c) (*off)[c + 1] = (*off)[c] + count[c + 1];
    list->assign(items.size(), 0);
    std::vector<int32_t> at(off->begin(), off->end() - 1);
    for (size_t i = 0; i < items.size(); ++i) (*list)[at[owner[i]]++] = int32_t(i);
}

size_t simt_scratch_bytes(const Problem& p) {
    // per-token adapter ids, adapter records, segment records, then xA and dY B^T scratch [T, 128] each
    return align256(sizeof(int32_t) * (size_t)p.T) + align256(32 * (size_t)(p.n_adapters + 1)) +
           align256(32 * (size_t)(p.segs.size() + 1)) + 2 * align256(sizeof(float) * (size_t)p.T * 128);
}

Layout layout_of(const Problem& p, const Plan& pl, bool backward) {
    Layout L;
    size_t at = 0;
    auto take = [&](size_t bytes) { size_t o = at; at = align256(at + bytes); return o; };
    L.status = take(256);
    L.counters = take(sizeof(int32_t) * 4 * pl.units.size());
    L.zero_end = at;
    L.tiles = take(sizeof(TileDesc) * pl.tiles.size());
    L.chunks = take(sizeof(Chunk) * pl.chunks.size());
    L.rowmap = take(sizeof(int32_t) * pl.rowmap.size());
    L.rowchunk = take(sizeof(int32_t) * pl.rowchunk.size());
    L.rowaux = take(sizeof(int32_t) * pl.rowaux.size());
    L.groups = take(sizeof(GradGroup) * pl.groups.size());
    L.tsegs = take(sizeof(TrainSeg) * pl.tsegs.size());
    L.atoms_a = take(sizeof(int32_t) * pl.atoms_a.size());
    L.atoms_b = take(sizeof(int32_t) * pl.atoms_b.size());
    L.boxes_a = take(sizeof(int32_t) * pl.boxes_a.size());
    L.boxes_b = take(sizeof(int32_t) * pl.boxes_b.size());
    L.units = take(sizeof(ShrinkUnit) * pl.units.size());
    L.seg_flags = take(sizeof(int32_t) * ((size_t)p.n_train + 1));
    L.splits = take(sizeof(SplitTile) * pl.splits.size());
    L.bgmv = take(sizeof(BgmvGroup) * pl.bgmv.size());
    for (int k = 0; k < 3; ++k) {
        L.items[k] = take(sizeof(WorkItem) * pl.items[k].size());
        L.cta_off[k] = take(sizeof(int32_t) * (std::max<size_t>(kMaxCtas, pl.items[k].size()) + 1));
    }
    L.plan_end = at;
    if (p.dt == LORA_BF16) {
        L.xg = take((size_t)pl.n_gtiles * kTileM * p.K * 2);
        L.z = take((size_t)pl.z_blocks * kZBlockBytes);
        L.part = take((size_t)pl.part_cols * kTileM * sizeof(float));
        L.part_main = take((size_t)pl.main_slots * 2 * kMainPartialFloats * sizeof(float));
        if (backward) {
            L.xat = take((size_t)p.S * LORA_MAX_RANK * pl.tcols * 2);
            L.dybt = take((size_t)p.S * LORA_MAX_RANK * pl.tcols * 2);
        }
    } else {
        L.simt = take(simt_scratch_bytes(p));
    }
    L.total = at;
    return L;
}

}  // namespace lora
