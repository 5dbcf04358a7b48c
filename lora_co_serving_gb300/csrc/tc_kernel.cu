// tc_kernel.cu -- persistent tcgen05 / TMEM / TMA kernel for every dense contraction of the layer.
//
// One kernel body runs all work-item kinds of a launch (see common.h):
//   shrink  : [128 tile rows] x [LoRA columns]  = x A^T  (or dY B^T)      -> Z / xa_save / transposed copies
//   main    : [128 tile rows] x [256 outputs]   = x Wt^T + Z Bstack       -> y       (forward)
//                                               = dY Wt  + Z Astack       -> dX      (backward)
//   grad    : [128 of N or K] x [r]             = dY^T xA  or  x^T dYB    -> dB, dA  (fp32)
// The expand of the LoRA layer ("DeltaServe: Host-Agnostic Co-Serving of Inference and Fine-Tuning for LLMs",
// section 2.2: W_eff = W + BA) is carried out as extra K-steps of the main GEMM over the tile's Z matrix
// (s_a * x A_a, masked to each row's own adapter) against the stacked rows of the tile's adapters, so the
// LoRA term accumulates in the same TMEM accumulator as x W and y is written once.
//
// Roles (192 threads, one CTA per SM, persistent over a host-assigned item list):
//   warp 0, lane 0 : TMA producer (cp.async.bulk.tensor into a 4-stage ring of 48 KB stages)
//   warp 1         : TMEM allocation; lane 0 issues tcgen05.mma (M=128) and tcgen05.commit
//   warps 2..5     : epilogue (tcgen05.ld from the double-buffered accumulator, conversion, stores)
// Every wait is bounded: on timeout the CTA records LORA_ERR_TIMEOUT in the status word and all roles stop.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.h"
#include "tc_kernel.h"

#include <utility>

namespace lora {

namespace {

constexpr int kABytes = kTileM * kBK * 2;            // 16 KB: 128 rows x 64 bf16
constexpr int kBBytes = kBN * kBK * 2;               // 32 KB: 256 rows x 64 bf16
constexpr int kStageBytes = kABytes + kBBytes;
// 1-CTA items of at most 64 LoRA columns (shrink passes, dA/dB): two k-blocks per stage, block s at s * kSubBytes
// (A: 16 KB, then B: up to 8 KB), so that twice the bytes are in flight
constexpr int kSubBytes = kABytes + 64 * kBK * 2;    // 24 KB
static_assert(2 * kSubBytes <= kStageBytes, "two k-blocks must fit a stage");
#ifndef LORA_GRAD_PACK
#define LORA_GRAD_PACK 1
#endif
#ifndef LORA_SHRINK_PACK
#define LORA_SHRINK_PACK 1
#endif
// 16-column groups a split finalize loads per round (1 or 2)
#ifndef LORA_FINALIZE_GROUPS
#define LORA_FINALIZE_GROUPS 2
#endif
__device__ __forceinline__ int grad_blocks_per_stage(int mma_n) { return (LORA_GRAD_PACK && mma_n <= 64) ? 2 : 1; }
__device__ __forceinline__ int shrink_blocks_per_stage(int mma_n) {
    return (LORA_SHRINK_PACK && mma_n <= 64) ? 2 : 1;
}
constexpr int kThreads = 192;
// Limit of every bounded wait (ns) on this device: 1 s unless lora_set_wait_limit changed it
__device__ uint64_t g_wait_limit_ns = 1000000000ull;
constexpr uint32_t kTmemCols = 512;                   // two 256-column fp32 accumulators

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ uint64_t global_timer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// try_wait that lets the hardware suspend the thread for up to `ns` nanoseconds while the phase is incomplete (it
// resumes as soon as the phase completes): for waits that are usually long, so that the waiting warp does not take
// issue slots from the warps it shares a scheduler with
__device__ __forceinline__ bool mbar_try_wait_hint(uint32_t bar, uint32_t parity, uint32_t ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(ns)
        : "memory");
    return ok != 0;
}

// Bounded wait on an mbarrier phase.  Returns false when the CTA is aborting (this wait timed out, or
// another role's did).  suspend_ns > 0: hinted try_wait (see mbar_try_wait_hint).
__device__ __noinline__ bool wait_phase_slow(uint32_t bar, uint32_t parity, volatile int* abort_flag, int32_t* status,
                                             uint32_t suspend_ns = 0) {
    const uint64_t t0 = global_timer();
    const uint64_t limit = g_wait_limit_ns;
    for (uint32_t spin = 1;; ++spin) {
        if (suspend_ns ? mbar_try_wait_hint(bar, parity, suspend_ns) : mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if ((spin & 31u) == 0 && global_timer() - t0 > limit) {
            *abort_flag = 1;
            atomicCAS(status, 0, LORA_ERR_TIMEOUT);
            return false;
        }
    }
}
// LORA_DEBUG_CHECKS: a store index derived from the plan is checked against its buffer's extent; a failing check
// records LORA_ERR_BOUNDS in the status word and the caller skips the store.
__device__ __forceinline__ bool dbg_ok(int32_t debug, int32_t* status, int64_t idx, int64_t extent) {
    if (!debug || (idx >= 0 && idx < extent)) return true;
    atomicCAS(status, 0, LORA_ERR_BOUNDS);
    return false;
}

// The first test of the phase is inlined, so a wait that is already satisfied costs no call (a call would also
// make every load still in flight complete first).
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int* abort_flag, int32_t* status) {
    if (mbar_try_wait(bar, parity)) return true;
    return wait_phase_slow(bar, parity, abort_flag, status);
}
// The epilogue's wait for a finished accumulator (one per item: usually long)
constexpr uint32_t kLongWaitNs = 20000;
__device__ __forceinline__ bool wait_phase_long(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                                int32_t* status) {
    if (mbar_try_wait(bar, parity)) return true;
    return wait_phase_slow(bar, parity, abort_flag, status, kLongWaitNs);
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int32_t c0, int32_t c1,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

// Programmatic dependent launch: the kernels of a call are launched so that each may start (its prologue: barrier
// setup, TMEM allocation) while the previous one drains; this wait holds the CTA until every earlier kernel of the
// stream has finished and its writes are visible, before anything it produced (or the caller's inputs) is read.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor, 128-byte swizzle, sm_100-family layout (version field = 1).
//   K-major operand: rows of 128 B, 8-row groups SBO apart (LBO unused).
//   MN-major operand: 64-element (128 B) MN atoms LBO apart, 8-row K groups SBO apart.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor, kind::f16: bf16 A and B, fp32 accumulator, M x N, operand majors (0 = K, 1 = MN).
__device__ __forceinline__ uint32_t instr_desc(int m, int n, int a_mn, int b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
           ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

struct Ring {
    int stage = 0;
    uint32_t phase = 0;
    __device__ __forceinline__ void next() {
        if (++stage == kStages) { stage = 0; phase ^= 1u; }
    }
};

// Lane 0 of the producer warp waits for the ring slot to be free and arms its barrier with the stage's byte
// count; the result is shared with the warp, whose 32 lanes then issue the stage's loads in parallel.
__device__ __forceinline__ bool acquire_stage(const Ring& ring, uint32_t bar_full, uint32_t bar_empty, uint32_t bytes,
                                              int lane, volatile int* abort_flag, int32_t* status) {
    int ok = 1;
    if (lane == 0) {
        ok = wait_phase(bar_empty + ring.stage * 8, ring.phase ^ 1u, abort_flag, status) ? 1 : 0;
        if (ok) mbar_expect_tx(bar_full + ring.stage * 8, bytes);
    }
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// An x A recompute item of a fine-tuning segment whose saved xA the flag table marks as usable: every role skips
// it (no stage, no accumulator), so the three roles stay in step.
__device__ __forceinline__ bool skipped_item(const KParams& P, const WorkItem& w) {
    return w.kind == kShrinkXa && P.seg_flags != nullptr && P.seg_flags[P.tiles[w.tile].seg] != 0;
}

// --------------------------------------------------------------------------------------------- producer (warp 0)
__device__ void run_producer(const KParams& P, uint8_t* smem, uint32_t bar_full, uint32_t bar_empty, int i0, int i1,
                             volatile int* abort_flag) {
    const int lane = threadIdx.x & 31;
    Ring ring;
    for (int ii = i0; ii < i1; ++ii) {
        const WorkItem w = P.items[ii];
        if (skipped_item(P, w)) continue;
        if (w.kind == kGradDb || w.kind == kGradDa) {
            // A: [128 of N or K] x 64 tokens, MN-major (two 64-wide boxes); B: r_pad rows of xA^T / dYB^T.  Items
            // of at most 64 LoRA columns take two token blocks per stage
            const GradGroup g = P.groups[w.tile];
            const CUtensorMap* mb = (w.kind == kGradDb) ? &P.tm_xat : &P.tm_dybt;
            const int natoms = w.mma_n / 8;
            const int per = grad_blocks_per_stage(w.mma_n);
            // token blocks [kb0, kb0 + nk) of the group's segments taken one after another (a split of the
            // reduction covers part of them)
            const int kb_end = w.kb0 + w.nk;
            int gb = 0;           // token block index over the item's segments
            for (int q = 0; q < g.nseg && gb < kb_end; ++q) {
                const TrainSeg s = P.tsegs[g.seg0 + q];
                const int nb = (s.len + kBK - 1) / kBK;
                if (gb + nb <= w.kb0) {
                    gb += nb;
                    continue;
                }
                const CUtensorMap* ma = (w.kind == kGradDb) ? &P.tm_seg_dy[g.seg0 + q] : &P.tm_seg_x[g.seg0 + q];
                for (int b = max(0, w.kb0 - gb); b < nb && gb + b < kb_end; ++b) {
                    const int i = gb + b - w.kb0;          // index of the block within the split
                    const int sub = i % per;
                    if (sub == 0) {
                        const int nsub = min(per, w.nk - i);
                        if (!acquire_stage(ring, bar_full, bar_empty, nsub * (kABytes + natoms * 1024), lane,
                                           abort_flag, P.status))
                            return;
                    }
                    const uint32_t full = bar_full + ring.stage * 8;
                    const uint32_t sa = smem_u32(smem + ring.stage * kStageBytes) + sub * kSubBytes;
                    const uint32_t sb = sa + kABytes;
                    if (lane < 2) tma_load_2d(sa + lane * 8192, ma, w.n0 + 64 * lane, b * kBK, full);
                    if (lane < natoms) tma_load_2d(sb + lane * 1024, mb, s.tpos0 + b * kBK, w.j0 + lane * 8, full);
                    if (sub == per - 1 || i == w.nk - 1) ring.next();
                }
                gb += nb;
            }
            continue;
        }
        const TileDesc td = P.tiles[w.tile];
        // shrink split: k-blocks [kb0, kb0 + nk) of the reduction; B = the pass's 8-row atoms of pool rows
        const CUtensorMap* ma = (w.kind == kShrinkFwd) ? (td.a_src ? &P.tm_xg : &P.tm_x)
                                : (w.kind == kShrinkDyb) ? &P.tm_dy : &P.tm_x;
        const bool use_b = (w.kind == kShrinkDyb);
        const CUtensorMap* mp = use_b ? &P.tm_pb : &P.tm_pa;
        const int natoms = w.mma_n / 8;
        const int32_t my_row = (lane < natoms) ? (use_b ? P.atoms_b : P.atoms_a)[td.atom0 + w.n0 / 8 + lane] : 0;
        // atom `lane` of the pass comes in a taller box when a run of atoms with consecutive pool rows starts at it
        // and ends inside the pass; atoms that no such box covers come one by one
        const int32_t my_box = (lane < natoms) ? (use_b ? P.boxes_b : P.boxes_a)[td.atom0 + w.n0 / 8 + lane] : 0;
        const bool lead = my_box > 1 && lane + my_box <= natoms;
        const uint32_t covered = __reduce_or_sync(0xffffffffu, lead ? (((1u << my_box) - 1u) << lane) : 0u);
        const int n_mine = (lane >= natoms) ? 0 : (lead ? my_box : (((covered >> lane) & 1u) ? 0 : 1));
        const CUtensorMap* my_map =
            (n_mine <= 1) ? mp : (use_b ? P.tm_pb_h : P.tm_pa_h) + (n_mine == 2 ? 0 : (n_mine == 4 ? 1 : 2));
        const int per = shrink_blocks_per_stage(w.mma_n);
        for (int i = 0; i < w.nk; ++i) {
            const int sub = i % per, kb = w.kb0 + i;
            if (sub == 0 &&
                !acquire_stage(ring, bar_full, bar_empty, min(per, w.nk - i) * (kABytes + natoms * 1024), lane,
                               abort_flag, P.status))
                return;
            const uint32_t full = bar_full + ring.stage * 8;
            const uint32_t sa = smem_u32(smem + ring.stage * kStageBytes) + sub * kSubBytes, sb = sa + kABytes;
            if (lane == 0) tma_load_2d(sa, ma, kb * kBK, td.a_row0, full);
            if (n_mine > 0) tma_load_2d(sb + lane * 1024, my_map, kb * kBK, my_row, full);
            if (sub == per - 1 || i == w.nk - 1) ring.next();
        }
    }
}

// --------------------------------------------------------------------------------------------- MMA issuer
__device__ void run_mma(const KParams& P, uint8_t* smem, uint32_t bar_full, uint32_t bar_empty, uint32_t bar_tfull,
                        uint32_t bar_tempty, uint32_t tmem, int i0, int i1, volatile int* abort_flag) {
    Ring ring;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int ii = i0; ii < i1; ++ii) {
        const WorkItem w = P.items[ii];
        if (skipped_item(P, w)) continue;
        if (!wait_phase(bar_tempty + acc * 8, acc_phase ^ 1u, abort_flag, P.status)) return;
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)acc * kBN;
        uint32_t accumulate = 0;
        // one stage: wait for it, issue `steps` MMAs of K=16 for each of its `nsub` blocks (`stride` bytes apart),
        // release it
        auto kblock = [&](int nsub, uint32_t stride, int steps, uint32_t idesc, int a_mn, int b_mn) -> bool {
            const uint32_t full = bar_full + ring.stage * 8, empty = bar_empty + ring.stage * 8;
            if (!wait_phase(full, ring.phase, abort_flag, P.status)) return false;
            tc_fence_after();
            for (int s = 0; s < nsub; ++s) {
                const uint32_t sa = smem_u32(smem + ring.stage * kStageBytes) + s * stride, sb = sa + kABytes;
                for (int k = 0; k < steps; ++k) {
                    const uint64_t ad = a_mn ? smem_desc(sa + k * 2048, 8192, 1024) : smem_desc(sa + k * 32, 16, 1024);
                    const uint64_t bd = b_mn ? smem_desc(sb + k * 2048, 8192, 1024) : smem_desc(sb + k * 32, 16, 1024);
                    mma_bf16(d, ad, bd, idesc, accumulate);
                    accumulate = 1;
                }
            }
            mma_commit(empty);
            ring.next();
            return true;
        };
        bool ok = true;
        if (w.kind == kGradDb || w.kind == kGradDa) {
            const uint32_t id = instr_desc(kTileM, w.mma_n, 1, 0);
            const int per = grad_blocks_per_stage(w.mma_n);
            for (int kb = 0; kb < w.nk && ok; kb += per) ok = kblock(min(per, w.nk - kb), kSubBytes, 4, id, 1, 0);
        } else {
            const uint32_t id = instr_desc(kTileM, w.mma_n, 0, 0);
            const int per = shrink_blocks_per_stage(w.mma_n);
            for (int kb = 0; kb < w.nk && ok; kb += per) ok = kblock(min(per, w.nk - kb), kSubBytes, 4, id, 0, 0);
        }
        if (!ok) return;
        mma_commit(bar_tfull + acc * 8);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
    }
}

// --------------------------------------------------------------------------------------------- epilogue
__device__ __forceinline__ void ld32_cols(uint32_t taddr, float (&v)[32]) {
    uint32_t a[16], b[16];
    tmem_ld16(taddr, a);
    tmem_ld16(taddr + 16, b);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        v[i] = __uint_as_float(a[i]);
        v[16 + i] = __uint_as_float(b[i]);
    }
}

// Finalize of one tile row of a shrink pass: keep the row's own adapter columns (everything else is zero) and
// write Z = bf16(s_a * xA) into the 128x64 shared-memory image the main pass bulk-loads, the unscaled xA of a
// fine-tuning row into xa_save (forward), and the transposed copy xA^T / dYB^T (backward; zero past the segment).
// Sliced layers: the chunk repeats every td.zstride columns, once per slice; its copy in region i holds slice
// i's values, which land at columns [i r, (i+1) r) of the saved / transposed layouts.
struct ShrinkRowOut {
    const KParams& P;
    const ShrinkUnit& u;
    int row;
    TileDesc td;
    int32_t rc, zc0, zr, save_off;
    float s;
    bool live;
    __nv_bfloat16* tdst;

    __device__ ShrinkRowOut(const KParams& P_, const ShrinkUnit& u_, int row_) : P(P_), u(u_), row(row_) {
        td = P.tiles[u.tile];
        rc = P.rowchunk[u.tile * kTileM + row];
        tdst = (u.kind == kShrinkDyb) ? P.dybt : (u.kind == kShrinkXa) ? P.xat : nullptr;
        live = rc >= 0;
        // backward tiles hold one adapter (at column 0): its columns are written for every row of the tile
        const int32_t ci = tdst ? td.chunk0 : rc;
        zc0 = 0; zr = 0; s = 0.f;
        if (ci >= 0 && (!tdst || td.nchunk > 0)) {
            const Chunk ch = P.chunks[ci];
            zc0 = ch.zcol; zr = ch.r; s = ch.scale;
        }
        save_off = (u.kind == kShrinkFwd && P.xa_save != nullptr) ? P.rowaux[u.tile * kTileM + row] : -1;
    }

    // columns [c, c+16) of the pass (all in one slice region: regions and chunks are 16-aligned)
    __device__ void put16(int c, const float (&acc)[16]) {
        const int d0 = u.n0 + c - zc0;
        const int reg = (td.zstride > 0 && d0 >= 0) ? d0 / td.zstride : 0;
        const int j0 = d0 - reg * td.zstride;        // column within the chunk's copy in region `reg`
        const int p0 = reg * zr + j0;                // the same column in the saved / transposed layouts
        float v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = (live && d0 >= 0 && j0 + i < zr) ? acc[i] : 0.f;
        if (u.kind != kShrinkXa && dbg_ok(P.debug, P.status, td.z_blk0 + (u.n0 + c) / kBK, P.db.z_blocks)) {
            const int zc = u.n0 + c;
            uint8_t* blk = P.zout + (size_t)(td.z_blk0 + zc / kBK) * kZBlockBytes + row * 128;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int chunk16 = ((zc % kBK) / 8 + h) ^ (row & 7);
                uint4 q;
                q.x = pack_bf16(s * v[8 * h + 0], s * v[8 * h + 1]);
                q.y = pack_bf16(s * v[8 * h + 2], s * v[8 * h + 3]);
                q.z = pack_bf16(s * v[8 * h + 4], s * v[8 * h + 5]);
                q.w = pack_bf16(s * v[8 * h + 6], s * v[8 * h + 7]);
                *reinterpret_cast<uint4*>(blk + chunk16 * 16) = q;
            }
        }
        if (d0 < 0) return;
        if (save_off >= 0 && dbg_ok(P.debug, P.status, (int64_t)save_off + p0 + min(16, zr - j0) - 1, P.db.xa_elems)) {
#pragma unroll
            for (int i = 0; i < 16; ++i)
                if (j0 + i < zr) P.xa_save[save_off + p0 + i] = __float2bfloat16_rn(v[i]);
        }
        if (tdst && dbg_ok(P.debug, P.status,
                           (int64_t)(p0 + min(16, zr - j0) - 1) * P.t_ld + td.tpos0 + row, P.db.t_elems)) {
#pragma unroll
            for (int i = 0; i < 16; ++i)
                if (j0 + i < zr) tdst[(size_t)(p0 + i) * P.t_ld + td.tpos0 + row] = __float2bfloat16_rn(v[i]);
        }
    }
};

// Columns [c, c + 16 G) of one row of a split reduction: the sum, in split order, of the unit's fp32 partials
// (p0: the row's first 4-column group of split 0; split s sits u.mma_n columns further per split).  Four splits'
// G 16-column groups are loaded (16 G loads of 16 bytes in flight per thread: the finalize is bound by L2 latency)
// before they are added.
template <int G>
__device__ __forceinline__ void sum_split_partials(const float* p0, const ShrinkUnit& u, int c, float (&v)[16 * G]) {
#pragma unroll
    for (int i = 0; i < 16 * G; ++i) v[i] = 0.f;
    for (int s0 = 0; s0 < u.nsplit; s0 += 4) {
        float4 a[4][4 * G];
#pragma unroll
        for (int sp = 0; sp < 4; ++sp)
#pragma unroll
            for (int q = 0; q < 4 * G; ++q)
                a[sp][q] = (s0 + sp < u.nsplit)
                               ? __ldcg(reinterpret_cast<const float4*>(p0 + ((size_t)(s0 + sp) * u.mma_n + c + 4 * q) *
                                                                                  kTileM))
                               : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int sp = 0; sp < 4; ++sp) {
            if (s0 + sp >= u.nsplit) break;
#pragma unroll
            for (int q = 0; q < 4 * G; ++q) {
                v[4 * q] += a[sp][q].x;
                v[4 * q + 1] += a[sp][q].y;
                v[4 * q + 2] += a[sp][q].z;
                v[4 * q + 3] += a[sp][q].w;
            }
        }
    }
}

// The finalize of a split unit's row: the split sums of columns [0, mma_n), handed to put(c, v) 16 columns at a time
// (two 16-column groups per round of loads where there are two)
template <class Put>
__device__ __forceinline__ void finalize_row(const float* p0, const ShrinkUnit& u, int mma_n, Put&& put) {
    int c = 0;
    for (; LORA_FINALIZE_GROUPS > 1 && c + 32 <= mma_n; c += 32) {
        float v[32];
        sum_split_partials<2>(p0, u, c, v);
        put(c, *reinterpret_cast<const float(*)[16]>(&v[0]));
        put(c + 16, *reinterpret_cast<const float(*)[16]>(&v[16]));
    }
    for (; c < mma_n; c += 16) {
        float v[16];
        sum_split_partials<1>(p0, u, c, v);
        put(c, v);
    }
}

// Writes one split's raw fp32 accumulator columns [0, mma_n) of this thread's row to its slot of the partial buffer
// (per 4 columns [C, C + 4): 128 rows of 4 floats at part + C * 128 + row * 4, so that a row's 4 columns are one
// 16-byte store and a warp's 32 rows one 512-byte run).
__device__ __forceinline__ void store_split_partial(float* dst, uint32_t taddr, int mma_n) {
    for (int c = 0; c < mma_n; c += 16) {
        uint32_t a[16];
        tmem_ld16(taddr + c, a);
        tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < 4; ++q)
            *reinterpret_cast<float4*>(dst + (size_t)(c + 4 * q) * kTileM) =
                make_float4(__uint_as_float(a[4 * q]), __uint_as_float(a[4 * q + 1]), __uint_as_float(a[4 * q + 2]),
                            __uint_as_float(a[4 * q + 3]));
    }
}

__device__ void run_epilogue(const KParams& P, uint32_t bar_tfull, uint32_t bar_tempty, uint32_t tmem, int i0, int i1,
                             volatile int* abort_flag) {
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int quarter = warp & 3;                 // TMEM lanes this warp may read
    const int row = quarter * 32 + lane;          // tile row = accumulator lane
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int ii = i0; ii < i1; ++ii) {
        const WorkItem w = P.items[ii];
        if (skipped_item(P, w)) continue;
        if (!wait_phase_long(bar_tfull + acc * 8, acc_phase, abort_flag, P.status)) return;
        tc_fence_after();
        const uint32_t taddr = tmem + (uint32_t)acc * kBN + ((uint32_t)(quarter * 32) << 16);
        if (w.kind == kGradDb || w.kind == kGradDa) {
            const GradGroup g = P.groups[w.tile];
            const bool is_b = (w.kind == kGradDb);
            const int32_t ld = is_b ? P.N : P.K;
            const int32_t m = w.n0 + row;
            // dB: accumulator column j is row j of the up factor (this item's slice columns); dA: row j0 + j of
            // the stacked down factors
            const int32_t jbase = is_b ? 0 : w.j0;
            const int32_t jend = is_b ? g.r : g.r * g.nslice;
            float* base = (is_b ? P.dB + (size_t)g.prow_b * P.N : P.dA + (size_t)g.prow_a * P.K) + (size_t)jbase * ld;
            // accumulator columns [c, c + 16) of this thread's row, scaled, into (or onto) the gradient
            auto put16 = [&](int c, const float (&v)[16]) {
                const int64_t last = ((int64_t)(is_b ? g.prow_b : g.prow_a) + jbase + min(c + 16, jend - jbase) - 1) * ld + m;
                if (m < ld && dbg_ok(P.debug, P.status, last, is_b ? P.db.grad_b : P.db.grad_a)) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int j = c + i;
                        if (jbase + j < jend) {
                            float* p = base + (size_t)j * ld + m;
                            const float val = g.scale * v[i];
                            *p = P.accumulate ? (*p + val) : val;
                        }
                    }
                }
            };
            if (w.nsplit <= 1) {
                for (int c = 0; c < w.mma_n; c += 16) {
                    uint32_t a[16];
                    tmem_ld16(taddr + c, a);
                    tmem_ld_wait();
                    float v[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(a[i]);
                    put16(c, v);
                }
            } else {
                // a split of the token range (the item's n_ext field holds its unit): raw fp32 partial sums; the
                // last split to arrive (per row quarter) sums all splits in split order and writes those 32 rows
                const ShrinkUnit u = P.units[w.n_ext];
                float* dst = P.part + (size_t)w.part * kTileM + row * 4;
                const bool part_ok = dbg_ok(P.debug, P.status, ((int64_t)u.part0 + (int64_t)u.nsplit * u.mma_n) * kTileM - 1,
                                            P.db.part_floats);
                if (part_ok) store_split_partial(dst, taddr, w.mma_n);
                tc_fence_before();
                mbar_arrive(bar_tempty + acc * 8);       // the accumulator is free; the rest reads global memory
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
                __threadfence();
                __syncwarp();
                int last = 0;
                int32_t* cnt = P.counters + w.n_ext * 4 + quarter;
                if (lane == 0) last = (atomicAdd(cnt, 1) == u.nsplit - 1) ? 1 : 0;
                last = __shfl_sync(0xffffffffu, last, 0);
                if (last && part_ok) {
                    __threadfence();
                    const float* p0 = P.part + (size_t)u.part0 * kTileM + row * 4;
                    finalize_row(p0, u, w.mma_n, put16);
                    __syncwarp();
                    if (lane == 0) *cnt = 0;              // ready for the next call on this workspace
                }
                continue;
            }
        } else {
            // shrink split (the item's n_ext field holds its shrink-unit index)
            const ShrinkUnit u = P.units[w.n_ext];
            if (u.nsplit == 1) {
                ShrinkRowOut out(P, u, row);
                for (int c = 0; c < w.mma_n; c += 16) {
                    uint32_t a[16];
                    tmem_ld16(taddr + c, a);
                    tmem_ld_wait();
                    float v[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(a[i]);
                    out.put16(c, v);
                }
            } else {
                // raw fp32 partial sums; the last split to arrive (per row quarter) sums all splits in split order
                // and finalizes those 32 rows
                float* dst = P.part + (size_t)w.part * kTileM + row * 4;
                const bool part_ok = dbg_ok(P.debug, P.status, ((int64_t)u.part0 + (int64_t)u.nsplit * u.mma_n) * kTileM - 1,
                                            P.db.part_floats);
                if (part_ok) store_split_partial(dst, taddr, w.mma_n);
                tc_fence_before();
                mbar_arrive(bar_tempty + acc * 8);       // the accumulator is free; the rest reads global memory
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
                __threadfence();
                __syncwarp();
                int last = 0;
                int32_t* cnt = P.counters + w.n_ext * 4 + quarter;
                if (lane == 0) last = (atomicAdd(cnt, 1) == u.nsplit - 1) ? 1 : 0;
                last = __shfl_sync(0xffffffffu, last, 0);
                if (last && part_ok) {
                    __threadfence();
                    ShrinkRowOut out(P, u, row);
                    const float* p0 = P.part + (size_t)u.part0 * kTileM + row * 4;
                    finalize_row(p0, u, w.mma_n, [&](int c, const float (&v)[16]) { out.put16(c, v); });
                    __syncwarp();
                    if (lane == 0) *cnt = 0;              // ready for the next call on this workspace
                }
                continue;
            }
        }
        tc_fence_before();
        mbar_arrive(bar_tempty + acc * 8);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
    }
}

__global__ void __launch_bounds__(kThreads, 1) lora_tc_kernel(const __grid_constant__ KParams P) {
    extern __shared__ uint8_t dsmem[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsmem) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 4);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const uint32_t bar_full = smem_u32(bars), bar_empty = bar_full + kStages * 8;
    const uint32_t bar_tfull = bar_empty + kStages * 8, bar_tempty = bar_tfull + 16;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar_full + s * 8, 1);
            mbar_init(bar_empty + s * 8, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar_tfull + b * 8, 1);
            mbar_init(bar_tempty + b * 8, 128);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    grid_dep_wait();
    const int i0 = P.cta_off[blockIdx.x], i1 = P.cta_off[blockIdx.x + 1];

    if (warp == 0) {
        run_producer(P, smem, bar_full, bar_empty, i0, i1, abort_flag);
    } else if (warp == 1) {
        if (lane == 0) run_mma(P, smem, bar_full, bar_empty, bar_tfull, bar_tempty, tmem, i0, i1, abort_flag);
    } else {
        run_epilogue(P, bar_tfull, bar_tempty, tmem, i0, i1, abort_flag);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
}

// =============================================================================================================
// Main pass on CTA pairs: tcgen05.mma.cta_group::2, M = 256 (one tile pair), N = 256 output columns.
//
// A cluster of two CTAs works on one item at a time.  CTA rank r holds the 128 rows of tile (2p + r) as the A
// operand and the 128-column half [n0 + 128 r, n0 + 128 r + 128) of the B operand; the leader (rank 0) issues
// the MMAs, which read both CTAs' shared memory and write each CTA's 128 accumulator lanes.  Each CTA moves
// only its own 32 KB per k-block (half of what one CTA needs for a 128x256 tile), so six stages fit.
// Both CTAs' TMA loads complete on the leader's "full" barrier; the leader's commits arrive on both CTAs'
// "empty" and "accumulator full" barriers; both CTAs' epilogue warps release the accumulator on the leader.
// =============================================================================================================
// Main-pass epilogue: a warp whose 32 rows are 32 consecutive output rows stages each 32-column chunk in shared
// memory and writes it with one TMA store (other warps, e.g. those of gathered decode tiles, store row by row).
// The staging buffers take the seventh pipeline stage's shared memory (6 and 7 stages measured alike).
#ifndef LORA_TMA_STORE
#define LORA_TMA_STORE 1
#endif
#ifndef LORA_MAIN_STAGES
#define LORA_MAIN_STAGES (LORA_TMA_STORE ? 6 : 7)
#endif
// L2 eviction priority of the main pass's TMA loads of the row operand (x / dY) and of W:
// 0 = normal, 1 = evict_first, 2 = evict_last.  evict_last on the rows once measured +21 % on an
// 8192 x 8192 x 28672 product, when each k-block still paid a call into the bounded wait; since that call is
// gone the plain policy is ~1 % faster on the co-serving step and the backward (seven 32-KB stages: +12 %).
#ifndef LORA_HINT_ROWS
#define LORA_HINT_ROWS 0
#endif
#ifndef LORA_HINT_W
#define LORA_HINT_W 0
#endif
// How many LoRA k-blocks ahead the pair kernel's producer reads the adapter-row table.
#ifndef LORA_ATOM_AHEAD
#define LORA_ATOM_AHEAD 4
#endif
constexpr int kAtomAhead = LORA_ATOM_AHEAD;
constexpr int kStages2 = LORA_MAIN_STAGES;
constexpr int kHalfN = kBN / 2;
constexpr int kA2Bytes = kTileM * kBK * 2;        // 16 KB
constexpr int kB2Bytes = kHalfN * kBK * 2;        // 16 KB
constexpr int kStage2Bytes = kA2Bytes + kB2Bytes;
constexpr int kOutChunkBytes = 32 * 32 * 2;       // 32 rows x 32 bf16 columns, 64-byte swizzled rows
constexpr int kOutStageBytes = LORA_TMA_STORE ? 4 * 2 * kOutChunkBytes : 0;   // 4 epilogue warps, 2 buffers each

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// shared::cluster address of the same shared variable in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// TMA load into this CTA's shared memory whose completion is signalled on an mbarrier of either CTA of the pair
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, int32_t c0, int32_t c1,
                                                 uint32_t bar_cluster) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
        "%3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar_cluster)
        : "memory");
}
// 3-D tile load of the same kind (pair-leader barrier)
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* map, int32_t c0, int32_t c1,
                                                 int32_t c2, uint32_t bar_cluster) {
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
        "%3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar_cluster)
        : "memory");
}
// Same, with an L2 cache-eviction policy (createpolicy) attached to the load
__device__ __forceinline__ void tma_load_2d_pair_hint(uint32_t dst, const CUtensorMap* map, int32_t c0, int32_t c1,
                                                      uint32_t bar_cluster, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], "
        "[%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar_cluster), "l"(policy)
        : "memory");
}
template <int HINT>
__device__ __forceinline__ void tma_load_hinted(uint32_t dst, const CUtensorMap* map, int32_t c0, int32_t c1,
                                                uint32_t bar_cluster) {
    if constexpr (HINT == 0) {
        tma_load_2d_pair(dst, map, c0, c1, bar_cluster);
    } else {
        uint64_t policy;
        if constexpr (HINT == 1)
            asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
        else
            asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(policy));
        tma_load_2d_pair_hint(dst, map, c0, c1, bar_cluster, policy);
    }
}

__device__ __forceinline__ void mma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                              uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// arrive (when the issued MMAs complete) on the barrier at this offset in both CTAs of the pair
__device__ __forceinline__ void mma_commit_pair(uint32_t bar) {
    const uint16_t mask = 3;
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
        "h"(mask)
        : "memory");
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}

struct Ring2 {
    int stage = 0;
    uint32_t phase = 0;
    __device__ __forceinline__ void next() {
        if (++stage == kStages2) { stage = 0; phase ^= 1u; }
    }
    __device__ __forceinline__ void advance(int n) {     // n x next()
        const int s = stage + n;
        phase ^= (uint32_t)((s / kStages2) & 1);
        stage = s % kStages2;
    }
};

// Lane 0 waits for this CTA's ring slot; the leader also arms its "full" barrier with the bytes of both CTAs.
__device__ __forceinline__ bool acquire_stage2(const Ring2& ring, uint32_t bar_full, uint32_t bar_empty,
                                               uint32_t bytes_per_cta, bool leader, int lane, volatile int* abort_flag,
                                               int32_t* status) {
    int ok = 1;
    if (lane == 0) {
        ok = wait_phase(bar_empty + ring.stage * 8, ring.phase ^ 1u, abort_flag, status) ? 1 : 0;
        if (ok && leader) mbar_expect_tx(bar_full + ring.stage * 8, 2 * bytes_per_cta);
    }
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

__device__ void run_producer2(const KParams& P, uint8_t* smem, uint32_t bar_full, uint32_t bar_empty, uint32_t rank,
                              int i0, int i1, volatile int* abort_flag) {
    const int lane = threadIdx.x & 31;
    const bool leader = (rank == 0);
    const uint32_t full_leader = mapa_shared(bar_full, 0);
    Ring2 ring;
    for (int ii = i0; ii < i1; ++ii) {
        const WorkItem w = P.items[ii];
        const TileDesc td = P.tiles[w.tile + rank];
        const bool fwd = (w.kind == kMainFwd);
        const CUtensorMap* ma = fwd ? (td.a_src ? &P.tm_xg : &P.tm_x) : &P.tm_dy;
        const int32_t nb = w.n0 + kHalfN * (int32_t)rank;     // first B column of this CTA's half
        // LoRA k-blocks' stacked adapter rows: per 8-row atom its pool row and the size of the TMA box that starts
        // there (lane L < 16: atom L >> 1 of block e, half L & 1)
        const CUtensorMap* mp = fwd ? &P.tm_pb : &P.tm_pa;
        const CUtensorMap* mph = fwd ? P.tm_pb_h : P.tm_pa_h;
        const int32_t* atoms = (fwd ? P.atoms_b : P.atoms_a) + td.atom0;
        const int32_t* boxes = (fwd ? P.boxes_b : P.boxes_a) + td.atom0;
        const int n_atoms = td.ext_k / 8;
        const int e0 = w.ext_c0 / kBK;
        auto atom_at = [&](int e, int32_t* box) -> int32_t {
            const int i = e * 8 + (lane >> 1);
            const bool in = lane < 16 && i < n_atoms;
            *box = in ? boxes[i] : 0;
            return in ? atoms[i] : 0;
        };
        // the LoRA k-blocks' atom rows and box sizes are read kAtomAhead blocks ahead of their use (a read of the
        // table is an L2 round trip, longer than a k-block's MMAs); the first blocks' are read before the dense
        // k-blocks, while lanes 1..31 have nothing else to do
        int32_t pre_row[kAtomAhead], pre_box[kAtomAhead];
#pragma unroll
        for (int j = 0; j < kAtomAhead; ++j) {
            pre_box[j] = 0;
            pre_row[j] = (j < w.n_ext) ? atom_at(e0 + j, &pre_box[j]) : 0;
        }
        // dense k-blocks: lane 0 alone waits for each free stage, arms the barrier and issues the stage's loads
        // (a freed stage is refilled with no warp-wide exchange on the way: the refill latency is what bounds the
        // pass); the other lanes only keep the ring position
        int ok = 1;
        if (lane == 0) {
            for (int kb = w.kb0; kb < w.kb0 + w.nk; ++kb) {
                if (!wait_phase(bar_empty + ring.stage * 8, ring.phase ^ 1u, abort_flag, P.status)) { ok = 0; break; }
                if (leader) mbar_expect_tx(bar_full + ring.stage * 8, 2 * kStage2Bytes);
                const uint32_t full = full_leader + ring.stage * 8;
                const uint32_t sa = smem_u32(smem + ring.stage * kStage2Bytes), sb = sa + kA2Bytes;
                tma_load_hinted<LORA_HINT_ROWS>(sa, ma, kb * kBK, td.a_row0, full);
                if (fwd) {
                    tma_load_hinted<LORA_HINT_W>(sb, &P.tm_w, kb * kBK, nb, full);                // Wt rows, K-major
                } else if (P.w3) {
                    tma_load_3d_pair(sb, &P.tm_w3, 0, kb * kBK, nb / 64, full);                   // both MN atoms
                } else {
                    tma_load_hinted<LORA_HINT_W>(sb, &P.tm_w, nb, kb * kBK, full);                // Wt, MN-major
                    tma_load_hinted<LORA_HINT_W>(sb + 8192, &P.tm_w, nb + 64, kb * kBK, full);
                }
                ring.next();
            }
        } else {
            ring.advance(w.nk);
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) return;
        // LoRA k-blocks: this tile's Z block and, per 8-row atom of stacked adapter rows, two 64-column MN boxes;
        // only the atoms of the item's LoRA columns [ext_c0, ext_c1)
        // (lane L < 16 loads half L & 1 of the box that starts at 8-row atom L >> 1, if one does: a run of atoms with
        // consecutive pool rows inside one chunk comes as one box of 16, 32 or 64 rows)
        auto lora_block = [&](int e, int32_t row, int32_t row_box) -> bool {
            const int q0 = (max(w.ext_c0, e * kBK) - e * kBK) / 8;
            const int q1 = (min(w.ext_c1, e * kBK + kBK) - e * kBK) / 8;
            if (!acquire_stage2(ring, bar_full, bar_empty, kZBlockBytes + (q1 - q0) * 2048, leader, lane, abort_flag,
                                P.status))
                return false;
            const uint32_t full = full_leader + ring.stage * 8;
            const uint32_t sa = smem_u32(smem + ring.stage * kStage2Bytes), sb = sa + kA2Bytes;
            if (lane == 0) tma_load_2d_pair(sa, &P.tm_z, 0, (td.z_blk0 + e) * kTileM, full);
            // a box that starts and ends inside the item's atoms [q0, q1) is loaded whole; every other atom of the
            // range comes on its own (a run of consecutive pool rows may straddle the item's first or last atom)
            const int q = lane >> 1, m = lane & 1;
            const bool in = lane < 16 && q >= q0 && q < q1;
            const int box = in ? row_box : 0;
            const bool lead = box > 1 && q + box <= q1;
            const uint32_t covered = __reduce_or_sync(0xffffffffu, (lead && m == 0) ? (((1u << box) - 1u) << q) : 0u);
            const int n_load = !in ? 0 : (lead ? box : (((covered >> q) & 1u) ? 0 : 1));
            if (n_load > 0) {
                const CUtensorMap* map = (n_load == 1) ? mp : mph + (n_load == 2 ? 0 : (n_load == 4 ? 1 : 2));
                tma_load_2d_pair(sb + m * 8192 + q * 1024, map, nb + 64 * m, row, full);
            }
            ring.next();
            return true;
        };
        const int e_end = e0 + w.n_ext;
        for (int eb = e0; eb < e_end; eb += kAtomAhead) {
#pragma unroll
            for (int j = 0; j < kAtomAhead; ++j) {
                const int e = eb + j;
                if (e >= e_end) break;
                const int32_t row = pre_row[j], row_box = pre_box[j];
                if (e + kAtomAhead < e_end) pre_row[j] = atom_at(e + kAtomAhead, &pre_box[j]);
                if (!lora_block(e, row, row_box)) return;
            }
        }
    }
}

__device__ void run_mma2(const KParams& P, uint8_t* smem, uint32_t bar_full, uint32_t bar_empty, uint32_t bar_tfull,
                         uint32_t bar_tempty, uint32_t tmem, int i0, int i1, volatile int* abort_flag) {
    Ring2 ring;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int ii = i0; ii < i1; ++ii) {
        const WorkItem w = P.items[ii];
        if (!wait_phase(bar_tempty + acc * 8, acc_phase ^ 1u, abort_flag, P.status)) return;
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)acc * kBN;
        uint32_t accumulate = 0;
        auto kblock = [&](int k0, int k1, uint32_t idesc, int b_mn) -> bool {
            const uint32_t full = bar_full + ring.stage * 8, empty = bar_empty + ring.stage * 8;
            if (!wait_phase(full, ring.phase, abort_flag, P.status)) return false;
            tc_fence_after();
            const uint32_t sa = smem_u32(smem + ring.stage * kStage2Bytes), sb = sa + kA2Bytes;
            for (int k = k0; k < k1; ++k) {
                const uint64_t ad = smem_desc(sa + k * 32, 16, 1024);
                const uint64_t bd = b_mn ? smem_desc(sb + k * 2048, 8192, 1024) : smem_desc(sb + k * 32, 16, 1024);
                mma_bf16_pair(d, ad, bd, idesc, accumulate);
                accumulate = 1;
            }
            mma_commit_pair(empty);
            ring.next();
            return true;
        };
        const int b_mn = (w.kind == kMainDx) ? 1 : 0;
        const uint32_t id_main = instr_desc(2 * kTileM, kBN, 0, b_mn);
        bool ok = true;
        for (int kb = 0; kb < w.nk && ok; ++kb) ok = kblock(0, 4, id_main, b_mn);
        const uint32_t id_ext = instr_desc(2 * kTileM, kBN, 0, 1);
        const int e0 = w.ext_c0 / kBK;
        for (int e = e0; e < e0 + w.n_ext && ok; ++e)
            ok = kblock((max(w.ext_c0, e * kBK) - e * kBK) / 16, (min(w.ext_c1, e * kBK + kBK) - e * kBK) / 16,
                        id_ext, 1);
        if (!ok) return;
        mma_commit_pair(bar_tfull + acc * 8);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
    }
}

__device__ __forceinline__ void store_row_bf16(const KParams& P, int32_t t, int32_t col0, const float (&v)[32]) {
    __nv_bfloat16* dst = P.out + (size_t)t * P.out_ld + col0;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        if (col0 + 8 * g + 8 <= P.out_cols) {
            uint4 q;
            q.x = pack_bf16(v[8 * g + 0], v[8 * g + 1]);
            q.y = pack_bf16(v[8 * g + 2], v[8 * g + 3]);
            q.z = pack_bf16(v[8 * g + 4], v[8 * g + 5]);
            q.w = pack_bf16(v[8 * g + 6], v[8 * g + 7]);
            *reinterpret_cast<uint4*>(dst + 8 * g) = q;
        }
    }
}

// TMA store of one staged 32 x 32 chunk (shared -> global), as its own bulk group
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int32_t c0, int32_t c1) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];\n\t"
                 "cp.async.bulk.commit_group;" ::"l"(reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1), "r"(src)
                 : "memory");
}
// a warp's 32 rows x 32 columns into its staging buffer: lane = row, 64-byte rows, 16-byte granules swizzled the
// way the tensor map's 64-byte swizzle reads them (granule g of row r at g ^ ((r >> 1) & 3))
__device__ __forceinline__ void stage_row_bf16(uint32_t buf, int lane, const float (&v)[32]) {
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        const uint32_t a = buf + lane * 64 + ((g ^ ((lane >> 1) & 3)) * 16);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(pack_bf16(v[8 * g + 0], v[8 * g + 1])),
                     "r"(pack_bf16(v[8 * g + 2], v[8 * g + 3])), "r"(pack_bf16(v[8 * g + 4], v[8 * g + 5])),
                     "r"(pack_bf16(v[8 * g + 6], v[8 * g + 7]))
                     : "memory");
    }
}

__device__ void run_epilogue2(const KParams& P, uint32_t bar_tfull, uint32_t bar_tempty, uint32_t tmem, uint32_t rank,
                              int i0, int i1, volatile int* abort_flag, uint32_t stage_out) {
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t tempty_leader = mapa_shared(bar_tempty, 0);
    int acc = 0;
    uint32_t acc_phase = 0;
    uint32_t nstore = 0;      // TMA stores issued by this warp (their buffers alternate)
    for (int ii = i0; ii < i1; ++ii) {
        const WorkItem w = P.items[ii];
        if (!wait_phase_long(bar_tfull + acc * 8, acc_phase, abort_flag, P.status)) break;
        tc_fence_after();
        const uint32_t taddr = tmem + (uint32_t)acc * kBN + ((uint32_t)(quarter * 32) << 16);
        const int32_t t = P.rowmap[(w.tile + rank) * kTileM + row];
        // K-split tiles: this split's fp32 partial goes to its slot, per CTA in 16-byte groups of 4 columns
        // ([64][128 rows][4]: a warp's rows write 512 contiguous bytes per group; rows without a token are
        // skipped); the reduce launch sums the slots
        float* part = (w.nsplit > 1)
                          ? P.part_main + ((size_t)(w.part + w.split) * 2 + rank) * kMainPartialFloats +
                                row * 4
                          : nullptr;
        const int32_t t0 = __shfl_sync(0xffffffffu, t, 0);
        bool bulk = LORA_TMA_STORE && part == nullptr && __all_sync(0xffffffffu, t >= 0 && t == t0 + lane);
        if (P.debug) {
            // the split slot, the row of this lane and the bulk store's 32 rows must lie in their buffers
            if (part && !dbg_ok(1, P.status, (int64_t)w.part + w.split, P.db.main_slots)) part = nullptr;
            if (bulk && !dbg_ok(1, P.status, (int64_t)t0 + 31, P.db.out_rows)) bulk = false;
        }
        const bool row_ok = t >= 0 && dbg_ok(P.debug, P.status, t, P.db.out_rows);
        const bool skip_split = (w.nsplit > 1 && part == nullptr);
        for (int c = 0; c < kBN; c += 32) {
            float v[32];
            ld32_cols(taddr + c, v);
            if (c + 32 == kBN) {
                // the accumulator has been read: hand it back to the leader's MMA before the last stores
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(tempty_leader + acc * 8);
            }
            if (bulk) {
                if (w.n0 + c >= P.out_cols) continue;          // past the last output column
                const uint32_t buf = stage_out + (nstore & 1u) * kOutChunkBytes;
                if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");   // buf's last store
                __syncwarp();
                stage_row_bf16(buf, lane, v);
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) tma_store_2d(&P.tm_out, buf, w.n0 + c, t0);
                ++nstore;
                continue;
            }
            if (!row_ok || skip_split) continue;
            if (part) {
#pragma unroll
                for (int i = 0; i < 32; i += 4)
                    __stcg(reinterpret_cast<float4*>(part + (size_t)(c + i) * kTileM),
                           make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]));
            } else {
                store_row_bf16(P, t, w.n0 + c, v);
            }
        }
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
    }
    // the staged chunks must be read, and written out, before the CTA exits
    if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    __syncwarp();
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    lora_main2_kernel(const __grid_constant__ KParams P) {
    extern __shared__ uint8_t dsmem[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsmem) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages2 * kStage2Bytes + kOutStageBytes);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kStages2 + 4);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const uint32_t bar_full = smem_u32(bars), bar_empty = bar_full + kStages2 * 8;
    const uint32_t bar_tfull = bar_empty + kStages2 * 8, bar_tempty = bar_tfull + 16;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t rank = cluster_ctarank();

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages2; ++s) {
            mbar_init(bar_full + s * 8, 1);      // used in the leader: its arm + both CTAs' TMA bytes
            mbar_init(bar_empty + s * 8, 1);     // the leader's commit
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar_tfull + b * 8, 1);     // the leader's commit
            mbar_init(bar_tempty + b * 8, 8);    // used in the leader: the 4 epilogue warps of each CTA
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    grid_dep_wait();
    const int pair = blockIdx.x >> 1;
    const int i0 = P.cta_off[pair], i1 = P.cta_off[pair + 1];

    if (warp == 0) {
        run_producer2(P, smem, bar_full, bar_empty, rank, i0, i1, abort_flag);
    } else if (warp == 1) {
        if (rank == 0 && lane == 0)
            run_mma2(P, smem, bar_full, bar_empty, bar_tfull, bar_tempty, tmem, i0, i1, abort_flag);
    } else {
        run_epilogue2(P, bar_tfull, bar_tempty, tmem, rank, i0, i1, abort_flag,
                      smem_u32(smem + kStages2 * kStage2Bytes) + (uint32_t)((warp - 2) * 2 * kOutChunkBytes));
    }
    __syncwarp();
    tc_fence_before();
    cluster_sync_all();
    tc_fence_after();
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
}

// --------------------------------------------------------------------------------------------- split reduce
// Sums the fp32 partials of every split output tile in split order and writes the tile's rows of the output.
// One block per (split tile, CTA half, row quarter, 64-column group); warp w sums 8 columns, lane = tile row, so
// every partial load is one coalesced 128-byte row of the column-major partial.
__global__ void __launch_bounds__(256) main_reduce_kernel(const SplitTile* __restrict__ splits,
                                                          const int32_t* __restrict__ rowmap,
                                                          const float* __restrict__ part, __nv_bfloat16* out,
                                                          int32_t out_ld, int32_t out_cols, int32_t debug,
                                                          int32_t* status, int64_t out_rows, int64_t main_slots) {
    grid_dep_wait();
    const int b = blockIdx.x;
    const SplitTile st = splits[b / 32];
    const int half = (b / 16) & 1, quarter = (b / 4) & 3, cgrp = b & 3;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int r = quarter * 32 + lane;
    const int c0 = cgrp * 64 + warp * 8;
    const int32_t t = rowmap[(st.tile + half) * kTileM + r];
    const int32_t col = st.n0 + c0;
    if (t < 0 || col + 8 > out_cols) return;
    if (!dbg_ok(debug, status, t, out_rows) || !dbg_ok(debug, status, (int64_t)st.part + st.nsplit - 1, main_slots))
        return;
    float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    // a row's 8 columns are two 16-byte groups; four splits' groups are loaded before they are added in order
    const float* p = part + ((size_t)st.part * 2 + half) * kMainPartialFloats + (size_t)c0 * kTileM + r * 4;
    for (int s0 = 0; s0 < st.nsplit; s0 += 4) {
        float4 a[4][2];
#pragma unroll
        for (int sp = 0; sp < 4; ++sp) {
            const float* ps = p + (size_t)(s0 + sp) * 2 * kMainPartialFloats;
            const bool in = s0 + sp < st.nsplit;
            a[sp][0] = in ? __ldcg(reinterpret_cast<const float4*>(ps)) : make_float4(0.f, 0.f, 0.f, 0.f);
            a[sp][1] = in ? __ldcg(reinterpret_cast<const float4*>(ps + 4 * kTileM)) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int sp = 0; sp < 4; ++sp) {
            if (s0 + sp >= st.nsplit) break;
            v[0] += a[sp][0].x; v[1] += a[sp][0].y; v[2] += a[sp][0].z; v[3] += a[sp][0].w;
            v[4] += a[sp][1].x; v[5] += a[sp][1].y; v[6] += a[sp][1].z; v[7] += a[sp][1].w;
        }
    }
    uint4 q;
    q.x = pack_bf16(v[0], v[1]);
    q.y = pack_bf16(v[2], v[3]);
    q.z = pack_bf16(v[4], v[5]);
    q.w = pack_bf16(v[6], v[7]);
    *reinterpret_cast<uint4*>(out + (size_t)t * out_ld + col) = q;
}

// Failure-path self-test: one thread waits, with the kernels' bounded wait, on an mbarrier that nothing ever
// arrives on.  The wait gives up after its time limit and records LORA_ERR_TIMEOUT in the status word; the
// kernel then returns normally, leaving the context usable.
__global__ void selftest_timeout_kernel(int32_t* status) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x == 0) wait_phase(smem_u32(&bar), 0, reinterpret_cast<volatile int*>(&abort_flag), status);
}

}  // namespace

size_t tc_smem_bytes() { return (size_t)kStages * kStageBytes + 1024 + 1024; }
size_t tc2_smem_bytes() { return (size_t)kStages2 * kStage2Bytes + kOutStageBytes + 1024 + 1024; }

cudaError_t set_wait_limit_ns(uint64_t ns) { return cudaMemcpyToSymbol(g_wait_limit_ns, &ns, sizeof(ns)); }

cudaError_t selftest_timeout_launch(int32_t* status, cudaStream_t stream) {
    selftest_timeout_kernel<<<1, 32, 0, stream>>>(status);
    return cudaGetLastError();
}

// cudaLaunchKernelEx with programmatic stream serialization (see grid_dep_wait)
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

cudaError_t tc2_launch(const KParams& P, int pairs, cudaStream_t stream) {
    static int configured[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && !configured[dev]) {
        e = cudaFuncSetAttribute(lora_main2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tc2_smem_bytes());
        if (e != cudaSuccess) return e;
        configured[dev] = 1;
    }
    return launch_pdl(lora_main2_kernel, dim3(2 * pairs), dim3(kThreads), tc2_smem_bytes(), stream, P);
}

cudaError_t main_reduce_launch(const SplitTile* splits, int32_t n_splits, const int32_t* rowmap, const float* part,
                               __nv_bfloat16* out, int32_t out_ld, int32_t out_cols, const KParams& P,
                               cudaStream_t stream) {
    if (n_splits <= 0) return cudaSuccess;
    return launch_pdl(main_reduce_kernel, dim3(n_splits * 32), dim3(256), 0, stream, splits, rowmap, part, out, out_ld,
                      out_cols, P.debug, P.status, P.db.out_rows, P.db.main_slots);
}

cudaError_t tc_launch(const KParams& P, int grid, cudaStream_t stream) {
    static int configured[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && !configured[dev]) {
        e = cudaFuncSetAttribute(lora_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tc_smem_bytes());
        if (e != cudaSuccess) return e;
        configured[dev] = 1;
    }
    return launch_pdl(lora_tc_kernel, dim3(grid), dim3(kThreads), tc_smem_bytes(), stream, P);
}

}  // namespace lora
