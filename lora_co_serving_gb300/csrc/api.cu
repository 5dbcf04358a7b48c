// api.cu -- the C ABI (include/lora_mixed.h): validation, planning, staging, tensor maps and launches.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <list>
#include <memory>
#include <mutex>
#include <string>
#include <vector>

#include "lora_mixed.h"
#include "plan.h"
#include "simt.h"
#include "tc_kernel.h"

using namespace lora;

namespace {

thread_local std::string g_err;
thread_local bool g_trace_on = false;
thread_local cudaEvent_t g_trace[8];

// Record the tracing event that opens (end = 0) or closes (end = 1) launch group `group`.
cudaError_t trace(int group, int end, cudaStream_t stream) {
    if (!g_trace_on) return cudaSuccess;
    return cudaEventRecord(g_trace[2 * group + end], stream);
}

int fail(int code, const std::string& msg) {
    g_err = msg;
    return code;
}

#define CUDA_TRY(expr)                                                                         \
    do {                                                                                       \
        cudaError_t e_ = (expr);                                                               \
        if (e_ != cudaSuccess) return fail(LORA_ERR_CUDA, std::string(#expr) + ": " + cudaGetErrorString(e_)); \
    } while (0)

// ------------------------------------------------------------------------------------------------ tensor maps
#ifndef LORA_L2_PROMOTION
#define LORA_L2_PROMOTION CU_TENSOR_MAP_L2_PROMOTION_NONE
#endif
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 2-D bf16 tensor [outer, inner] with row stride `ld` elements, 128-byte swizzled boxes {box_in, box_out}.
bool encode_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t ld, uint32_t box_in,
               uint32_t box_out, std::string* err, bool swizzle = true) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) { *err = "cuTensorMapEncodeTiled is not available from the driver"; return false; }
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {ld * 2};
    cuuint32_t box[2] = {box_in, box_out};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                    LORA_L2_PROMOTION,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        *err = "cuTensorMapEncodeTiled failed (" + std::to_string((int)r) + ") for a [" + std::to_string(outer) +
               ", " + std::to_string(inner) + "] tensor";
        return false;
    }
    return true;
}

// Wt [N, K] as a 3-D tensor [K/64][N][64] (K a multiple of 64): a {64, 64, 2} box holds rows [n, n + 64) of two
// consecutive 64-column chunks, one 8 KB MN-major atom block after the other, as the backward's B operand wants
#ifndef LORA_W3
#define LORA_W3 1
#endif
bool encode_w3(CUtensorMap* m, const void* base, uint64_t K, uint64_t N) {
    EncodeTiledFn fn = encode_fn();
    if (!fn || K % 64 != 0) return false;
    cuuint64_t dims[3] = {64, N, K / 64};
    cuuint64_t strides[2] = {K * 2, 128};
    cuuint32_t box[3] = {64, 64, 2};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, LORA_L2_PROMOTION,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The main pass's output map: [rows, cols] bf16 rows ld elements apart, 32 x 32 boxes with 64-byte swizzle (the
// epilogue's staging layout)
bool encode_out(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint64_t ld, std::string* err) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) { *err = "cuTensorMapEncodeTiled is not available from the driver"; return false; }
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {ld * 2};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, LORA_L2_PROMOTION,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        *err = "cuTensorMapEncodeTiled failed (" + std::to_string((int)r) + ") for the [" + std::to_string(rows) +
               ", " + std::to_string(cols) + "] output";
        return false;
    }
    return true;
}

// ------------------------------------------------------------------------------------------------ device info
int sm_count() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev < 64 && cache[dev]) return cache[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev < 64) cache[dev] = n;
    return n;
}

// ------------------------------------------------------------------------------------------------ host staging
// The plan travels host -> workspace through a small ring of pinned buffers per device, so the copy is
// truly asynchronous.  A slot is reused only after the event recorded behind its copy has completed.
struct StagingRing {
    static constexpr int kSlots = 8;
    struct Slot {
        void* host = nullptr;
        size_t cap = 0;
        cudaEvent_t ev = nullptr;
        bool pending = false;
    };
    std::mutex mu;
    Slot slot[kSlots];
    int next = 0;
};
StagingRing g_rings[64];

// Set for the duration of a call made by an entry point that must not allocate: the plan is then copied
// straight from the (pageable) host blob instead of through the pinned ring, which allocates on first use.
thread_local bool g_direct_upload = false;

// Plans uploaded by calls made while their stream is being captured into a CUDA graph: the graph's copy node
// reads this host memory at every replay, so each such copy is kept for the life of the process.
std::mutex g_captured_mu;
std::vector<void*> g_captured;

int stage_copy(void* dst, const void* src, size_t bytes, cudaStream_t stream) {
    if (bytes == 0) return LORA_OK;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    CUDA_TRY(cudaStreamIsCapturing(stream, &cs));
    if (cs == cudaStreamCaptureStatusActive) {
        // no ring slot (a later call would overwrite it before a replay) and no wait: a pinned copy of its own,
        // allocated with this thread's capture rules relaxed (an allocation is not stream work)
        cudaStreamCaptureMode mode = cudaStreamCaptureModeRelaxed;
        CUDA_TRY(cudaThreadExchangeStreamCaptureMode(&mode));
        void* h = nullptr;
        const cudaError_t e = cudaHostAlloc(&h, bytes, cudaHostAllocPortable);
        cudaThreadExchangeStreamCaptureMode(&mode);
        if (e != cudaSuccess) return fail(LORA_ERR_CUDA, std::string("cudaHostAlloc: ") + cudaGetErrorString(e));
        std::memcpy(h, src, bytes);
        {
            std::lock_guard<std::mutex> lock(g_captured_mu);
            g_captured.push_back(h);
        }
        CUDA_TRY(cudaMemcpyAsync(dst, h, bytes, cudaMemcpyHostToDevice, stream));
        return LORA_OK;
    }
    if (g_direct_upload) {
        CUDA_TRY(cudaMemcpyAsync(dst, src, bytes, cudaMemcpyHostToDevice, stream));
        return LORA_OK;
    }
    int dev = 0;
    CUDA_TRY(cudaGetDevice(&dev));
    if (dev >= 64) {   // unusual device index: fall back to a pageable copy
        CUDA_TRY(cudaMemcpyAsync(dst, src, bytes, cudaMemcpyHostToDevice, stream));
        return LORA_OK;
    }
    StagingRing& R = g_rings[dev];
    std::lock_guard<std::mutex> lock(R.mu);
    StagingRing::Slot& s = R.slot[R.next];
    R.next = (R.next + 1) % StagingRing::kSlots;
    if (s.pending) {
        CUDA_TRY(cudaEventSynchronize(s.ev));
        s.pending = false;
    }
    if (!s.ev) CUDA_TRY(cudaEventCreateWithFlags(&s.ev, cudaEventDisableTiming));
    if (s.cap < bytes) {
        if (s.host) CUDA_TRY(cudaFreeHost(s.host));
        s.host = nullptr;
        size_t cap = std::max<size_t>(bytes, 1 << 16);
        CUDA_TRY(cudaHostAlloc(&s.host, cap, cudaHostAllocPortable));
        s.cap = cap;
    }
    std::memcpy(s.host, src, bytes);
    CUDA_TRY(cudaMemcpyAsync(dst, s.host, bytes, cudaMemcpyHostToDevice, stream));
    CUDA_TRY(cudaEventRecord(s.ev, stream));
    s.pending = true;
    return LORA_OK;
}

template <class T>
void put(std::vector<uint8_t>& blob, size_t off, const std::vector<T>& v) {
    if (!v.empty()) std::memcpy(blob.data() + off, v.data(), sizeof(T) * v.size());
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Write the plan (tiles ... per-CTA item ranges) into a host blob laid out exactly like the workspace prefix.  Each
// launch's items go in the order of its CTA lists, so that CTA c runs items [off[c], off[c + 1]) in place.
void build_blob(const Plan& pl, const Layout& L, const std::vector<int32_t> (&off)[3],
                const std::vector<int32_t> (&lst)[3], std::vector<uint8_t>* blob) {
    blob->assign(L.plan_end - L.tiles, 0);
    auto at = [&](size_t o) { return o - L.tiles; };
    std::vector<uint8_t>& b = *blob;
    put(b, at(L.tiles), pl.tiles);
    put(b, at(L.chunks), pl.chunks);
    put(b, at(L.rowmap), pl.rowmap);
    put(b, at(L.rowchunk), pl.rowchunk);
    put(b, at(L.rowaux), pl.rowaux);
    put(b, at(L.groups), pl.groups);
    put(b, at(L.tsegs), pl.tsegs);
    put(b, at(L.atoms_a), pl.atoms_a);
    put(b, at(L.atoms_b), pl.atoms_b);
    put(b, at(L.boxes_a), pl.boxes_a);
    put(b, at(L.boxes_b), pl.boxes_b);
    put(b, at(L.units), pl.units);
    put(b, at(L.splits), pl.splits);
    put(b, at(L.bgmv), pl.bgmv);
    for (int k = 0; k < 3; ++k) {
        std::vector<WorkItem> ordered(lst[k].size());
        for (size_t j = 0; j < ordered.size(); ++j) ordered[j] = pl.items[k][lst[k][j]];
        put(b, at(L.items[k]), ordered);
        put(b, at(L.cta_off[k]), off[k]);
    }
}

void fill_plan_pointers(KParams* P, uint8_t* ws, const Layout& L, int launch) {
    P->tiles = reinterpret_cast<const TileDesc*>(ws + L.tiles);
    P->chunks = reinterpret_cast<const Chunk*>(ws + L.chunks);
    P->rowmap = reinterpret_cast<const int32_t*>(ws + L.rowmap);
    P->rowchunk = reinterpret_cast<const int32_t*>(ws + L.rowchunk);
    P->rowaux = reinterpret_cast<const int32_t*>(ws + L.rowaux);
    P->groups = reinterpret_cast<const GradGroup*>(ws + L.groups);
    P->tsegs = reinterpret_cast<const TrainSeg*>(ws + L.tsegs);
    P->items = reinterpret_cast<const WorkItem*>(ws + L.items[launch]);
    P->cta_off = reinterpret_cast<const int32_t*>(ws + L.cta_off[launch]);
    P->atoms_a = reinterpret_cast<const int32_t*>(ws + L.atoms_a);
    P->atoms_b = reinterpret_cast<const int32_t*>(ws + L.atoms_b);
    P->boxes_a = reinterpret_cast<const int32_t*>(ws + L.boxes_a);
    P->boxes_b = reinterpret_cast<const int32_t*>(ws + L.boxes_b);
    P->part = reinterpret_cast<float*>(ws + L.part);
    P->part_main = reinterpret_cast<float*>(ws + L.part_main);
    P->units = reinterpret_cast<const ShrinkUnit*>(ws + L.units);
    P->counters = reinterpret_cast<int32_t*>(ws + L.counters);
    P->status = reinterpret_cast<int32_t*>(ws + L.status);
}

int check_workspace(void* workspace, size_t ws_bytes, size_t need) {
    if (!workspace) return fail(LORA_ERR_WORKSPACE, "workspace is NULL");
    if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0)
        return fail(LORA_ERR_WORKSPACE, "workspace must be 256-byte aligned");
    if (ws_bytes < need)
        return fail(LORA_ERR_WORKSPACE, "workspace too small: need " + std::to_string(need) + " bytes, got " +
                                            std::to_string(ws_bytes));
    return LORA_OK;
}

// ------------------------------------------------------------------------------------------------ float32 path
struct F32Blob {
    std::vector<uint8_t> bytes;
    size_t tok = 0, ad = 0, segs = 0, xa = 0, dyb = 0;
};

void f32_layout(const Problem& p, size_t base, F32Blob* fb) {
    auto al = [](size_t v) { return (v + 255) & ~size_t(255); };
    fb->tok = base;
    fb->ad = fb->tok + al(sizeof(int32_t) * (size_t)p.T);
    fb->segs = fb->ad + al(32 * (size_t)(p.n_adapters + 1));
    fb->xa = fb->segs + al(32 * (size_t)(p.segs.size() + 1));
    fb->dyb = fb->xa + al(sizeof(float) * (size_t)p.T * 128);
    fb->bytes.assign(fb->xa - fb->tok, 0);
    std::vector<int32_t> tok(p.T, -1);
    std::vector<F32Seg> segs(p.segs.size());
    int64_t xo = 0;
    int32_t n_train_seen = 0;
    for (size_t i = 0; i < p.segs.size(); ++i) {
        const auto& s = p.segs[i];
        for (int32_t t = s.start; t < s.start + s.len; ++t) tok[t] = s.adapter_id;
        F32Seg f{};
        f.start = s.start; f.len = s.len; f.adapter = s.adapter_id; f.is_train = s.is_train;
        f.xoff = -1;
        f.order = -1;
        if (s.is_train) {
            f.xoff = int32_t(xo);
            xo += (int64_t)s.len * p.rank[s.adapter_id];
            f.order = n_train_seen++;
        }
        segs[i] = f;
    }
    std::vector<AdapterRec> ad(p.n_adapters);
    for (int32_t a = 0; a < p.n_adapters; ++a) {
        ad[a] = AdapterRec{p.a_off[a], p.b_off[a], p.rank[a], p.scale[a], 0, 0};
    }
    put(fb->bytes, fb->tok - base, tok);
    put(fb->bytes, fb->ad - base, ad);
    put(fb->bytes, fb->segs - base, segs);
}

int begin_call(const Layout& L, const Plan& pl, void* ws, size_t bytes_plan, const void* blob, cudaStream_t stream) {
    uint8_t* w = static_cast<uint8_t*>(ws);
    CUDA_TRY(cudaMemsetAsync(w + L.status, 0, L.zero_end - L.status, stream));
    // Z columns outside a tile's own adapters must read as zero in the main pass
    if (pl.z_blocks > 0) CUDA_TRY(cudaMemsetAsync(w + L.z, 0, (size_t)pl.z_blocks * kZBlockBytes, stream));
    return stage_copy(w + L.tiles, blob, bytes_plan, stream);
}

#ifndef LORA_MAIN_PERSISTENT
#define LORA_MAIN_PERSISTENT 1
#endif
// Per-launch CTA assignment: shrink and grad items over single CTAs, main items over CTA pairs.
void assign_all(const Plan& pl, int sms, std::vector<int32_t> (&off)[3], std::vector<int32_t> (&lst)[3], int (&grid)[3]) {
    for (int k = 0; k < 3; ++k) {
        const int n = (int)pl.items[k].size();
        if (k == 1 && !LORA_MAIN_PERSISTENT) {
            // one CTA pair per item, dispatched by the hardware in item order
            grid[k] = n;
            off[k].resize(n + 1);
            lst[k].resize(n);
            for (int i = 0; i <= n; ++i) off[k][i] = i;
            for (int i = 0; i < n; ++i) lst[k][i] = i;
            continue;
        }
        const int units = (k == 1) ? sms / 2 : sms;
        grid[k] = std::min<int>(std::min(units, kMaxCtas), n);
        if (grid[k] > 0) assign_items(pl.items[k], pl, grid[k], &off[k], &lst[k]);
    }
}

cudaError_t launch_group(int k, KParams* P, uint8_t* ws, const Layout& L, const int (&grid)[3], cudaStream_t stream) {
    if (grid[k] == 0) return cudaSuccess;
    fill_plan_pointers(P, ws, L, k);
    return (k == 1) ? tc2_launch(*P, grid[k], stream) : tc_launch(*P, grid[k], stream);
}

// The reduce of the main pass's split output tiles (after the main launch, on the same stream).
cudaError_t launch_reduce(const Plan& pl, const KParams& P, uint8_t* ws, const Layout& L, cudaStream_t stream) {
    if (pl.splits.empty()) return cudaSuccess;
    return main_reduce_launch(reinterpret_cast<const SplitTile*>(ws + L.splits), int32_t(pl.splits.size()),
                              reinterpret_cast<const int32_t*>(ws + L.rowmap), reinterpret_cast<const float*>(ws + L.part_main),
                              P.out, P.out_ld, P.out_cols, P, stream);
}


// ------------------------------------------------------------------------------------------------ plan cache
// Validation, the tile plan, the workspace layout, the per-CTA item lists and the plan blob depend only on the
// call's shape, segment table and pool description (host arrays), not on any device pointer.  A serving step
// reuses one segment table for every projection of every layer, so each thread keeps its last few plans and a
// call whose inputs are byte-for-byte those of a kept plan reuses it (compared in full, no hashing).
struct Prepared {
    int32_t kind = 0, T = 0, K = 0, N = 0, S = 1, opts = 0;
    int32_t bounds[LORA_MAX_SLICES + 1] = {0, 0, 0, 0, 0};
    std::vector<lora_segment_t> segs;
    std::vector<int64_t> a_off, b_off;
    std::vector<int32_t> rank;
    std::vector<float> scale;
    Problem p;
    Plan pl;
    Layout L;
    int sms = 0;                         // the CTA lists below were made for this many SMs
    std::vector<int32_t> off[3], lst[3];
    int grid[3] = {0, 0, 0};
    std::vector<uint8_t> blob;
    // The launch parameters (tensor maps and pointers) of the last call made with this plan, and the pointers and
    // flags they were built from: a call that repeats them copies the parameters instead of encoding every tensor
    // map again (a dozen or more driver calls per call).
    std::unique_ptr<KParams> params;
    std::vector<uintptr_t> params_key;
};

// The cached launch parameters of `pr` when they were built from `key`, else null (the caller builds them and
// keeps them with keep_params).
const KParams* cached_params(const Prepared* pr, const std::vector<uintptr_t>& key) {
    return (pr->params && pr->params_key == key) ? pr->params.get() : nullptr;
}
void keep_params(Prepared* pr, const KParams& P, std::vector<uintptr_t>&& key) {
    if (!pr->params) pr->params.reset(new KParams);
    *pr->params = P;
    pr->params_key = std::move(key);
}
constexpr size_t kPlanCacheEntries = 8;
thread_local std::list<std::unique_ptr<Prepared>> g_plans;

template <class T>
bool same(const std::vector<T>& v, const T* a, size_t n) {
    return v.size() == n && (n == 0 || std::memcmp(v.data(), a, sizeof(T) * n) == 0);
}

bool matches(const Prepared& e, int32_t kind, int32_t T, int32_t K, int32_t N, const lora_pool_t* pool,
             const lora_slices_t* slices, const lora_segment_t* segs, int32_t n_segs, int32_t opts) {
    const int32_t S = slices ? slices->n_slices : 1;
    if (e.kind != kind || e.T != T || e.K != K || e.N != N || e.S != S || e.opts != opts) return false;
    if (slices && (S < 1 || S > LORA_MAX_SLICES || !slices->col_bounds ||
                   std::memcmp(e.bounds, slices->col_bounds, sizeof(int32_t) * (S + 1)) != 0))
        return false;
    const size_t P = pool->n_adapters > 0 ? size_t(pool->n_adapters) : 0;
    if (e.rank.size() != P || (P > 0 && (!pool->a_off || !pool->b_off || !pool->rank || !pool->scale))) return false;
    return same(e.segs, segs, n_segs > 0 ? size_t(n_segs) : 0) && same(e.rank, pool->rank, P) &&
           same(e.a_off, pool->a_off, P) && same(e.b_off, pool->b_off, P) && same(e.scale, pool->scale, P);
}

// The bf16 plan of a call: from the cache, or validated and planned now (kind 0: forward; 1: backward with
// opts = want_dx | want_da << 1 | want_db << 2 | recompute << 3 | per_segment << 4).
int prepare(int32_t kind, int32_t T, int32_t K, int32_t N, const lora_pool_t* pool, const lora_slices_t* slices,
            const lora_segment_t* segs, int32_t n_segs, int32_t opts, Prepared** out) {
    if (pool && n_segs >= 0 && (n_segs == 0 || segs)) {
        for (auto it = g_plans.begin(); it != g_plans.end(); ++it) {
            if (matches(**it, kind, T, K, N, pool, slices, segs, n_segs, opts)) {
                g_plans.splice(g_plans.begin(), g_plans, it);
                *out = g_plans.front().get();
                return LORA_OK;
            }
        }
    }
    auto e = std::make_unique<Prepared>();
    std::string err;
    int rc = validate(T, K, N, LORA_BF16, pool, segs, n_segs, &e->p, &err, slices);
    if (rc != LORA_OK) return fail(rc, err);
    e->kind = kind; e->T = T; e->K = K; e->N = N; e->opts = opts;
    e->S = e->p.S;
    std::memcpy(e->bounds, e->p.bounds, sizeof(e->bounds));
    e->segs.assign(segs, segs + n_segs);
    const size_t P = size_t(pool->n_adapters);
    if (P > 0) {
        e->a_off.assign(pool->a_off, pool->a_off + P);
        e->b_off.assign(pool->b_off, pool->b_off + P);
        e->rank.assign(pool->rank, pool->rank + P);
        e->scale.assign(pool->scale, pool->scale + P);
    }
    // the cached problem reads the entry's own copies of the pool arrays
    e->p.a_off = e->a_off.data(); e->p.b_off = e->b_off.data();
    e->p.rank = e->rank.data(); e->p.scale = e->scale.data();
    if (kind == 0) plan_forward(e->p, &e->pl);
    else plan_backward(e->p, opts & 1, opts & 2, opts & 4, opts & 8, &e->pl, opts & 16);
    e->L = layout_of(e->p, e->pl, kind == 1);
    g_plans.push_front(std::move(e));
    if (g_plans.size() > kPlanCacheEntries) g_plans.pop_back();
    *out = g_plans.front().get();
    return LORA_OK;
}

// The per-CTA item lists and the plan blob of a prepared call for this device's SM count.
void assign_for(Prepared* e, int sms) {
    if (e->sms == sms) return;
    assign_all(e->pl, sms, e->off, e->lst, e->grid);
    build_blob(e->pl, e->L, e->off, e->lst, &e->blob);
    e->sms = sms;
}
}  // namespace

namespace lora {
int forward_scratch_bytes(int32_t T, int32_t K, int32_t N, lora_dtype_t dt, const lora_pool_t* pool,
                          const lora_segment_t* segs, int32_t n_segs, size_t* out) {
    if (dt == LORA_BF16) {
        Prepared* pr = nullptr;
        const int rc = prepare(0, T, K, N, pool, nullptr, segs, n_segs, 0, &pr);
        if (rc != LORA_OK) return rc;
        *out = pr->L.total;
        return LORA_OK;
    }
    Problem p;
    std::string err;
    const int rc = validate(T, K, N, dt, pool, segs, n_segs, &p, &err);
    if (rc != LORA_OK) return fail(rc, err);
    Plan empty;
    *out = layout_of(p, empty, false).total;
    return LORA_OK;
}

// Scoped switch to direct (non-staged) plan uploads for the calling thread; see g_direct_upload.
DirectUpload::DirectUpload() : prev_(g_direct_upload) { g_direct_upload = true; }
DirectUpload::~DirectUpload() { g_direct_upload = prev_; }
void set_last_error(const char* msg) { g_err = msg; }
}  // namespace lora

// ================================================================================================== C ABI
extern "C" {

const char* lora_last_error(void) { return g_err.c_str(); }

size_t lora_sliced_workspace_size(int32_t T, int32_t K, int32_t N, lora_dtype_t dt, const lora_pool_t* pool,
                                  const lora_slices_t* slices, const lora_segment_t* segs, int32_t n_segs) {
    Problem p;
    std::string err;
    int rc = validate(T, K, N, dt, pool, segs, n_segs, &p, &err, slices);
    if (rc != LORA_OK) { g_err = err; return 0; }
    Plan f, b;
    plan_forward(p, &f);
    plan_backward(p, true, true, true, true, &b);
    return std::max(layout_of(p, f, false).total, layout_of(p, b, true).total);
}

size_t lora_workspace_size(int32_t T, int32_t K, int32_t N, lora_dtype_t dt, const lora_pool_t* pool,
                           const lora_segment_t* segs, int32_t n_segs) {
    return lora_sliced_workspace_size(T, K, N, dt, pool, nullptr, segs, n_segs);
}

size_t lora_sliced_xa_size(lora_dtype_t dt, const lora_pool_t* pool, const lora_slices_t* slices,
                           const lora_segment_t* segs, int32_t n_segs) {
    if (dt != LORA_BF16 && dt != LORA_F32) { g_err = "unknown dtype"; return 0; }
    if (!pool || (n_segs > 0 && !segs) || n_segs < 0) { g_err = "NULL pool or segments"; return 0; }
    int32_t S = 1;
    if (slices) {
        if (slices->n_slices < 1 || slices->n_slices > LORA_MAX_SLICES) { g_err = "n_slices outside [1, 4]"; return 0; }
        S = slices->n_slices;
    }
    size_t elems = 0;
    for (int32_t i = 0; i < n_segs; ++i) {
        const lora_segment_t& s = segs[i];
        if (!s.is_train || s.len <= 0) continue;
        if (s.adapter_id < 0 || s.adapter_id >= pool->n_adapters || !pool->rank) { g_err = "bad adapter id"; return 0; }
        elems += (size_t)s.len * (size_t)S * (size_t)pool->rank[s.adapter_id];
    }
    return elems * (dt == LORA_BF16 ? 2 : 4);
}

size_t lora_xa_size(lora_dtype_t dt, const lora_pool_t* pool, const lora_segment_t* segs, int32_t n_segs) {
    return lora_sliced_xa_size(dt, pool, nullptr, segs, n_segs);
}

int lora_set_trace_events(void* const* events) {
    if (!events) {
        g_trace_on = false;
        return LORA_OK;
    }
    for (int i = 0; i < 8; ++i) {
        if (!events[i]) return fail(LORA_ERR_INVALID_ARG, "trace events must be non-NULL");
        g_trace[i] = static_cast<cudaEvent_t>(events[i]);
    }
    g_trace_on = true;
    return LORA_OK;
}

int lora_selftest_wait_timeout(void* workspace, size_t ws_bytes, void* stream_) {
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255) != 0 || ws_bytes < 256)
        return fail(LORA_ERR_WORKSPACE, "workspace must be non-NULL, 256-byte aligned and at least 256 bytes");
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    CUDA_TRY(cudaMemsetAsync(workspace, 0, 256, stream));
    CUDA_TRY(selftest_timeout_launch(static_cast<int32_t*>(workspace), stream));
    return LORA_OK;
}

int lora_set_wait_limit(uint64_t ns) {
    if (ns < 1000000ull || ns > 60000000000ull)
        return fail(LORA_ERR_INVALID_ARG, "the wait limit must lie between 1 ms and 60 s");
    CUDA_TRY(set_wait_limit_ns(ns));
    return LORA_OK;
}

int lora_workspace_status(const void* workspace, void* stream) {
    if (!workspace) return fail(LORA_ERR_WORKSPACE, "workspace is NULL");
    CUDA_TRY(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)));
    int32_t st = 0;
    CUDA_TRY(cudaMemcpy(&st, workspace, sizeof(st), cudaMemcpyDeviceToHost));
    if (st != 0) return fail(st, "a kernel gave up a bounded wait; outputs of that call are incomplete");
    return LORA_OK;
}

int lora_plan_check(int32_t T, int32_t K, int32_t N, const lora_pool_t* pool, const lora_slices_t* slices,
                    const lora_segment_t* segs, int32_t n_segs, int32_t backward) {
    Problem p;
    std::string err;
    int rc = validate(T, K, N, LORA_BF16, pool, segs, n_segs, &p, &err, slices);
    if (rc != LORA_OK) return fail(rc, err);
    Plan pl;
    if (backward) plan_backward(p, true, true, true, true, &pl);
    else plan_forward(p, &pl);
    rc = check_plan(p, pl, backward != 0, &err);
    if (rc != LORA_OK) return fail(rc, err);
    return LORA_OK;
}

int lora_plan_describe(int32_t T, int32_t K, int32_t N, const lora_pool_t* pool, const lora_segment_t* segs,
                       int32_t n_segs, int32_t* n_tiles_out, int32_t* rows_out, int32_t* info_out, int32_t cap) {
    Problem p;
    std::string err;
    int rc = validate(T, K, N, LORA_BF16, pool, segs, n_segs, &p, &err);
    if (rc != LORA_OK) return fail(rc, err);
    Plan pl;
    plan_forward(p, &pl);
    const int32_t nt = int32_t(pl.tiles.size());
    if (n_tiles_out) *n_tiles_out = nt;
    if (nt > cap) return fail(LORA_ERR_LIMIT, "capacity too small for " + std::to_string(nt) + " tiles");
    for (int32_t i = 0; i < nt; ++i) {
        if (rows_out) std::memcpy(rows_out + (size_t)i * kTileM, &pl.rowmap[(size_t)i * kTileM], sizeof(int32_t) * kTileM);
        if (info_out) {
            info_out[4 * i + 0] = pl.tiles[i].a_src;
            info_out[4 * i + 1] = pl.tiles[i].nchunk;
            info_out[4 * i + 2] = pl.tiles[i].ext_k;
            info_out[4 * i + 3] = pl.tiles[i].a_src ? -1 : pl.tiles[i].a_row0;
        }
    }
    return LORA_OK;
}

}  // extern "C"

namespace {

// The forward's launch parameters: tensor maps of x, the gathered rows, W, Z, the pools and y, and the pointers the
// kernels use.  LORA_OK, LORA_ERR_CUDA (a tensor map the driver refused) or a LORA_DEBUG_CHECKS plan error.
int forward_params(int32_t T, int32_t K, int32_t N, const void* x, const void* Wt, const lora_pool_t* pool,
                   const Problem& p, const Plan& pl, const Layout& L, uint8_t* ws, void* y, bool save, void* xa_save,
                   uint32_t flags, KParams* out, std::string* err) {
    KParams& P = *out;
    std::memset(&P, 0, sizeof(P));
    if (!encode_2d(&P.tm_x, x, K, T, K, 64, 128, err)) return LORA_ERR_CUDA;
    if (pl.n_gtiles > 0 && !encode_2d(&P.tm_xg, ws + L.xg, K, (uint64_t)pl.n_gtiles * kTileM, K, 64, 128, err))
        return LORA_ERR_CUDA;
    if (!encode_2d(&P.tm_w, Wt, K, N, K, 64, 128, err)) return LORA_ERR_CUDA;
    if (pl.z_blocks > 0 &&
        !encode_2d(&P.tm_z, ws + L.z, 64, (uint64_t)pl.z_blocks * kTileM, 64, 64, 128, err, false))
        return LORA_ERR_CUDA;
    if (p.rows_a > 0 && !encode_2d(&P.tm_pa, pool->A, K, p.rows_a, K, 64, 8, err)) return LORA_ERR_CUDA;
    if (p.rows_b > 0 && !encode_2d(&P.tm_pb, pool->B, N, p.rows_b, N, 64, 8, err)) return LORA_ERR_CUDA;
    for (int h = 0; h < 3; ++h) {      // taller boxes for runs of consecutive atoms (shrink: A rows; main: B rows)
        if (p.rows_a > 0 && !encode_2d(&P.tm_pa_h[h], pool->A, K, p.rows_a, K, 64, 16u << h, err))
            return LORA_ERR_CUDA;
        if (p.rows_b > 0 && !encode_2d(&P.tm_pb_h[h], pool->B, N, p.rows_b, N, 64, 16u << h, err))
            return LORA_ERR_CUDA;
    }
    P.zin = ws + L.z;
    P.zout = ws + L.z;
    P.out = static_cast<__nv_bfloat16*>(y);
    P.out_ld = N;
    P.out_cols = N;
    if (!encode_out(&P.tm_out, y, N, T, N, err)) return LORA_ERR_CUDA;
    P.xa_save = save ? static_cast<__nv_bfloat16*>(xa_save) : nullptr;
    P.K = K;
    P.N = N;
    if (flags & LORA_DEBUG_CHECKS) {
        const int rc = check_plan(p, pl, false, err);
        if (rc != LORA_OK) return rc;
        P.debug = 1;
        P.db = DebugBounds{T, pl.z_blocks, save ? p.xa_elems : 0, 0, pl.part_cols * kTileM, pl.main_slots, 0, 0, T,
                           (int64_t)pl.n_gtiles * kTileM};
    }
    return LORA_OK;
}

// The forward of lora_mixed_forward and lora_sliced_forward (slices: NULL = one slice).
int forward_impl(int32_t T, int32_t K, int32_t N, lora_dtype_t dt, const void* x, const void* Wt,
                 const lora_pool_t* pool, const lora_slices_t* slices, const lora_segment_t* segs, int32_t n_segs,
                 void* y, void* xa_save, uint32_t flags, void* workspace, size_t ws_bytes, cudaStream_t stream) {
    Problem pv;
    Prepared* pr = nullptr;
    std::string err;
    int rc;
    if (dt == LORA_BF16) {
        rc = prepare(0, T, K, N, pool, slices, segs, n_segs, 0, &pr);
        if (rc != LORA_OK) return rc;
    } else {
        rc = validate(T, K, N, dt, pool, segs, n_segs, &pv, &err, slices);
        if (rc != LORA_OK) return fail(rc, err);
    }
    const Problem& p = pr ? pr->p : pv;
    if (flags & ~uint32_t(LORA_SAVE_XA | LORA_RECOMPUTE_XA | LORA_ACCUMULATE_GRAD | LORA_DEBUG_CHECKS))
        return fail(LORA_ERR_INVALID_ARG, "unknown flag bits");
    const bool save = (flags & LORA_SAVE_XA) && p.xa_elems > 0;
    if (T > 0 && (!x || !Wt || !y)) return fail(LORA_ERR_INVALID_ARG, "x, Wt and y must be non-NULL");
    if (p.n_adapters > 0 && (!pool->A || !pool->B)) return fail(LORA_ERR_INVALID_ARG, "pool A/B must be non-NULL");
    if (save && !xa_save) return fail(LORA_ERR_INVALID_ARG, "LORA_SAVE_XA needs xa_save");
    if (dt == LORA_BF16 && T > 0 &&
        (!aligned16(x) || !aligned16(Wt) || !aligned16(y) || (p.n_adapters && (!aligned16(pool->A) || !aligned16(pool->B)))))
        return fail(LORA_ERR_ALIGNMENT, "x, Wt, y, A and B must be 16-byte aligned");

    if (dt == LORA_F32) {
        Plan empty;
        Layout L = layout_of(p, empty, false);
        rc = check_workspace(workspace, ws_bytes, L.total);
        if (rc) return rc;
        if (T == 0) return LORA_OK;
        F32Blob fb;
        f32_layout(p, L.simt, &fb);
        uint8_t* w = static_cast<uint8_t*>(workspace);
        CUDA_TRY(cudaMemsetAsync(w + L.status, 0, 256, stream));
        rc = stage_copy(w + fb.tok, fb.bytes.data(), fb.bytes.size(), stream);
        if (rc) return rc;
        F32Args a{};
        a.T = T; a.K = K; a.N = N;
        a.x = static_cast<const float*>(x); a.Wt = static_cast<const float*>(Wt);
        a.A = static_cast<const float*>(pool->A); a.B = static_cast<const float*>(pool->B);
        a.ad = reinterpret_cast<const AdapterRec*>(w + fb.ad);
        a.tok_ad = reinterpret_cast<const int32_t*>(w + fb.tok);
        a.segs = reinterpret_cast<const F32Seg*>(w + fb.segs);
        a.n_segs = int32_t(p.segs.size());
        a.xa = reinterpret_cast<float*>(w + fb.xa);
        a.y = static_cast<float*>(y);
        a.xa_save = save ? static_cast<float*>(xa_save) : nullptr;
        a.xa_elems = p.xa_elems;
        CUDA_TRY(f32_forward(a, stream));
        return LORA_OK;
    }

    const Plan& pl = pr->pl;
    const Layout& L = pr->L;
    rc = check_workspace(workspace, ws_bytes, L.total);
    if (rc) return rc;
    if (T == 0) return LORA_OK;
    const int sms = sm_count();
    if (sms <= 0) return fail(LORA_ERR_CUDA, "no CUDA device available");
    assign_for(pr, sms);
    const int(&grid)[3] = pr->grid;
    const std::vector<uint8_t>& blob = pr->blob;

    uint8_t* ws = static_cast<uint8_t*>(workspace);
    KParams P;
    std::vector<uintptr_t> key = {uintptr_t(x), uintptr_t(Wt), uintptr_t(pool->A), uintptr_t(pool->B),
                                  uintptr_t(workspace), uintptr_t(y), uintptr_t(save ? xa_save : nullptr), flags};
    if (const KParams* c = cached_params(pr, key)) {
        P = *c;
    } else {
        rc = forward_params(T, K, N, x, Wt, pool, p, pl, L, ws, y, save, xa_save, flags, &P, &err);
        if (rc != LORA_OK) return fail(rc, err);
        keep_params(pr, P, std::move(key));
    }
    const SimtDebug dbg{P.debug, reinterpret_cast<int32_t*>(ws + L.status), T, (int64_t)pl.n_gtiles * kTileM,
                        pl.z_blocks, P.db.xa_elems, 0};

    rc = begin_call(L, pl, workspace, blob.size(), blob.data(), stream);
    if (rc) return rc;
    CUDA_TRY(trace(0, 0, stream));
    const int32_t* grows = reinterpret_cast<const int32_t*>(ws + L.rowmap) + (size_t)pl.g_tile0 * kTileM;
    if (!pl.bgmv.empty())       // the CUDA-core decode shrink, which also fills the gathered buffer
        CUDA_TRY(bgmv_shrink(x, grows, ws + L.xg, K, pool->A, reinterpret_cast<const BgmvGroup*>(ws + L.bgmv),
                             int32_t(pl.bgmv.size()), reinterpret_cast<const Chunk*>(ws + L.chunks),
                             reinterpret_cast<const TileDesc*>(ws + L.tiles), p.S, ws + L.z, dbg, stream));
    else if (pl.n_gtiles > 0)
        CUDA_TRY(gather_rows(x, K, grows, ws + L.xg, pl.n_gtiles * kTileM, dbg, stream));
    CUDA_TRY(launch_group(0, &P, ws, L, grid, stream));
    CUDA_TRY(trace(0, 1, stream));
    CUDA_TRY(trace(1, 0, stream));
    CUDA_TRY(launch_group(1, &P, ws, L, grid, stream));
    CUDA_TRY(launch_reduce(pl, P, ws, L, stream));
    CUDA_TRY(trace(1, 1, stream));
    return LORA_OK;
}

// The backward's launch parameters: tensor maps of x, dY, W, the pools, the transposed xA / dYB buffers, Z, every
// fine-tuning segment's rows of x and dY and dX, and the pointers the kernels use.  LORA_OK, LORA_ERR_CUDA (a tensor
// map the driver refused) or a LORA_DEBUG_CHECKS plan error.
int backward_params(int32_t T, int32_t K, int32_t N, const void* x, const void* Wt, const lora_pool_t* pool,
                    const void* dY, void* dX, float* dA, float* dB, bool acc, bool recompute, bool per_segment,
                    const Problem& p, const Plan& pl, const Layout& L, uint8_t* ws, uint32_t flags, KParams* out,
                    std::string* err) {
    KParams& P = *out;
    std::memset(&P, 0, sizeof(P));
    const uint64_t Pcols = (uint64_t)pl.tcols;
    if (!encode_2d(&P.tm_x, x, K, T, K, 64, 128, err)) return LORA_ERR_CUDA;
    if (!encode_2d(&P.tm_dy, dY, N, T, N, 64, 128, err)) return LORA_ERR_CUDA;
    if (!encode_2d(&P.tm_w, Wt, K, N, K, 64, 64, err)) return LORA_ERR_CUDA;
    P.w3 = (LORA_W3 && encode_w3(&P.tm_w3, Wt, K, N)) ? 1 : 0;      // else two 2-D boxes per stage
    if (!encode_2d(&P.tm_pa, pool->A, K, p.rows_a, K, 64, 8, err)) return LORA_ERR_CUDA;
    if (!encode_2d(&P.tm_pb, pool->B, N, p.rows_b, N, 64, 8, err)) return LORA_ERR_CUDA;
    for (int h = 0; h < 3; ++h) {      // taller boxes for runs of consecutive atoms (shrinks and the dX pass)
        if (!encode_2d(&P.tm_pa_h[h], pool->A, K, p.rows_a, K, 64, 16u << h, err)) return LORA_ERR_CUDA;
        if (!encode_2d(&P.tm_pb_h[h], pool->B, N, p.rows_b, N, 64, 16u << h, err)) return LORA_ERR_CUDA;
    }
    const uint64_t trows = (uint64_t)p.S * LORA_MAX_RANK;
    if (!encode_2d(&P.tm_xat, ws + L.xat, Pcols, trows, Pcols, 64, 8, err)) return LORA_ERR_CUDA;
    if (!encode_2d(&P.tm_dybt, ws + L.dybt, Pcols, trows, Pcols, 64, 8, err)) return LORA_ERR_CUDA;
    if (pl.z_blocks > 0 &&
        !encode_2d(&P.tm_z, ws + L.z, 64, (uint64_t)pl.z_blocks * kTileM, 64, 64, 128, err, false))
        return LORA_ERR_CUDA;
    const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
    const __nv_bfloat16* db = static_cast<const __nv_bfloat16*>(dY);
    for (size_t q = 0; q < pl.tsegs.size(); ++q) {
        const TrainSeg& s = pl.tsegs[q];
        if (!encode_2d(&P.tm_seg_dy[q], db + (size_t)s.start * N, N, s.len, N, 64, 64, err)) return LORA_ERR_CUDA;
        if (!encode_2d(&P.tm_seg_x[q], xb + (size_t)s.start * K, K, s.len, K, 64, 64, err)) return LORA_ERR_CUDA;
    }
    P.zin = ws + L.z;
    P.zout = ws + L.z;
    P.out = static_cast<__nv_bfloat16*>(dX);
    P.out_ld = K;
    P.out_cols = K;
    if (dX != nullptr && !encode_out(&P.tm_out, dX, K, T, K, err)) return LORA_ERR_CUDA;
    P.xat = reinterpret_cast<__nv_bfloat16*>(ws + L.xat);
    P.dybt = reinterpret_cast<__nv_bfloat16*>(ws + L.dybt);
    P.t_ld = int32_t(Pcols);
    P.dA = dA;
    P.dB = dB;
    P.K = K;
    P.N = N;
    P.accumulate = acc ? 1 : 0;
    P.seg_flags = per_segment ? reinterpret_cast<const int32_t*>(ws + L.seg_flags) : nullptr;
    if (flags & LORA_DEBUG_CHECKS) {
        const int rc = check_plan(p, pl, true, err);
        if (rc != LORA_OK) return rc;
        P.debug = 1;
        P.db = DebugBounds{T, pl.z_blocks, recompute ? 0 : p.xa_elems, (int64_t)p.S * LORA_MAX_RANK * pl.tcols,
                           pl.part_cols * kTileM, pl.main_slots, p.rows_a * K, p.rows_b * N, T, 0};
    }
    return LORA_OK;
}

// The backward of lora_mixed_backward and lora_mixed_backward_flagged (xa_valid: device flag table or null).
int backward_impl(int32_t T, int32_t K, int32_t N, lora_dtype_t dt, const void* x, const void* Wt,
                  const lora_pool_t* pool, const lora_slices_t* slices, const lora_segment_t* segs, int32_t n_segs,
                  const void* dY, const void* xa_saved, const int32_t* xa_valid, void* dX, float* dA, float* dB,
                  uint32_t flags, void* workspace, size_t ws_bytes, cudaStream_t stream) {
    const bool per_segment = (xa_valid != nullptr);
    const bool recompute = !per_segment && ((xa_saved == nullptr) || (flags & LORA_RECOMPUTE_XA));
    Problem pv;
    Prepared* pr = nullptr;
    std::string err;
    int rc;
    if (dt == LORA_BF16) {
        const int32_t opts = (dX != nullptr) | (dA != nullptr) << 1 | (dB != nullptr) << 2 | int32_t(recompute) << 3 |
                             int32_t(per_segment) << 4;
        rc = prepare(1, T, K, N, pool, slices, segs, n_segs, opts, &pr);
        if (rc != LORA_OK) return rc;
    } else {
        rc = validate(T, K, N, dt, pool, segs, n_segs, &pv, &err, slices);
        if (rc != LORA_OK) return fail(rc, err);
    }
    const Problem& p = pr ? pr->p : pv;
    if (flags & ~uint32_t(LORA_SAVE_XA | LORA_RECOMPUTE_XA | LORA_ACCUMULATE_GRAD | LORA_DEBUG_CHECKS))
        return fail(LORA_ERR_INVALID_ARG, "unknown flag bits");
    if (per_segment && (xa_saved == nullptr || (flags & LORA_RECOMPUTE_XA)))
        return fail(LORA_ERR_INVALID_ARG, "a flag table needs xa_saved and excludes LORA_RECOMPUTE_XA");
    const bool acc = (flags & LORA_ACCUMULATE_GRAD) != 0;
    if (p.n_train > 0) {
        if (!x || !Wt || !dY) return fail(LORA_ERR_INVALID_ARG, "x, Wt and dY must be non-NULL");
        if (!pool->A || !pool->B) return fail(LORA_ERR_INVALID_ARG, "pool A/B must be non-NULL");
        if (dt == LORA_BF16 && (!aligned16(x) || !aligned16(Wt) || !aligned16(dY) || (dX && !aligned16(dX)) ||
                                !aligned16(pool->A) || !aligned16(pool->B)))
            return fail(LORA_ERR_ALIGNMENT, "x, Wt, dY, dX, A and B must be 16-byte aligned");
        if ((dA && (reinterpret_cast<uintptr_t>(dA) & 3)) || (dB && (reinterpret_cast<uintptr_t>(dB) & 3)))
            return fail(LORA_ERR_ALIGNMENT, "dA and dB must be 4-byte aligned");
    }

    if (dt == LORA_F32) {
        Plan empty;
        Layout L = layout_of(p, empty, true);
        rc = check_workspace(workspace, ws_bytes, L.total);
        if (rc) return rc;
        if (p.n_train == 0) return LORA_OK;
        F32Blob fb;
        f32_layout(p, L.simt, &fb);
        uint8_t* w = static_cast<uint8_t*>(workspace);
        CUDA_TRY(cudaMemsetAsync(w + L.status, 0, 256, stream));
        rc = stage_copy(w + fb.tok, fb.bytes.data(), fb.bytes.size(), stream);
        if (rc) return rc;
        if (per_segment)        // the call's view of the flag table, taken when the call reaches the GPU
            CUDA_TRY(cudaMemcpyAsync(w + L.seg_flags, xa_valid, sizeof(int32_t) * p.n_train,
                                     cudaMemcpyDeviceToDevice, stream));
        // adapter groups in order of first appearance by start (host arrays)
        std::vector<int32_t> g_ad, g_r;
        std::vector<float> g_s;
        std::vector<int64_t> g_ao, g_bo;
        int32_t train_tokens = 0;
        for (const auto& s : p.segs) {
            if (!s.is_train) continue;
            train_tokens += s.len;
            if (std::find(g_ad.begin(), g_ad.end(), s.adapter_id) == g_ad.end()) {
                g_ad.push_back(s.adapter_id);
                g_r.push_back(p.rank[s.adapter_id]);
                g_s.push_back(p.scale[s.adapter_id]);
                g_ao.push_back(p.a_off[s.adapter_id]);
                g_bo.push_back(p.b_off[s.adapter_id]);
            }
        }
        F32Args a{};
        a.T = T; a.K = K; a.N = N;
        a.x = static_cast<const float*>(x); a.Wt = static_cast<const float*>(Wt);
        a.A = static_cast<const float*>(pool->A); a.B = static_cast<const float*>(pool->B);
        a.ad = reinterpret_cast<const AdapterRec*>(w + fb.ad);
        a.tok_ad = reinterpret_cast<const int32_t*>(w + fb.tok);
        a.segs = reinterpret_cast<const F32Seg*>(w + fb.segs);
        a.n_segs = int32_t(p.segs.size());
        a.xa = reinterpret_cast<float*>(w + fb.xa);
        a.dyb = reinterpret_cast<float*>(w + fb.dyb);
        a.xa_saved = recompute ? nullptr : static_cast<const float*>(xa_saved);
        a.seg_flags = per_segment ? reinterpret_cast<const int32_t*>(w + L.seg_flags) : nullptr;
        a.xa_elems = p.xa_elems;
        a.dY = static_cast<const float*>(dY);
        a.dX = static_cast<float*>(dX);
        a.dA = dA; a.dB = dB;
        a.accumulate = acc ? 1 : 0;
        a.train_tokens = train_tokens;
        a.n_groups = int32_t(g_ad.size());
        a.group_adapter = g_ad.data(); a.group_r = g_r.data(); a.group_scale = g_s.data();
        a.group_a_off = g_ao.data(); a.group_b_off = g_bo.data();
        CUDA_TRY(f32_backward(a, stream));
        return LORA_OK;
    }

    const Plan& pl = pr->pl;
    const Layout& L = pr->L;
    rc = check_workspace(workspace, ws_bytes, L.total);
    if (rc) return rc;
    if (p.n_train == 0) return LORA_OK;
    const int sms = sm_count();
    if (sms <= 0) return fail(LORA_ERR_CUDA, "no CUDA device available");
    assign_for(pr, sms);
    const int(&grid)[3] = pr->grid;
    const std::vector<uint8_t>& blob = pr->blob;

    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const uint64_t Pcols = (uint64_t)pl.tcols;
    int32_t max_len = 0;
    for (const TrainSeg& s : pl.tsegs) max_len = std::max(max_len, s.len);
    KParams P;
    std::vector<uintptr_t> key = {uintptr_t(x),  uintptr_t(Wt), uintptr_t(pool->A),  uintptr_t(pool->B),
                                  uintptr_t(dY), uintptr_t(dX), uintptr_t(dA),       uintptr_t(dB),
                                  uintptr_t(workspace), flags, uintptr_t(acc), uintptr_t(recompute),
                                  uintptr_t(per_segment)};
    if (const KParams* c = cached_params(pr, key)) {
        P = *c;
    } else {
        rc = backward_params(T, K, N, x, Wt, pool, dY, dX, dA, dB, acc, recompute, per_segment, p, pl, L, ws, flags,
                             &P, &err);
        if (rc != LORA_OK) return fail(rc, err);
        keep_params(pr, P, std::move(key));
    }
    const SimtDebug dbg{P.debug, reinterpret_cast<int32_t*>(ws + L.status), T, 0, pl.z_blocks, P.db.xa_elems,
                        P.db.t_elems};

    rc = begin_call(L, pl, workspace, blob.size(), blob.data(), stream);
    if (rc) return rc;
    if (per_segment)            // the call's view of the flag table, taken when the call reaches the GPU
        CUDA_TRY(cudaMemcpyAsync(ws + L.seg_flags, xa_valid, sizeof(int32_t) * p.n_train, cudaMemcpyDeviceToDevice,
                                 stream));
    CUDA_TRY(trace(2, 0, stream));
    if (!recompute && dB) {
        int32_t max_r = 0;
        for (const TrainSeg& s : pl.tsegs) max_r = std::max(max_r, s.r);
        CUDA_TRY(xat_from_saved(xa_saved, reinterpret_cast<const TrainSeg*>(ws + L.tsegs), int32_t(pl.tsegs.size()),
                                max_len, max_r, ws + L.xat, int32_t(Pcols), P.seg_flags, dbg, stream));
    }
    CUDA_TRY(launch_group(0, &P, ws, L, grid, stream));
    CUDA_TRY(trace(2, 1, stream));
    CUDA_TRY(trace(3, 0, stream));
    CUDA_TRY(launch_group(1, &P, ws, L, grid, stream));
    CUDA_TRY(launch_reduce(pl, P, ws, L, stream));
    CUDA_TRY(launch_group(2, &P, ws, L, grid, stream));
    CUDA_TRY(trace(3, 1, stream));
    return LORA_OK;
}

}  // namespace

extern "C" {

int lora_mixed_forward(int32_t T, int32_t K, int32_t N, lora_dtype_t dt, const void* x, const void* Wt,
                       const lora_pool_t* pool, const lora_segment_t* segs, int32_t n_segs, void* y, void* xa_save,
                       uint32_t flags, void* workspace, size_t ws_bytes, void* stream) {
    return forward_impl(T, K, N, dt, x, Wt, pool, nullptr, segs, n_segs, y, xa_save, flags, workspace, ws_bytes,
                        static_cast<cudaStream_t>(stream));
}

int lora_sliced_forward(int32_t T, int32_t K, int32_t N, lora_dtype_t dt, const void* x, const void* Wt,
                        const lora_pool_t* pool, const lora_slices_t* slices, const lora_segment_t* segs,
                        int32_t n_segs, void* y, void* xa_save, uint32_t flags, void* workspace, size_t ws_bytes,
                        void* stream) {
    if (!slices) return fail(LORA_ERR_INVALID_ARG, "slices is NULL");
    return forward_impl(T, K, N, dt, x, Wt, pool, slices, segs, n_segs, y, xa_save, flags, workspace, ws_bytes,
                        static_cast<cudaStream_t>(stream));
}

int lora_mixed_backward(int32_t T, int32_t K, int32_t N, lora_dtype_t dt, const void* x, const void* Wt,
                        const lora_pool_t* pool, const lora_segment_t* segs, int32_t n_segs, const void* dY,
                        const void* xa_saved, void* dX, float* dA, float* dB, uint32_t flags, void* workspace,
                        size_t ws_bytes, void* stream) {
    return backward_impl(T, K, N, dt, x, Wt, pool, nullptr, segs, n_segs, dY, xa_saved, nullptr, dX, dA, dB, flags,
                         workspace, ws_bytes, static_cast<cudaStream_t>(stream));
}

int lora_sliced_backward(int32_t T, int32_t K, int32_t N, lora_dtype_t dt, const void* x, const void* Wt,
                         const lora_pool_t* pool, const lora_slices_t* slices, const lora_segment_t* segs,
                         int32_t n_segs, const void* dY, const void* xa_saved, void* dX, float* dA, float* dB,
                         uint32_t flags, void* workspace, size_t ws_bytes, void* stream) {
    if (!slices) return fail(LORA_ERR_INVALID_ARG, "slices is NULL");
    return backward_impl(T, K, N, dt, x, Wt, pool, slices, segs, n_segs, dY, xa_saved, nullptr, dX, dA, dB, flags,
                         workspace, ws_bytes, static_cast<cudaStream_t>(stream));
}

int lora_mixed_backward_flagged(int32_t T, int32_t K, int32_t N, lora_dtype_t dt, const void* x, const void* Wt,
                                const lora_pool_t* pool, const lora_segment_t* segs, int32_t n_segs, const void* dY,
                                const void* xa_saved, const int32_t* xa_valid, void* dX, float* dA, float* dB,
                                uint32_t flags, void* workspace, size_t ws_bytes, void* stream) {
    if (!xa_valid) return fail(LORA_ERR_INVALID_ARG, "xa_valid (device flag table) is NULL");
    return backward_impl(T, K, N, dt, x, Wt, pool, nullptr, segs, n_segs, dY, xa_saved, xa_valid, dX, dA, dB, flags,
                         workspace, ws_bytes, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
