/*
 * lora_mixed.h -- C ABI of the mixed-batch multi-adapter LoRA linear layer.
 *
 * One call computes, for a batch whose tokens are split into segments that
 * each name their own adapter (decode tokens, prefill segments and
 * fine-tuning segments alike):
 *
 *     y[t,:] = x[t,:] W + s_a * (x[t,:] A_a) B_a          (row-vector form)
 *
 * which is the LoRA layer W_eff = W + BA ("DeltaServe: Host-Agnostic
 * Co-Serving of Inference and Fine-Tuning for LLMs", section 2.2; "MOLT: A
 * Fine-Grained GPU Memory Sharing System for LLM Serving with Opportunistic
 * Fine-Tuning", section 2.1, h(x) = Wx + BAx) batched over many adapters in
 * one base-model pass (multi-LoRA batching, DeltaServe section 2.2), with
 * fine-tuning samples carried as ordinary prefill-like entries on their own
 * adapter (DeltaServe section 3.2, "Mixed forward batch").  A second call
 * computes the LoRA backward of the fine-tuning segments (DeltaServe section
 * 3.2, "Backward subprocess": LoRA gradients from captured activations, with
 * unsaved intermediates recomputed):
 *
 *     v      = dY B_a^T
 *     dX     = dY W^T + s_a * v A_a^T
 *     dB_a  += s_a * (x A_a)^T dY          summed over a's fine-tuning tokens
 *     dA_a  += s_a * x^T v                 (stored transposed, see below)
 *
 * Layouts (all row-major, element offsets, no padding):
 *   x   [T,K]          layer input, one row per token
 *   Wt  [N,K]          the frozen weight stored transposed (nn.Linear layout)
 *   A   pool of blocks; adapter a's block is A_a stored as [r_a, K]
 *       (the paper's A in R^{r x k}), starting at element a_off[a]
 *   B   pool of blocks; adapter a's block is [r_a, N] (the paper's B^T),
 *       starting at element b_off[a]
 *   y   [T,N]
 *   dA, dB  float32, shaped exactly like the A and B pools (same offsets)
 *
 * Conventions shared by every entry point:
 *   - Device pointers unless marked HOST.  The caller owns every buffer; the
 *     library allocates no device memory and keeps no pointer after a call.
 *   - Everything is validated on the host before anything is launched.  On
 *     error the call returns a negative LORA_ERR_* code, writes nothing,
 *     launches nothing, and lora_last_error() describes the problem.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and the call returns without waiting for it.  Segment-table
 *     planning happens on the host; the plan travels into `workspace` by an
 *     asynchronous copy from a small library-owned ring of pinned host
 *     buffers (allocated on first use, per device; a slot is reused only
 *     after its previous copy has completed), so the host-side segment array
 *     may be reused as soon as the call returns.
 *   - Two calls that share a workspace must not overlap on the GPU.
 *   - CUDA graphs: a call made while `stream` is being captured records the same work into the graph and
 *     blocks on nothing; its plan is uploaded from a pinned host copy of its own that the library keeps for
 *     the life of the process (one per captured call), so the graph may be replayed any number of times, at
 *     any later point.  A replay reads the device buffers and the workspace that were captured.
 *   - Kernels never wait without a bound.  If one gives up, it records a
 *     nonzero code in the workspace's status word; lora_workspace_status()
 *     reads it.
 */
#ifndef LORA_MIXED_H
#define LORA_MIXED_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* One batch segment: tokens [start, start+len) use adapter `adapter_id`
 * (-1: base projection only).  is_train != 0 marks a fine-tuning segment;
 * it must name an adapter (>= 0).  The segments of a call must cover [0, T)
 * exactly once, in any order; zero-length segments are ignored. */
typedef struct lora_segment {
    int32_t start;
    int32_t len;
    int32_t adapter_id;
    int32_t is_train;
} lora_segment_t;

/* The stacked adapter pool (MOLT section 2.1: each adapter holds r(d+k)
 * trainable values; here each adapter keeps its own rank, no padding to a
 * common maximum). */
typedef struct lora_pool {
    const void* A;          /* device, element type of the call; blocks [r_a, K] */
    const void* B;          /* device, element type of the call; blocks [r_a, N] */
    const int64_t* a_off;   /* HOST [n_adapters]; a multiple of K */
    const int64_t* b_off;   /* HOST [n_adapters]; a multiple of N */
    const int32_t* rank;    /* HOST [n_adapters]; 1 <= r_a <= 128 */
    const float* scale;     /* HOST [n_adapters]; s_a (LoRA alpha / r) */
    int32_t n_adapters;
} lora_pool_t;

typedef enum lora_dtype { LORA_BF16 = 0, LORA_F32 = 1 } lora_dtype_t;

/* flags */
enum {
    LORA_SAVE_XA = 1,          /* forward: write x A_a of fine-tuning rows to xa_save */
    LORA_RECOMPUTE_XA = 2,     /* backward: recompute x A_a even if xa_saved is given */
    LORA_ACCUMULATE_GRAD = 4,  /* backward: add into dA/dB instead of overwriting */
    LORA_DEBUG_CHECKS = 8      /* bf16 calls: before any launch the host checks every index of the call's plan
                                  against the buffer it addresses (LORA_ERR_BOUNDS on a violation, nothing
                                  launched), and every kernel checks each store index it derives from the plan;
                                  a failing store is skipped and LORA_ERR_BOUNDS recorded in the status word
                                  (lora_workspace_status).  Slower; a stand-in for a memory checker. */
};

/* return codes */
enum {
    LORA_OK = 0,
    LORA_ERR_INVALID_ARG = -1,  /* null pointer, negative size, bad flag combination */
    LORA_ERR_SEGMENTS = -2,     /* segments overlap, leave a gap, or leave [0,T) */
    LORA_ERR_ADAPTER = -3,      /* adapter id out of range, or pool offsets out of shape */
    LORA_ERR_TRAIN_BASE = -4,   /* fine-tuning segment on adapter -1 */
    LORA_ERR_ALIGNMENT = -5,    /* bf16: x/Wt/A/B/y/dY/dX not 16-byte aligned, or K, N not multiples of 8 */
    LORA_ERR_WORKSPACE = -6,    /* workspace missing, too small or not 256-byte aligned */
    LORA_ERR_DTYPE = -7,        /* unknown dtype */
    LORA_ERR_CUDA = -8,         /* a CUDA runtime call failed (message in lora_last_error) */
    LORA_ERR_RANK = -9,         /* rank outside [1, 128] */
    LORA_ERR_LIMIT = -10,       /* beyond a documented size limit (see below) */
    LORA_ERR_TIMEOUT = -11,     /* reported by lora_workspace_status: a kernel gave up waiting */
    LORA_ERR_BOUNDS = -12       /* LORA_DEBUG_CHECKS: a plan index outside its buffer (host check, or a kernel
                                   skipped a store and recorded it in the status word) */
};

/* Limits: T, K, N < 2^31; sum over segments of len*r fits in int32;
 * at most 48 fine-tuning segments per call; bf16 path: K, N multiples of 8. */
#define LORA_MAX_RANK 128
#define LORA_MAX_TRAIN_SEGMENTS 48

/* Bytes of device workspace that lora_mixed_forward and lora_mixed_backward
 * need for this segment table (the larger of the two).  Returns 0 and sets
 * lora_last_error on invalid input; a valid empty batch still needs a small
 * nonzero workspace (the status word). */
size_t lora_workspace_size(int32_t T, int32_t K, int32_t N, lora_dtype_t dt, const lora_pool_t* pool,
                           const lora_segment_t* segs /* HOST */, int32_t n_segs);

/* Bytes of the saved-activation buffer: for every fine-tuning segment, in
 * increasing start order, a [len, r_a] row-major block of x A_a in the call's
 * element type (DeltaServe section 3.2: activation capture for the
 * fine-tuning rows of a mixed batch).  Returns 0 on invalid input. */
size_t lora_xa_size(lora_dtype_t dt, const lora_pool_t* pool, const lora_segment_t* segs /* HOST */,
                    int32_t n_segs);

/* Forward over every segment of the batch.
 *   x [T,K], Wt [N,K], y [T,N] in element type dt; y is written for all T rows.
 *   xa_save: with LORA_SAVE_XA, receives x A_a of the fine-tuning rows
 *            (layout of lora_xa_size); otherwise ignored, may be NULL.
 *   workspace: device, 256-byte aligned, >= lora_workspace_size bytes. */
int lora_mixed_forward(int32_t T, int32_t K, int32_t N, lora_dtype_t dt, const void* x, const void* Wt,
                       const lora_pool_t* pool, const lora_segment_t* segs /* HOST */, int32_t n_segs, void* y,
                       void* xa_save, uint32_t flags, void* workspace, size_t ws_bytes, void* stream);

/* LoRA backward of the fine-tuning segments.
 *   dY [T,N]: only fine-tuning rows are read.
 *   xa_saved: the forward's xa_save for the same segment table, or NULL to
 *             recompute x A_a (also recomputed under LORA_RECOMPUTE_XA).
 *   dX [T,K]: only fine-tuning rows are written.  May be NULL (skipped).
 *   dA, dB:   float32, pool-shaped.  Blocks of adapters with a fine-tuning
 *             segment are overwritten (or added to, LORA_ACCUMULATE_GRAD);
 *             all other entries are left untouched.  Contributions of
 *             several segments on one adapter are summed in a fixed order,
 *             so repeated calls give bitwise-identical results.  */
int lora_mixed_backward(int32_t T, int32_t K, int32_t N, lora_dtype_t dt, const void* x, const void* Wt,
                        const lora_pool_t* pool, const lora_segment_t* segs /* HOST */, int32_t n_segs,
                        const void* dY, const void* xa_saved, void* dX, float* dA, float* dB, uint32_t flags,
                        void* workspace, size_t ws_bytes, void* stream);

/* Forward pass for callers that cannot allocate device memory (no counterpart on the pages: this is a
 * deployment concern of this library, not part of the method).  Same arguments and results as
 * lora_mixed_forward, but its scratch lives in a fixed library-owned device array of
 * LORA_STATIC_WORKSPACE_BYTES, held by every GPU that loads the library until the process exits; the call
 * allocates nothing.  A batch whose forward scratch (the workspace lora_mixed_forward would need for it)
 * exceeds the array is rejected with LORA_ERR_LIMIT before any launch.  All calls share the array: two calls
 * that overlap on the GPU race and must be ordered by the caller.  Every call that is not being captured into
 * a CUDA graph looks up the array's address on the current device; a call made during a capture reuses the
 * address found last on that device, so make one call on the device before capturing (a captured call keeps
 * a pinned host copy of its plan, like every other entry point). */
#define LORA_STATIC_WORKSPACE_BYTES (64u << 20)
int lora_mixed_forward_static(int32_t T, int32_t K, int32_t N, lora_dtype_t dt, const void* x, const void* Wt,
                              const lora_pool_t* pool, const lora_segment_t* segs /* HOST */, int32_t n_segs,
                              void* y, void* xa_save, uint32_t flags, void* stream);

/* lora_workspace_status for the library-owned array of lora_mixed_forward_static on the current device: waits for
 * `stream`, then returns LORA_OK or LORA_ERR_TIMEOUT if a kernel of the last static call gave up a bounded wait
 * (that call's outputs are then incomplete).  Blocking.  No counterpart on the pages. */
int lora_static_status(void* stream);

/* AdamW hyperparameters for lora_adamw_step (DeltaServe section 4.1 trains with lr 1e-3, weight decay
 * 0.01; betas and eps are the usual 0.9, 0.999, 1e-8).  step is the 1-based update count. */
typedef struct lora_adamw {
    float lr;
    float beta1;
    float beta2;
    float eps;
    float weight_decay;
    int32_t step;
} lora_adamw_t;

/* The fine-tuning step after the backward: AdamW, in place, on the blocks of the listed adapters
 * (DeltaServe section 3.2, "Backward subprocess": optimizer updates applied directly to the shared adapter
 * weights):
 *     m <- b1 m + (1-b1) g;   v <- b2 v + (1-b2) g^2
 *     w <- w (1 - lr wd) - lr/(1-b1^step) * m / (sqrt(v)/sqrt(1-b2^step) + eps)
 *   A, B:       the pool's weights (device, element type dt), updated in place.
 *   A_master, B_master: optional fp32 master weights shaped like the pools (NULL: update A/B directly).
 *               With masters, AdamW runs on the masters and A/B receive them rounded to dt.
 *   dA, dB:     fp32 gradients shaped like the pools (lora_mixed_backward's outputs).
 *   mA, vA, mB, vB: fp32 first and second moments shaped like the pools, updated in place (zero before
 *               the first step).
 *   adapters:   HOST [n_upd] distinct adapter ids (at most 48); only their blocks are read or written.
 * Validated on the host; one launch on `stream`. */
int lora_adamw_step(lora_dtype_t dt, const lora_pool_t* pool, int32_t K, int32_t N, void* A, void* B, float* A_master,
                    float* B_master, const float* dA, const float* dB, float* mA, float* vA, float* mB, float* vB,
                    const int32_t* adapters /* HOST */, int32_t n_upd, const lora_adamw_t* hp, void* stream);

/* lora_mixed_backward with the save/recompute choice made per fine-tuning segment on the device, from a
 * flag table that another stream or process may rewrite between calls (in the spirit of MOLT section 4.3,
 * "flexible activation checkpointing": whether an activation's slot is still backed is known only when the
 * backward is dispatched, and unbacked activations are recomputed).
 *   xa_valid: device int32 [number of fine-tuning segments], in increasing segment-start order; nonzero =
 *             the segment's block of xa_saved holds its x A, zero = recompute it.  The call copies the table
 *             on its stream when it starts on the GPU; all its kernels use that copy.
 *   xa_saved: required (read only for flagged segments); LORA_RECOMPUTE_XA is not allowed.
 * Everything else as lora_mixed_backward. */
int lora_mixed_backward_flagged(int32_t T, int32_t K, int32_t N, lora_dtype_t dt, const void* x, const void* Wt,
                                const lora_pool_t* pool, const lora_segment_t* segs /* HOST */, int32_t n_segs,
                                const void* dY, const void* xa_saved, const int32_t* xa_valid, void* dX, float* dA,
                                float* dB, uint32_t flags, void* workspace, size_t ws_bytes, void* stream);

/* ---- Sliced (fused) projections ----
 * A decoder layer applies one adapter to several projections of the same input: DeltaServe section 4.1 puts
 * its fine-tuning adapter on every attention projection of Llama 3-8B, whose q, k and v projections all read
 * the layer's normalised hidden state (and an MLP's gate and up projections share theirs).  A sliced call
 * runs such projections as one layer over the concatenated weight: output columns [b_i, b_{i+1}) form slice
 * i, and each slice is an ordinary LoRA linear layer on the shared x:
 *
 *     y[:, b_i:b_{i+1}] = x W_i + s_a (x A_{a,i}) B_{a,i}
 *     dX = sum over slices of (dY_i W_i^T + s_a (dY_i B_{a,i}^T) A_{a,i}^T)       (dY_i = dY[:, b_i:b_{i+1}])
 *
 * Pool layout of a sliced call: adapter a's block in A stacks its down factors, slice i's [r_a, K] factor at
 * rows [i r_a, (i+1) r_a) (n_slices * r_a rows from a_off[a]); its block in B is [r_a, N], whose columns
 * [b_i, b_{i+1}) are slice i's up factor.  dA and dB are shaped like these pools.  The saved-activation
 * buffer holds, per fine-tuning segment in increasing start order, a [len, n_slices * r_a] block: slice i's
 * x A_{a,i} in columns [i r_a, (i+1) r_a).
 * Limits: bf16 only; 1 <= n_slices <= LORA_MAX_SLICES; col_bounds[0] = 0 < col_bounds[1] < ... <
 * col_bounds[n_slices] = N with the interior bounds multiples of 256.  A one-slice call is exactly the
 * corresponding lora_mixed_* call; slices = NULL means one slice. */
#define LORA_MAX_SLICES 4
typedef struct lora_slices {
    int32_t n_slices;
    const int32_t* col_bounds;   /* HOST [n_slices + 1] */
} lora_slices_t;

/* lora_workspace_size / lora_xa_size for a sliced layer. */
size_t lora_sliced_workspace_size(int32_t T, int32_t K, int32_t N, lora_dtype_t dt, const lora_pool_t* pool,
                                  const lora_slices_t* slices, const lora_segment_t* segs /* HOST */,
                                  int32_t n_segs);
size_t lora_sliced_xa_size(lora_dtype_t dt, const lora_pool_t* pool, const lora_slices_t* slices,
                           const lora_segment_t* segs /* HOST */, int32_t n_segs);

/* lora_mixed_forward / lora_mixed_backward of a sliced layer (same arguments otherwise; validation errors
 * for bad slices: LORA_ERR_INVALID_ARG, or LORA_ERR_DTYPE for a float32 call with more than one slice). */
int lora_sliced_forward(int32_t T, int32_t K, int32_t N, lora_dtype_t dt, const void* x, const void* Wt,
                        const lora_pool_t* pool, const lora_slices_t* slices, const lora_segment_t* segs /* HOST */,
                        int32_t n_segs, void* y, void* xa_save, uint32_t flags, void* workspace, size_t ws_bytes,
                        void* stream);
int lora_sliced_backward(int32_t T, int32_t K, int32_t N, lora_dtype_t dt, const void* x, const void* Wt,
                         const lora_pool_t* pool, const lora_slices_t* slices, const lora_segment_t* segs /* HOST */,
                         int32_t n_segs, const void* dY, const void* xa_saved, void* dX, float* dA, float* dB,
                         uint32_t flags, void* workspace, size_t ws_bytes, void* stream);

/* Message of the last failing call on this thread ("" if none). */
const char* lora_last_error(void);

/* Waits for `stream`, then reads the workspace status word of the last call
 * that used `workspace`: LORA_OK, or LORA_ERR_TIMEOUT if a kernel gave up a
 * bounded wait (its outputs are then incomplete).  Blocking. */
int lora_workspace_status(const void* workspace, void* stream);

/* Tracing (per-step timing, cf. DeltaServe section 3.1: engine hooks record
 * per-step execution time).  With `events` non-NULL, every later call on the
 * calling thread records events[2*i] just before and events[2*i+1] just after
 * its launch group i on the call's stream:
 *   i = 0: forward shrink pass (row gather + x A of every tile)
 *   i = 1: forward main pass   (x W plus the fused LoRA expand, writes y)
 *   i = 2: backward shrink pass (dY B^T, and x A when recomputed)
 *   i = 3: backward main pass   (dX, dA, dB)
 * `events` points to 8 cudaEvent_t handles owned by the caller; the array is
 * copied, the events must outlive the calls.  NULL switches tracing off.
 * A call that has no work in group i still records both of its events. */
int lora_set_trace_events(void* const* events);

/* Setup of the failure path (no counterpart on the pages): the limit, in nanoseconds, of every bounded wait in
 * the library's kernels on the current device (default 1 s; accepted 1 ms to 60 s).  A kernel whose wait runs
 * out records LORA_ERR_TIMEOUT in its workspace status word and returns (lora_workspace_status reports it); on a
 * GPU shared by time slicing or preemption, where a healthy call can be held off the GPU for longer than that,
 * raise it.  A synchronous copy to the device: call it before the calls it should govern, not while they run or
 * while a stream is being captured.  Returns LORA_OK, LORA_ERR_INVALID_ARG (out of range; nothing changes) or
 * LORA_ERR_CUDA. */
int lora_set_wait_limit(uint64_t ns);

/* Diagnostic of the failure path (no counterpart on the pages): launches one thread that waits, with the
 * same bounded wait as every kernel of the library, on a barrier that nothing ever completes.  After the
 * wait's limit (about one second unless lora_set_wait_limit changed it) it records LORA_ERR_TIMEOUT in the workspace status word and returns, so
 * lora_workspace_status() then reports LORA_ERR_TIMEOUT and the CUDA context stays usable.  Needs the first
 * 256 bytes of a 256-byte aligned workspace. */
int lora_selftest_wait_timeout(void* workspace, size_t ws_bytes, void* stream);

/* Diagnostic (no counterpart on the pages): plans a bf16 forward (backward = 0) or backward (backward != 0, every
 * output requested, x A recomputed) for this table and runs the host check of LORA_DEBUG_CHECKS on it: LORA_OK, a
 * validation error, or LORA_ERR_BOUNDS (lora_last_error names the index).  Host only; slices may be NULL. */
int lora_plan_check(int32_t T, int32_t K, int32_t N, const lora_pool_t* pool, const lora_slices_t* slices,
                    const lora_segment_t* segs /* HOST */, int32_t n_segs, int32_t backward);

/* Diagnostic: the forward tile plan of a segment table, for host-side tests.
 *   n_tiles_out: number of 128-row tiles.
 *   rows_out [cap*128]: token row held by each tile row, -1 for none.
 *   info_out [cap*4]: per tile {gathered (1: rows copied out of x, 0: a
 *              contiguous window of x), number of adapters, LoRA columns
 *              (sum of ranks rounded up to 16), first x row of the window}.
 * Returns LORA_OK, a validation error, or LORA_ERR_LIMIT if cap is short. */
int lora_plan_describe(int32_t T, int32_t K, int32_t N, const lora_pool_t* pool, const lora_segment_t* segs,
                       int32_t n_segs, int32_t* n_tiles_out, int32_t* rows_out, int32_t* info_out, int32_t cap);

#ifdef __cplusplus
}
#endif

#endif /* LORA_MIXED_H */
