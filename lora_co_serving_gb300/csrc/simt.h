// simt.h -- CUDA-core helper kernels and the float32 path.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.h"
#include "lora_mixed.h"

namespace lora {

struct AdapterRec {     // float32 path: one pool entry
    int64_t a_off, b_off;
    int32_t r;
    float scale;
    int32_t pad0, pad1;
};

struct F32Seg {         // float32 path: one segment, increasing start
    int32_t start, len, adapter, is_train;
    int32_t xoff;       // fine-tuning segments: offset of the [len, r] block in the saved-activation buffer
    int32_t order;      // fine-tuning segments: index among them in increasing start order
    int32_t pad1, pad2;
};

struct F32Args {
    int32_t T, K, N;
    const float* x;
    const float* Wt;
    const float* A;
    const float* B;
    const AdapterRec* ad;
    const int32_t* tok_ad;
    const F32Seg* segs;
    int32_t n_segs;
    float* xa;               // scratch [T, 128]
    float* dyb;              // scratch [T, 128]
    float* y;
    float* xa_save;
    const float* xa_saved;
    const int32_t* seg_flags;       // device snapshot of the per-segment flag table, or null
    int64_t xa_elems;
    const float* dY;
    float* dX;
    float* dA;
    float* dB;
    int32_t accumulate;
    int32_t train_tokens;
    int32_t n_groups;
    const int32_t* group_adapter;   // HOST arrays
    const int32_t* group_r;
    const float* group_scale;
    const int64_t* group_a_off;
    const int64_t* group_b_off;
};

// LORA_DEBUG_CHECKS for the CUDA-core kernels: when `on`, store (and row) indices are checked against these extents;
// a failing check skips the access and records LORA_ERR_BOUNDS in *status.
struct SimtDebug {
    int32_t on;
    int32_t* status;
    int64_t x_rows, g_rows, z_blocks, xa_elems, t_elems;
};

cudaError_t gather_rows(const void* x, int32_t K, const int32_t* rows, void* out, int32_t n_rows, const SimtDebug& dbg,
                        cudaStream_t s);
// Z = bf16(s x A) of the gathered rows listed in `groups` (device arrays; S slices), written into the Z images of
// their tiles (zout: the zeroed Z blocks); also fills the gathered buffer xg from x (grows: token row of every
// gathered row, -1 for none).
cudaError_t bgmv_shrink(const void* x, const int32_t* grows, void* xg, int32_t K, const void* A,
                        const BgmvGroup* groups, int32_t n_groups, const Chunk* chunks, const TileDesc* tiles, int32_t S,
                        void* zout, const SimtDebug& dbg, cudaStream_t s);
cudaError_t xat_from_saved(const void* xa_saved, const TrainSeg* tsegs, int32_t n_tsegs, int32_t max_len,
                           int32_t max_r, void* xat, int32_t P, const int32_t* seg_flags, const SimtDebug& dbg,
                           cudaStream_t s);
cudaError_t f32_forward(const F32Args& a, cudaStream_t s);
cudaError_t f32_backward(const F32Args& a, cudaStream_t s);

}  // namespace lora
