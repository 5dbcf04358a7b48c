// adamw.cu -- lora_adamw_step: AdamW on the fine-tuning adapters' blocks of the pool, in place.
//
// After the LoRA backward, the fine-tuning step updates the shared adapter weights directly with AdamW
// ("DeltaServe: Host-Agnostic Co-Serving of Inference and Fine-Tuning for LLMs", section 3.2; AdamW with
// learning rate 1e-3 and weight decay 0.01 in section 4.1).  One element per thread and step:
//   m <- b1 m + (1-b1) g;  v <- b2 v + (1-b2) g^2;  w <- w (1 - lr wd) - (lr / (1-b1^t)) m / (sqrt(v)/sqrt(1-b2^t) + eps)
// on fp32 master weights when the caller keeps them (the bf16 pool then receives the rounded master), or on
// the pool itself.  Memory-bound: 16-byte vector accesses, one CTA row of the grid per adapter block.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>

#include <string>

#include "lora_mixed.h"
#include "plan.h"

namespace {

constexpr int kMaxBlocks = 2 * LORA_MAX_TRAIN_SEGMENTS;

struct AdamBlocks {
    int64_t off[kMaxBlocks];     // element offset of the block in its pool
    int64_t count[kMaxBlocks];   // elements (r_a * K or r_a * N), a multiple of 4 when vectorised
    int32_t is_b[kMaxBlocks];    // 0: A pool, 1: B pool
    int32_t n;
};

struct AdamArgs {
    void* w[2];                  // pool A / B (bf16 or fp32)
    float* master[2];            // fp32 master copies, or null
    const float* g[2];
    float* m[2];
    float* v[2];
    float b1, b2, one_minus_b1, one_minus_b2, decay, step_size, inv_sqrt_bc2, eps;
    int32_t bf16;
};

__device__ __forceinline__ void adam_one(float& w, float g, float& m, float& v, const AdamArgs& a) {
    m = fmaf(a.b1, m, a.one_minus_b1 * g);
    v = fmaf(a.b2, v, a.one_minus_b2 * g * g);
    const float denom = sqrtf(v) * a.inv_sqrt_bc2 + a.eps;
    w = w * a.decay - a.step_size * (m / denom);
}

__global__ void adamw_kernel(const __grid_constant__ AdamBlocks B, const __grid_constant__ AdamArgs a) {
    const int blk = blockIdx.y;
    const int p = B.is_b[blk];
    const int64_t off = B.off[blk], n = B.count[blk];
    const float* g = a.g[p] + off;
    float* m = a.m[p] + off;
    float* v = a.v[p] + off;
    float* mw = a.master[p] ? a.master[p] + off : nullptr;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i * 4 < n; i += stride) {
        const int64_t e = i * 4;
        if (e + 4 <= n && ((off + e) & 3) == 0) {
            const float4 gq = *reinterpret_cast<const float4*>(g + e);
            float4 mq = *reinterpret_cast<float4*>(m + e);
            float4 vq = *reinterpret_cast<float4*>(v + e);
            float w4[4];
            if (mw) {
                const float4 wq = *reinterpret_cast<const float4*>(mw + e);
                w4[0] = wq.x; w4[1] = wq.y; w4[2] = wq.z; w4[3] = wq.w;
            } else if (a.bf16) {
                const __nv_bfloat16* wb = static_cast<const __nv_bfloat16*>(a.w[p]) + off + e;
                for (int k = 0; k < 4; ++k) w4[k] = __bfloat162float(wb[k]);
            } else {
                const float4 wq = *reinterpret_cast<const float4*>(static_cast<const float*>(a.w[p]) + off + e);
                w4[0] = wq.x; w4[1] = wq.y; w4[2] = wq.z; w4[3] = wq.w;
            }
            adam_one(w4[0], gq.x, mq.x, vq.x, a);
            adam_one(w4[1], gq.y, mq.y, vq.y, a);
            adam_one(w4[2], gq.z, mq.z, vq.z, a);
            adam_one(w4[3], gq.w, mq.w, vq.w, a);
            *reinterpret_cast<float4*>(m + e) = mq;
            *reinterpret_cast<float4*>(v + e) = vq;
            if (mw) *reinterpret_cast<float4*>(mw + e) = make_float4(w4[0], w4[1], w4[2], w4[3]);
            if (a.bf16) {
                __nv_bfloat16* wb = static_cast<__nv_bfloat16*>(a.w[p]) + off + e;
                for (int k = 0; k < 4; ++k) wb[k] = __float2bfloat16_rn(w4[k]);
            } else if (!mw) {
                *reinterpret_cast<float4*>(static_cast<float*>(a.w[p]) + off + e) =
                    make_float4(w4[0], w4[1], w4[2], w4[3]);
            }
        } else {
            for (int64_t k = e; k < n && k < e + 4; ++k) {
                float w1;
                if (mw) w1 = mw[k];
                else if (a.bf16) w1 = __bfloat162float(static_cast<const __nv_bfloat16*>(a.w[p])[off + k]);
                else w1 = static_cast<const float*>(a.w[p])[off + k];
                float m1 = m[k], v1 = v[k];
                adam_one(w1, g[k], m1, v1, a);
                m[k] = m1;
                v[k] = v1;
                if (mw) mw[k] = w1;
                if (a.bf16) static_cast<__nv_bfloat16*>(a.w[p])[off + k] = __float2bfloat16_rn(w1);
                else if (!mw) static_cast<float*>(a.w[p])[off + k] = w1;
            }
        }
    }
}

}  // namespace

extern "C" int lora_adamw_step(lora_dtype_t dt, const lora_pool_t* pool, int32_t K, int32_t N, void* A, void* B,
                               float* A_master, float* B_master, const float* dA, const float* dB, float* mA,
                               float* vA, float* mB, float* vB, const int32_t* adapters, int32_t n_upd,
                               const lora_adamw_t* hp, void* stream) {
    if (dt != LORA_BF16 && dt != LORA_F32) { lora::set_last_error("unknown dtype"); return LORA_ERR_DTYPE; }
    if (!pool || !hp || K <= 0 || N <= 0 || n_upd < 0 || (n_upd > 0 && !adapters)) {
        lora::set_last_error("lora_adamw_step: NULL argument or bad size");
        return LORA_ERR_INVALID_ARG;
    }
    if (n_upd > LORA_MAX_TRAIN_SEGMENTS) {
        lora::set_last_error("lora_adamw_step: more than 48 adapters in one call");
        return LORA_ERR_LIMIT;
    }
    if (hp->step < 1 || !(hp->lr >= 0.f) || !(hp->beta1 >= 0.f && hp->beta1 < 1.f) ||
        !(hp->beta2 >= 0.f && hp->beta2 < 1.f) || !(hp->eps > 0.f)) {
        lora::set_last_error("lora_adamw_step: step must be >= 1, lr >= 0, betas in [0,1), eps > 0");
        return LORA_ERR_INVALID_ARG;
    }
    if (n_upd == 0) return LORA_OK;
    if (!A || !B || !dA || !dB || !mA || !vA || !mB || !vB) {
        lora::set_last_error("lora_adamw_step: weights, gradients and moments must be non-NULL");
        return LORA_ERR_INVALID_ARG;
    }
    AdamBlocks blocks{};
    int64_t maxc = 0;
    for (int32_t i = 0; i < n_upd; ++i) {
        const int32_t a = adapters[i];
        if (a < 0 || a >= pool->n_adapters) {
            lora::set_last_error("lora_adamw_step: adapter id out of range");
            return LORA_ERR_ADAPTER;
        }
        for (int32_t j = 0; j < i; ++j)
            if (adapters[j] == a) {
                lora::set_last_error("lora_adamw_step: adapter listed twice");
                return LORA_ERR_INVALID_ARG;
            }
        const int32_t r = pool->rank[a];
        if (r < 1 || r > LORA_MAX_RANK) { lora::set_last_error("rank outside [1,128]"); return LORA_ERR_RANK; }
        for (int p = 0; p < 2; ++p) {
            const int k = blocks.n++;
            blocks.is_b[k] = p;
            blocks.off[k] = p ? pool->b_off[a] : pool->a_off[a];
            blocks.count[k] = (int64_t)r * (p ? N : K);
            if (blocks.off[k] < 0) { lora::set_last_error("negative pool offset"); return LORA_ERR_ADAPTER; }
            maxc = blocks.count[k] > maxc ? blocks.count[k] : maxc;
        }
    }
    AdamArgs a{};
    a.w[0] = A; a.w[1] = B;
    a.master[0] = A_master; a.master[1] = B_master;
    a.g[0] = dA; a.g[1] = dB;
    a.m[0] = mA; a.m[1] = mB;
    a.v[0] = vA; a.v[1] = vB;
    a.b1 = hp->beta1; a.b2 = hp->beta2;
    a.one_minus_b1 = 1.f - hp->beta1; a.one_minus_b2 = 1.f - hp->beta2;
    const double bc1 = 1.0 - pow((double)hp->beta1, (double)hp->step);
    const double bc2 = 1.0 - pow((double)hp->beta2, (double)hp->step);
    a.decay = (float)(1.0 - (double)hp->lr * (double)hp->weight_decay);
    a.step_size = (float)((double)hp->lr / bc1);
    a.inv_sqrt_bc2 = (float)(1.0 / sqrt(bc2));
    a.eps = hp->eps;
    a.bf16 = (dt == LORA_BF16) ? 1 : 0;
    const int threads = 256;
    int64_t gx = (maxc / 4 + threads - 1) / threads;
    if (gx < 1) gx = 1;
    if (gx > 1024) gx = 1024;
    dim3 grid((unsigned)gx, (unsigned)blocks.n);
    adamw_kernel<<<grid, threads, 0, static_cast<cudaStream_t>(stream)>>>(blocks, a);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        lora::set_last_error((std::string("adamw launch: ") + cudaGetErrorString(e)).c_str());
        return LORA_ERR_CUDA;
    }
    return LORA_OK;
}
