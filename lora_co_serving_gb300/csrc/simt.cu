// simt.cu -- CUDA-core kernels: row gathering, saved-xA transposition, and the float32 path.
//
// The float32 path (LORA_F32) evaluates the layer and its LoRA backward with one thread per output
// element and float32 accumulation.  It serves the small float32 layers; bf16 layers take the
// tcgen05 path in tc_kernel.cu.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.h"
#include "simt.h"

namespace lora {

namespace {

// LORA_DEBUG_CHECKS: idx inside [0, extent), else LORA_ERR_BOUNDS is recorded and the caller skips the access
__device__ __forceinline__ bool dbg_ok(const SimtDebug& d, int64_t idx, int64_t extent) {
    if (!d.on || (idx >= 0 && idx < extent)) return true;
    atomicCAS(d.status, 0, LORA_ERR_BOUNDS);
    return false;
}

__global__ void gather_rows_kernel(const uint4* __restrict__ x, int32_t k8, const int32_t* __restrict__ rows,
                                   uint4* __restrict__ out, int32_t n_rows, const SimtDebug dbg) {
    for (int32_t i = blockIdx.x; i < n_rows; i += gridDim.x) {
        const int32_t t = rows[i];
        if (t >= 0 && !dbg_ok(dbg, t, dbg.x_rows)) continue;
        uint4* dst = out + (size_t)i * k8;
        if (t >= 0) {
            const uint4* src = x + (size_t)t * k8;
            for (int32_t v = threadIdx.x; v < k8; v += blockDim.x) dst[v] = src[v];
        } else {
            const uint4 z = make_uint4(0, 0, 0, 0);
            for (int32_t v = threadIdx.x; v < k8; v += blockDim.x) dst[v] = z;
        }
    }
}

// The shrink of the gathered decode rows on CUDA cores (see BgmvGroup).  Block = one work unit: a run of up to
// kBgmvRows rows sharing a chunk, and 8 of its LoRA columns.  Thread i of the block's kBgmvThreads takes the 16-byte
// pieces i, i + kBgmvThreads, ... of K; per piece it loads the unit's 8 rows of A and the run's rows of x and
// accumulates the kBgmvRows x 8 products in fp32.  A warp's partial sums are combined by a halving shuffle tree
// (every sum is formed by the same tree over the lanes), the warps' in warp order through shared memory, so each
// result depends on its own row of x and row of A alone.  Thread t < kBgmvRows * 8 writes Z = bf16(s * xA) of run
// row t / 8, column t % 8.
#ifndef LORA_BGMV_THREADS
#define LORA_BGMV_THREADS 128
#endif
#ifndef LORA_BGMV_UNROLL
#define LORA_BGMV_UNROLL 2
#endif
constexpr int kBgmvUnroll = LORA_BGMV_UNROLL;    // K-loop unroll (2: the next pieces' loads issue before the
                                                  // sums; 1024 decode rows 23.6 -> 21.7 us, 4 no faster)
constexpr int kBgmvThreads = LORA_BGMV_THREADS;   // 128 threads and 4 rows per unit measured fastest (decode batches of
                                                  // 256 and 1024 tokens: 16 and 24 us against 18 and 26 with 8 rows)
__global__ void __launch_bounds__(kBgmvThreads) bgmv_z_kernel(const uint4* __restrict__ xsrc, int32_t k8,
                                                     const int32_t* __restrict__ grows, uint4* __restrict__ xg,
                                                     const uint4* __restrict__ A, const BgmvGroup* __restrict__ groups,
                                                     const Chunk* __restrict__ chunks,
                                                     const TileDesc* __restrict__ tiles, int32_t S,
                                                     uint8_t* __restrict__ zout, const SimtDebug dbg) {
    constexpr int kSums = kBgmvRows * 8;      // the unit's row x column sums
    static_assert(kSums == 32 || kSums == 64, "4 or 8 rows per unit");
    __shared__ float red[kBgmvThreads / 32][kSums];
    const BgmvGroup u = groups[blockIdx.x];
    const uint4 zero = make_uint4(0, 0, 0, 0);
    if (dbg.on) {      // the run's gathered rows and their token rows must lie in their buffers
        bool ok = dbg_ok(dbg, (int64_t)u.g_row0 + u.n_rows - 1, dbg.g_rows);
        for (int i = 0; ok && i < u.n_rows; ++i) ok = dbg_ok(dbg, max(grows[u.g_row0 + i], 0), dbg.x_rows);
        if (!ok) return;
    }
    if (u.chunk < 0) {
        // copy-only unit: rows of base-only decode tokens (and zeros for the empty rows of the last tile)
        for (int i = 0; i < u.n_rows; ++i) {
            const int32_t t = grows[u.g_row0 + i];
            uint4* dst = xg + (size_t)(u.g_row0 + i) * k8;
            for (int32_t v = threadIdx.x; v < k8; v += kBgmvThreads) dst[v] = (t >= 0) ? xsrc[(size_t)t * k8 + v] : zero;
        }
        return;
    }
    const Chunk ch = chunks[u.chunk];
    const int32_t r_all = S * ch.r;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const bool copy = (u.j0 == 0);      // this unit also writes the run's rows into the gathered buffer
    const uint4* xr[kBgmvRows];
#pragma unroll
    for (int i = 0; i < kBgmvRows; ++i) xr[i] = xsrc + (size_t)(i < u.n_rows ? grows[u.g_row0 + i] : 0) * k8;
    float acc[kSums];
#pragma unroll
    for (int i = 0; i < kSums; ++i) acc[i] = 0.f;
#pragma unroll kBgmvUnroll
    for (int32_t v = threadIdx.x; v < k8; v += kBgmvThreads) {
        uint4 a[8], x[kBgmvRows];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            a[j] = (u.j0 + j < r_all) ? A[(size_t)(ch.prow_a + u.j0 + j) * k8 + v] : zero;
#pragma unroll
        for (int i = 0; i < kBgmvRows; ++i) x[i] = (i < u.n_rows) ? xr[i][v] : zero;
        if (copy) {
#pragma unroll
            for (int i = 0; i < kBgmvRows; ++i)
                if (i < u.n_rows) xg[(size_t)(u.g_row0 + i) * k8 + v] = x[i];
        }
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            float af[8][2], xf[kBgmvRows][2];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float2 f = __bfloat1622float2(reinterpret_cast<const __nv_bfloat162*>(&a[j])[h]);
                af[j][0] = f.x;
                af[j][1] = f.y;
            }
#pragma unroll
            for (int i = 0; i < kBgmvRows; ++i) {
                const float2 f = __bfloat1622float2(reinterpret_cast<const __nv_bfloat162*>(&x[i])[h]);
                xf[i][0] = f.x;
                xf[i][1] = f.y;
            }
#pragma unroll
            for (int i = 0; i < kBgmvRows; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    acc[i * 8 + j] = fmaf(xf[i][0], af[j][0], acc[i * 8 + j]);
                    acc[i * 8 + j] = fmaf(xf[i][1], af[j][1], acc[i * 8 + j]);
                }
        }
    }
    // halving tree: at each stage a lane keeps one half of its sums and adds its partner's copy of that half;
    // afterwards lane l holds sums [l * kSums / 32, (l + 1) * kSums / 32)
#pragma unroll
    for (int st = 0; st < 5; ++st) {
        const int off = 16 >> st, half = (kSums / 2) >> st;
        const bool up = (lane & off) != 0;
#pragma unroll
        for (int k = 0; k < half; ++k) {
            const float send = up ? acc[k] : acc[k + half];
            const float keep = up ? acc[k + half] : acc[k];
            acc[k] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
    }
#pragma unroll
    for (int k = 0; k < kSums / 32; ++k) red[warp][lane * (kSums / 32) + k] = acc[k];
    __syncthreads();
    const int t = threadIdx.x;
    if (t >= kSums) return;
    float sum = red[0][t];
#pragma unroll
    for (int w = 1; w < kBgmvThreads / 32; ++w) sum += red[w][t];
    const int i = t / 8, j = u.j0 + t % 8;
    if (i >= u.n_rows || j >= r_all) return;
    const TileDesc td = tiles[u.tile];
    const int32_t reg = j / ch.r, jj = j - reg * ch.r;
    const int32_t zc = reg * td.zstride + ch.zcol + jj;
    const int row = u.row0 + i;
    if (!dbg_ok(dbg, td.z_blk0 + zc / 64, dbg.z_blocks)) return;
    uint8_t* blk = zout + (size_t)(td.z_blk0 + zc / 64) * kZBlockBytes + row * 128;
    const int chunk16 = ((zc % 64) / 8) ^ (row & 7);
    *reinterpret_cast<__nv_bfloat16*>(blk + chunk16 * 16 + (zc % 8) * 2) = __float2bfloat16_rn(ch.scale * sum);
}

// xat[j, tpos0 + t] = xa_saved[xoff + t*r + j] for t < len, 0 for len <= t < roundup(len, 128); with a flag
// table, only for the segments it marks as saved (the others are recomputed by the shrink).  A transpose in 32 x 32
// tiles through shared memory: block (t tile, j tile, segment), reads along j and writes along t are coalesced.
__global__ void __launch_bounds__(256) xat_from_saved_kernel(const __nv_bfloat16* __restrict__ xa_saved,
                                                             const TrainSeg* __restrict__ tsegs, int32_t n_tsegs,
                                                             __nv_bfloat16* __restrict__ xat, int32_t P,
                                                             const int32_t* __restrict__ seg_flags,
                                                             const SimtDebug dbg) {
    __shared__ __nv_bfloat16 tile[32][34];
    const TrainSeg s = tsegs[blockIdx.z];
    if (seg_flags != nullptr && seg_flags[s.order] == 0) return;
    const int32_t span = (s.len + 127) / 128 * 128;
    const int32_t t0 = blockIdx.x * 32, j0 = blockIdx.y * 32;
    if (t0 >= span || j0 >= s.r) return;
    const int tx = threadIdx.x % 32, ty = threadIdx.x / 32;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int32_t t = t0 + ty + 8 * k, j = j0 + tx;
        __nv_bfloat16 v = __float2bfloat16_rn(0.f);
        if (t < s.len && j < s.r && dbg_ok(dbg, (int64_t)s.xoff + (int64_t)t * s.r + j, dbg.xa_elems))
            v = xa_saved[(size_t)s.xoff + (size_t)t * s.r + j];
        tile[ty + 8 * k][tx] = v;
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int32_t j = j0 + ty + 8 * k, t = t0 + tx;
        if (j < s.r && t < span && dbg_ok(dbg, (int64_t)j * P + s.tpos0 + t, dbg.t_elems))
            xat[(size_t)j * P + s.tpos0 + t] = tile[tx][ty + 8 * k];
    }
}

// ------------------------------------------------------------------------------------- float32 path
__global__ void f32_shrink_kernel(const float* __restrict__ x, const float* __restrict__ A,
                                  const AdapterRec* __restrict__ ad, const int32_t* __restrict__ tok_ad,
                                  const F32Seg* __restrict__ segs, int32_t n_segs, int32_t K,
                                  float* __restrict__ xa, int32_t train_only) {
    // one thread per (token, j) over the listed segments
    int64_t total = 0;
    for (int32_t s = 0; s < n_segs; ++s) total += (int64_t)segs[s].len * LORA_MAX_RANK;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        int64_t rem = i / LORA_MAX_RANK;
        const int32_t j = (int32_t)(i % LORA_MAX_RANK);
        int32_t s = 0;
        while (rem >= segs[s].len) { rem -= segs[s].len; ++s; }
        if (train_only && !segs[s].is_train) continue;
        const int32_t t = segs[s].start + (int32_t)rem;
        const int32_t a = tok_ad[t];
        if (a < 0 || j >= ad[a].r) continue;
        const float* xr = x + (size_t)t * K;
        const float* Ar = A + ad[a].a_off + (size_t)j * K;
        float acc = 0.f;
        for (int32_t k = 0; k < K; ++k) acc = fmaf(xr[k], Ar[k], acc);
        xa[(size_t)t * LORA_MAX_RANK + j] = acc;
    }
}

__global__ void f32_forward_kernel(const float* __restrict__ x, const float* __restrict__ Wt,
                                   const float* __restrict__ B, const AdapterRec* __restrict__ ad,
                                   const int32_t* __restrict__ tok_ad, const float* __restrict__ xa, int32_t T,
                                   int32_t K, int32_t N, float* __restrict__ y) {
    const int64_t total = (int64_t)T * N;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int32_t t = (int32_t)(i / N), n = (int32_t)(i % N);
        const float* xr = x + (size_t)t * K;
        const float* wr = Wt + (size_t)n * K;
        float acc = 0.f;
        for (int32_t k = 0; k < K; ++k) acc = fmaf(xr[k], wr[k], acc);
        const int32_t a = tok_ad[t];
        if (a >= 0) {
            float lo = 0.f;
            const float* Bb = B + ad[a].b_off + n;
            for (int32_t j = 0; j < ad[a].r; ++j) lo = fmaf(xa[(size_t)t * LORA_MAX_RANK + j], Bb[(size_t)j * N], lo);
            acc = fmaf(ad[a].scale, lo, acc);
        }
        y[i] = acc;
    }
}

// copy xA of fine-tuning rows to / from the packed saved-activation layout
__global__ void f32_xa_pack_kernel(float* __restrict__ xa, float* __restrict__ packed, const F32Seg* __restrict__ segs,
                                   int32_t n_segs, const AdapterRec* __restrict__ ad, int32_t to_packed,
                                   const int32_t* __restrict__ seg_flags) {
    for (int32_t s = 0; s < n_segs; ++s) {
        if (!segs[s].is_train) continue;
        if (seg_flags != nullptr && seg_flags[segs[s].order] == 0) continue;
        const int32_t r = ad[segs[s].adapter].r;
        const int64_t n = (int64_t)segs[s].len * r;
        for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
            const int32_t t = segs[s].start + (int32_t)(i / r), j = (int32_t)(i % r);
            float* p = packed + segs[s].xoff + i;
            float* q = xa + (size_t)t * LORA_MAX_RANK + j;
            if (to_packed) *p = *q; else *q = *p;
        }
    }
}

__global__ void f32_dyb_kernel(const float* __restrict__ dY, const float* __restrict__ B,
                               const AdapterRec* __restrict__ ad, const F32Seg* __restrict__ segs, int32_t n_segs,
                               int32_t N, float* __restrict__ dyb) {
    for (int32_t s = 0; s < n_segs; ++s) {
        if (!segs[s].is_train) continue;
        const AdapterRec rec = ad[segs[s].adapter];
        const int64_t n = (int64_t)segs[s].len * rec.r;
        for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
            const int32_t t = segs[s].start + (int32_t)(i / rec.r), j = (int32_t)(i % rec.r);
            const float* d = dY + (size_t)t * N;
            const float* Bj = B + rec.b_off + (size_t)j * N;
            float acc = 0.f;
            for (int32_t c = 0; c < N; ++c) acc = fmaf(d[c], Bj[c], acc);
            dyb[(size_t)t * LORA_MAX_RANK + j] = acc;
        }
    }
}

__global__ void f32_dx_kernel(const float* __restrict__ dY, const float* __restrict__ Wt, const float* __restrict__ A,
                              const AdapterRec* __restrict__ ad, const F32Seg* __restrict__ segs, int32_t n_segs,
                              const float* __restrict__ dyb, int32_t K, int32_t N, float* __restrict__ dX) {
    for (int32_t s = 0; s < n_segs; ++s) {
        if (!segs[s].is_train) continue;
        const AdapterRec rec = ad[segs[s].adapter];
        const int64_t n = (int64_t)segs[s].len * K;
        for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
            const int32_t t = segs[s].start + (int32_t)(i / K), k = (int32_t)(i % K);
            const float* d = dY + (size_t)t * N;
            float acc = 0.f;
            for (int32_t c = 0; c < N; ++c) acc = fmaf(d[c], Wt[(size_t)c * K + k], acc);
            float lo = 0.f;
            for (int32_t j = 0; j < rec.r; ++j)
                lo = fmaf(dyb[(size_t)t * LORA_MAX_RANK + j], A[rec.a_off + (size_t)j * K + k], lo);
            dX[(size_t)t * K + k] = fmaf(rec.scale, lo, acc);
        }
    }
}

// dB[j, n] (or dA[j, k]) of one adapter: sum over its fine-tuning segments in increasing start order
__global__ void f32_grad_kernel(const float* __restrict__ act, const float* __restrict__ other, int32_t ld_other,
                                const F32Seg* __restrict__ segs, int32_t n_segs, int32_t adapter, int32_t r,
                                float scale, int32_t width, float* __restrict__ out, int32_t accumulate) {
    // out[j*width + c] = s * sum_t act[t, j] * other[t, c]
    const int64_t total = (int64_t)r * width;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int32_t j = (int32_t)(i / width), c = (int32_t)(i % width);
        float acc = 0.f;
        for (int32_t s = 0; s < n_segs; ++s) {
            if (!segs[s].is_train || segs[s].adapter != adapter) continue;
            for (int32_t t = segs[s].start; t < segs[s].start + segs[s].len; ++t)
                acc = fmaf(act[(size_t)t * LORA_MAX_RANK + j], other[(size_t)t * ld_other + c], acc);
        }
        out[i] = accumulate ? out[i] + scale * acc : scale * acc;
    }
}

inline int grid_for(int64_t n) {
    int64_t g = (n + 255) / 256;
    return (int)(g < 1 ? 1 : (g > 4096 ? 4096 : g));
}

}  // namespace

cudaError_t gather_rows(const void* x, int32_t K, const int32_t* rows, void* out, int32_t n_rows, const SimtDebug& dbg,
                        cudaStream_t s) {
    if (n_rows <= 0) return cudaSuccess;
    gather_rows_kernel<<<n_rows < 65535 ? n_rows : 65535, 256, 0, s>>>(
        static_cast<const uint4*>(x), K / 8, rows, static_cast<uint4*>(out), n_rows, dbg);
    return cudaGetLastError();
}

cudaError_t bgmv_shrink(const void* x, const int32_t* grows, void* xg, int32_t K, const void* A,
                        const BgmvGroup* groups, int32_t n_groups, const Chunk* chunks, const TileDesc* tiles, int32_t S,
                        void* zout, const SimtDebug& dbg, cudaStream_t s) {
    if (n_groups <= 0) return cudaSuccess;
    bgmv_z_kernel<<<n_groups, kBgmvThreads, 0, s>>>(static_cast<const uint4*>(x), K / 8, grows, static_cast<uint4*>(xg),
                                                    static_cast<const uint4*>(A), groups, chunks, tiles, S,
                                                    static_cast<uint8_t*>(zout), dbg);
    return cudaGetLastError();
}

cudaError_t xat_from_saved(const void* xa_saved, const TrainSeg* tsegs, int32_t n_tsegs, int32_t max_len,
                           int32_t max_r, void* xat, int32_t P, const int32_t* seg_flags, const SimtDebug& dbg,
                           cudaStream_t s) {
    if (n_tsegs <= 0) return cudaSuccess;
    dim3 grid((max_len + 127) / 128 * 4, (max_r + 31) / 32, n_tsegs);
    xat_from_saved_kernel<<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(xa_saved), tsegs, n_tsegs,
                                               static_cast<__nv_bfloat16*>(xat), P, seg_flags, dbg);
    return cudaGetLastError();
}

cudaError_t f32_forward(const F32Args& a, cudaStream_t s) {
    f32_shrink_kernel<<<grid_for((int64_t)a.T * LORA_MAX_RANK), 256, 0, s>>>(a.x, a.A, a.ad, a.tok_ad, a.segs,
                                                                               a.n_segs, a.K, a.xa, 0);
    f32_forward_kernel<<<grid_for((int64_t)a.T * a.N), 256, 0, s>>>(a.x, a.Wt, a.B, a.ad, a.tok_ad, a.xa, a.T, a.K,
                                                                     a.N, a.y);
    if (a.xa_save)
        f32_xa_pack_kernel<<<grid_for(a.xa_elems), 256, 0, s>>>(a.xa, a.xa_save, a.segs, a.n_segs, a.ad, 1, nullptr);
    return cudaGetLastError();
}

cudaError_t f32_backward(const F32Args& a, cudaStream_t s) {
    // xA of the fine-tuning rows: recomputed, then (all, or the segments the flag table marks) taken from the
    // saved copy instead
    if (!a.xa_saved || a.seg_flags)
        f32_shrink_kernel<<<grid_for((int64_t)a.T * LORA_MAX_RANK), 256, 0, s>>>(a.x, a.A, a.ad, a.tok_ad, a.segs,
                                                                                   a.n_segs, a.K, a.xa, 1);
    if (a.xa_saved)
        f32_xa_pack_kernel<<<grid_for(a.xa_elems), 256, 0, s>>>(a.xa, const_cast<float*>(a.xa_saved), a.segs, a.n_segs,
                                                                a.ad, 0, a.seg_flags);
    f32_dyb_kernel<<<grid_for((int64_t)a.train_tokens * LORA_MAX_RANK), 256, 0, s>>>(a.dY, a.B, a.ad, a.segs,
                                                                                       a.n_segs, a.N, a.dyb);
    if (a.dX)
        f32_dx_kernel<<<grid_for((int64_t)a.train_tokens * a.K), 256, 0, s>>>(a.dY, a.Wt, a.A, a.ad, a.segs, a.n_segs,
                                                                              a.dyb, a.K, a.N, a.dX);
    for (int32_t g = 0; g < a.n_groups; ++g) {
        const int32_t ad = a.group_adapter[g], r = a.group_r[g];
        if (a.dB)
            f32_grad_kernel<<<grid_for((int64_t)r * a.N), 256, 0, s>>>(a.xa, a.dY, a.N, a.segs, a.n_segs, ad, r,
                                                                       a.group_scale[g], a.N,
                                                                       a.dB + a.group_b_off[g], a.accumulate);
        if (a.dA)
            f32_grad_kernel<<<grid_for((int64_t)r * a.K), 256, 0, s>>>(a.dyb, a.x, a.K, a.segs, a.n_segs, ad, r,
                                                                       a.group_scale[g], a.K,
                                                                       a.dA + a.group_a_off[g], a.accumulate);
    }
    return cudaGetLastError();
}

}  // namespace lora
