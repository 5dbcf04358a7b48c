// noalloc.cu -- lora_mixed_forward_static: the forward pass with library-owned scratch, for callers that
// cannot allocate device memory.
//
// Some callers of this layer cannot call cudaMalloc or any allocating routine while they run a batch: a
// serving engine whose memory pool owns every byte of the device (allocations outside it would break its
// accounting or fail once the pool has reserved the free memory), or a code path that must not allocate
// because it runs inside a timing-critical step or while another component holds the allocator.  For them
// the forward pass's scratch (segment plan, gathered decode rows, the per-tile LoRA operand Z, shrink partial
// sums, status word and split counters) lives in one fixed array in device memory, declared below.
//
// Costs and limits:
//   * every GPU that loads the library holds the array (LORA_STATIC_WORKSPACE_BYTES) until the process exits;
//   * a batch whose forward scratch would exceed it is rejected with LORA_ERR_LIMIT before anything is launched;
//   * all calls share the array, which keeps whatever the last call left in it; each call zeroes the parts
//     that must start at zero (status word, split counters, Z) itself, but two calls that overlap on the GPU
//     (different streams, or different host threads without ordering) race on it;
//   * the array's device address is looked up (cudaGetSymbolAddress, with the call's device current) on every
//     call that is not being captured into a CUDA graph, so a device reset or a new primary context is picked
//     up; a call made during a capture reuses the address looked up last on that device, so make one call on
//     the device before capturing;
//   * the status word of the array (a kernel that gave up a bounded wait) is read by lora_static_status.
#include <cuda_runtime.h>

#include <mutex>
#include <string>

#include "lora_mixed.h"
#include "plan.h"

namespace {

// The scratch.  In host code this name is only a stand-in for the device array: its device address comes
// from cudaGetSymbolAddress, per device.
static __device__ __align__(256) unsigned char g_static_ws[LORA_STATIC_WORKSPACE_BYTES];

std::mutex g_mu;
void* g_addr[64] = {nullptr};

// The array's device address on the current device (see the notes above), or LORA_ERR_CUDA.
int static_address(cudaStream_t stream, void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= 64) {
        lora::set_last_error(e != cudaSuccess ? cudaGetErrorString(e) : "device index beyond 63");
        return LORA_ERR_CUDA;
    }
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    e = cudaStreamIsCapturing(stream, &cs);
    if (e != cudaSuccess) {
        lora::set_last_error((std::string("cudaStreamIsCapturing: ") + cudaGetErrorString(e)).c_str());
        return LORA_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    if (cs != cudaStreamCaptureStatusActive || !g_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_ws);       // with device `dev` current
        if (e != cudaSuccess) {
            lora::set_last_error((std::string("cudaGetSymbolAddress: ") + cudaGetErrorString(e)).c_str());
            return LORA_ERR_CUDA;
        }
        g_addr[dev] = p;
    }
    *out = g_addr[dev];
    return LORA_OK;
}

}  // namespace

extern "C" int lora_mixed_forward_static(int32_t T, int32_t K, int32_t N, lora_dtype_t dt, const void* x,
                                         const void* Wt, const lora_pool_t* pool, const lora_segment_t* segs,
                                         int32_t n_segs, void* y, void* xa_save, uint32_t flags, void* stream) {
    size_t need = 0;
    int rc = lora::forward_scratch_bytes(T, K, N, dt, pool, segs, n_segs, &need);
    if (rc != LORA_OK) return rc;                           // lora_last_error() already describes the problem
    if (need > (size_t)LORA_STATIC_WORKSPACE_BYTES) {
        const std::string msg = "lora_mixed_forward_static: this batch needs " + std::to_string(need) +
                                " bytes of scratch, more than the fixed " +
                                std::to_string((size_t)LORA_STATIC_WORKSPACE_BYTES) +
                                " bytes; split the batch or use lora_mixed_forward with a caller workspace";
        lora::set_last_error(msg.c_str());
        return LORA_ERR_LIMIT;
    }
    void* ws = nullptr;
    rc = static_address(static_cast<cudaStream_t>(stream), &ws);
    if (rc != LORA_OK) return rc;
    lora::DirectUpload direct;                              // no pinned staging ring: nothing is allocated
    return lora_mixed_forward(T, K, N, dt, x, Wt, pool, segs, n_segs, y, xa_save, flags, ws,
                              (size_t)LORA_STATIC_WORKSPACE_BYTES, stream);
}

extern "C" int lora_static_status(void* stream) {
    void* ws = nullptr;
    const int rc = static_address(static_cast<cudaStream_t>(stream), &ws);
    if (rc != LORA_OK) return rc;
    return lora_workspace_status(ws, stream);
}
