// pkv_attn_decode_noalloc: attn_decode for callers that cannot allocate device memory.
//
// Some callers of this library have no way to hand it a workspace at call time: a serving
// loop that froze its device-memory budget after start-up, or a host program that embeds
// the library without a device allocator of its own.  This entry point runs exactly the
// same decode kernels as pkv_attn_decode, but its scratch (the device error word and the
// partial softmax records of split-KV / cascade items) lives in one fixed array below,
// reserved when the library is loaded.  The caller still supplies every input and output.
//
// Rules of use
//   * The array is shared by every call in the process: calls whose work overlaps on the
//     GPU (different streams, or different host threads without ordering) race on it.
//   * A plan whose workspace_bytes exceed PKV_NOALLOC_WORKSPACE_BYTES is rejected with
//     PKV_E_WORKSPACE; nothing is launched.
//   * The first call on a device looks up the array's device address on that device (with
//     the device current) and caches it; make that first call before any stream capture.
//   * Each call clears the error word on its stream before launching; the records need no
//     clearing because every record the merge reads is written by the same call.
//   * pkv_get_noalloc_device_error reads that error word (the array's address is private to
//     this file, so pkv_get_device_error cannot be pointed at it).
// No cudaMalloc, cudaFree or allocating library routine is called here.

#include <cuda_runtime.h>

#include <mutex>

#include "../../include/pkv.h"

namespace {

__device__ __align__(256) unsigned char g_noalloc_scratch[PKV_NOALLOC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
void *g_scratch_ptr[kMaxDevices] = {nullptr};
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device (set-up on first use).
int scratch_for_current_device(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PKV_E_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return PKV_E_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return PKV_OK;
}

}  // namespace

extern "C" int pkv_attn_decode_noalloc(const pkv_pool *pool, const pkv_batch *batch, const void *q, void *o,
                                       float sm_scale, const pkv_plan_info *info, const void *plan_dev,
                                       void *stream) {
    if (!info) return PKV_E_INVALID;
    if (info->workspace_bytes > (size_t)PKV_NOALLOC_WORKSPACE_BYTES) return PKV_E_WORKSPACE;
    void *ws = nullptr;
    int rc = scratch_for_current_device(&ws);
    if (rc) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(ws, 0, sizeof(int32_t), s) != cudaSuccess) return PKV_E_CUDA;  // error word
    return pkv_attn_decode(pool, batch, q, o, sm_scale, info, plan_dev, ws, PKV_NOALLOC_WORKSPACE_BYTES, stream);
}

extern "C" int pkv_get_noalloc_device_error(void *stream, int32_t *raw) {
    void *ws = nullptr;
    int rc = scratch_for_current_device(&ws);
    if (rc) return rc;
    return pkv_get_device_error(ws, stream, raw);
}
