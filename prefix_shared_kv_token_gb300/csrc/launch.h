// Host-side helpers shared by the C-ABI entry points: argument validation, device
// properties, tensor-map encoding through the driver entry point.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/pkv.h"

namespace pkv {

int num_sms();  // SMs of the current device (cached per device)

// Launch with programmatic stream serialization (pdl = true): the kernel may be scheduled
// while the previous kernel in the stream still runs (once all that kernel's CTAs issued
// pdl_trigger or exited), so launch latency and set-up overlap the previous kernel's tail.
// The kernel must call pdl_wait before it reads anything earlier work wrote, and before it
// exits.  pdl = false is an ordinary stream launch (pdl_wait then returns at once).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              bool pdl, Args &&...args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// cudaEvent_t pair set by pkv_set_kernel_events (consumed by the next pkv_attn_extend)
extern void *g_kernel_events[2];

// Limit of a pipeline wait inside the attention kernels for the next launches, in ns
// (pkv_set_wait_limit_ns; 2 s by default).
uint64_t wait_limit_ns();

inline int validate_pool(const pkv_pool *p) {
    if (!p || !p->k || !p->v) return PKV_E_INVALID;
    if (p->num_slots <= 0 || p->num_kv_heads <= 0) return PKV_E_INVALID;
    if (p->head_dim != 64 && p->head_dim != 128) return PKV_E_UNSUPPORTED;
    if (p->dtype != PKV_BF16 && p->dtype != PKV_FP8_E4M3) return PKV_E_UNSUPPORTED;
    if (p->num_slots * (int64_t)p->num_kv_heads >= ((int64_t)1 << 31)) return PKV_E_UNSUPPORTED;
    // rows start 16-byte aligned (bulk copies and vector loads); the arrays 128-byte aligned
    // unless interleaved, where v sits one K row after k
    if (reinterpret_cast<uintptr_t>(p->k) & 127) return PKV_E_INVALID;
    if (reinterpret_cast<uintptr_t>(p->v) & 15) return PKV_E_INVALID;
    const int64_t row = (int64_t)p->num_kv_heads * p->head_dim;
    if (p->slot_stride != 0 && (p->slot_stride < row || ((p->slot_stride * (p->dtype == PKV_BF16 ? 2 : 1)) & 15)))
        return PKV_E_INVALID;
    if (p->dtype == PKV_FP8_E4M3 && !(p->k_scale > 0.f && p->v_scale > 0.f)) return PKV_E_INVALID;
    return PKV_OK;
}

// Bytes from one slot's row to the next in the pool's k and v arrays.
inline int64_t slot_bytes(const pkv_pool *p) {
    const int64_t stride = p->slot_stride != 0 ? p->slot_stride : (int64_t)p->num_kv_heads * p->head_dim;
    return stride * (p->dtype == PKV_BF16 ? 2 : 1);
}

// The interleaved layout [slot][K row | V row]: a slot's K and V rows are one contiguous run.
inline bool kv_interleaved(const pkv_pool *p) {
    const int64_t row_bytes = (int64_t)p->num_kv_heads * p->head_dim * (p->dtype == PKV_BF16 ? 2 : 1);
    return slot_bytes(p) == 2 * row_bytes &&
           reinterpret_cast<uintptr_t>(p->v) == reinterpret_cast<uintptr_t>(p->k) + (uintptr_t)row_bytes;
}

// log2 of the batch table's page size (0 for a token table, page_size 0 or 1); -1 when the
// page size is not a power of two in [1, 4096].
inline int page_shift_of(const pkv_batch *b) {
    const int32_t ps = b->page_size <= 1 ? 1 : b->page_size;
    if (ps > 4096 || (ps & (ps - 1))) return -1;
    int sh = 0;
    while ((1 << sh) < ps) ++sh;
    return sh;
}

// cuTensorMapEncodeTiled, resolved once through cudaGetDriverEntryPoint (no -lcuda needed).
CUresult encode_tiled(CUtensorMap *map, CUtensorMapDataType dtype, cuuint32_t rank, void *base,
                      const cuuint64_t *dims, const cuuint64_t *strides_bytes, const cuuint32_t *box,
                      CUtensorMapSwizzle swizzle);

// Tensor-core pass of a decode plan over its widely shared spans, in two launches' worth of
// steps: the gather of the spans' keys and their members' query rows, then the extend
// kernel writing partial records (after_decode: the decode kernel was launched in between,
// so the pass reads the gather's output without waiting for that kernel, and waits for it
// before it exits).  No-ops when the plan has no such spans.
int decode_span_gather(const pkv_pool *pool, const pkv_batch *batch, const void *q, const pkv_plan_info *info,
                       const uint8_t *plan, uint8_t *ws, cudaStream_t s);
int decode_span_attend(const pkv_pool *pool, const void *q, float sm_scale, const pkv_plan_info *info,
                       const uint8_t *plan, uint8_t *ws, float *rec_acc, float *rec_ml, cudaStream_t s,
                       bool after_decode);

}  // namespace pkv
