// kv_store: scatter the K/V rows of newly computed tokens into their pool slots.
//
// The pool is indexed per token: a radix-tree node's value lists the KV-pool index of each
// of its tokens ("[SGLang] RadixAttention: Radix Tree 기반 프리픽스 캐싱의 핵심", "Radix Tree
// 구조도" and TreeNode.value), and tokens missing from the cache get their K/V computed and
// stored before the node is inserted ("SGLang: Treating LLM Interactions as Programs ...",
// architecture figure: compute missing KV tensors, insert node).
//
// Design: a pure bandwidth kernel.  One token row per (token, K|V) is Hkv*d elements,
// contiguous in both source and destination, so each thread moves 16-byte vectors and a warp
// covers 512 contiguous source bytes; the grid is a multiple of the SM count and grid-strides
// over all rows.  bf16 pools copy bits; fp8 pools divide by the per-tensor scale in IEEE
// fp32 and round to E4M3 with saturation (cvt.rn.satfinite).  Slots outside [0, num_slots)
// are skipped and reported in the error word instead of being written.

#include "../../include/pkv.h"
#include "common.cuh"
#include "launch.h"

namespace pkv {

template <bool FP8>
__global__ void __launch_bounds__(256) kv_store_kernel(const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
                                                       const int32_t *__restrict__ loc, int64_t n, int32_t vec_per_row,
                                                       uint8_t *__restrict__ k_pool, uint8_t *__restrict__ v_pool,
                                                       int64_t num_slots, float k_scale, float v_scale,
                                                       int32_t *__restrict__ err) {
    // vec_per_row: 16-byte source vectors in one token row (Hkv * d * 2 / 16)
    const int64_t per_tensor = n * (int64_t)vec_per_row;
    const int64_t total = 2 * per_tensor;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += stride) {
        const bool is_v = idx >= per_tensor;
        const int64_t j = is_v ? idx - per_tensor : idx;
        const int64_t tok = j / vec_per_row;
        const int32_t part = (int32_t)(j - tok * vec_per_row);
        const int32_t slot = __ldg(loc + tok);
        if (slot < 0 || (int64_t)slot >= num_slots) {
            set_error(err, DERR_SLOT_RANGE);
            continue;
        }
        const uint4 x = __ldcs((is_v ? v_new : k_new) + j);  // streamed once
        uint8_t *pool = is_v ? v_pool : k_pool;
        if constexpr (!FP8) {
            uint4 *dst = reinterpret_cast<uint4 *>(pool) + (int64_t)slot * vec_per_row + part;
            *dst = x;
        } else {
            const float s = is_v ? v_scale : k_scale;
            const uint32_t w[4] = {x.x, x.y, x.z, x.w};
            uint16_t c[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                c[i] = f32x2_to_e4m3x2(__fdiv_rn(bf16_lo(w[i]), s), __fdiv_rn(bf16_hi(w[i]), s));
            uint2 y;
            y.x = (uint32_t)c[0] | ((uint32_t)c[1] << 16);
            y.y = (uint32_t)c[2] | ((uint32_t)c[3] << 16);
            uint2 *dst = reinterpret_cast<uint2 *>(pool) + (int64_t)slot * vec_per_row + part;
            *dst = y;
        }
    }
}

}  // namespace pkv

extern "C" int pkv_kv_store(const pkv_pool *pool, const void *k_new, const void *v_new,
                            const int32_t *out_cache_loc, int64_t n, void *workspace, void *stream) {
    using namespace pkv;
    int rc = validate_pool(pool);
    if (rc) return rc;
    if (n < 0) return PKV_E_INVALID;
    if (n == 0) return PKV_OK;
    if (!k_new || !v_new || !out_cache_loc) return PKV_E_INVALID;
    if ((reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new)) & 15) return PKV_E_INVALID;
    const int64_t row_bytes = (int64_t)pool->num_kv_heads * pool->head_dim * 2;  // bf16 source row
    const int32_t vec_per_row = (int32_t)(row_bytes / 16);
    const int64_t total = 2 * n * vec_per_row;
    const int threads = 256;
    int64_t blocks = (total + threads - 1) / threads;
    const int64_t cap = (int64_t)num_sms() * 8;  // 8 resident blocks of 256 per SM
    if (blocks > cap) blocks = cap;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (pool->dtype == PKV_BF16)
        kv_store_kernel<false><<<(unsigned)blocks, threads, 0, s>>>(
            reinterpret_cast<const uint4 *>(k_new), reinterpret_cast<const uint4 *>(v_new), out_cache_loc, n,
            vec_per_row, reinterpret_cast<uint8_t *>(pool->k), reinterpret_cast<uint8_t *>(pool->v), pool->num_slots,
            1.f, 1.f, reinterpret_cast<int32_t *>(workspace));
    else
        kv_store_kernel<true><<<(unsigned)blocks, threads, 0, s>>>(
            reinterpret_cast<const uint4 *>(k_new), reinterpret_cast<const uint4 *>(v_new), out_cache_loc, n,
            vec_per_row, reinterpret_cast<uint8_t *>(pool->k), reinterpret_cast<uint8_t *>(pool->v), pool->num_slots,
            pool->k_scale, pool->v_scale, reinterpret_cast<int32_t *>(workspace));
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_E_CUDA;
}
