// kv_store: scatter the K/V rows of newly computed tokens into their pool slots.
//
// The pool is indexed per token: a radix-tree node's value lists the KV-pool index of each
// of its tokens ("[SGLang] RadixAttention: Radix Tree 기반 프리픽스 캐싱의 핵심", "Radix Tree
// 구조도" and TreeNode.value), and tokens missing from the cache get their K/V computed and
// stored before the node is inserted ("SGLang: Treating LLM Interactions as Programs ...",
// architecture figure: compute missing KV tensors, insert node).
//
// Design: a pure bandwidth kernel.  One token row per (token, K|V) is Hkv*d elements,
// contiguous in both source and destination.  A warp moves one row at a time (its slot read
// once, lanes striding the row's 16-byte vectors with four loads in flight); the grid is a
// multiple of the SM count and grid-strides over all rows.  bf16 pools copy bits; fp8 pools divide by the per-tensor scale in IEEE
// fp32 and round to E4M3 with saturation (cvt.rn.satfinite).  Slots outside [0, num_slots)
// are skipped and reported in the error word instead of being written.

#include "../../include/pkv.h"
#include "common.cuh"
#include "launch.h"

namespace pkv {

// CTX: each row is also written, as the bf16 values the pool now holds (fp8: the stored code
// converted exactly, unscaled), to row ctx_row[token] of the caller's context arrays
// (ctx_rows rows; a row outside them records DERR_POSITION with the token and the row, and
// that copy is skipped).
template <bool FP8, bool CTX>
__global__ void __launch_bounds__(256) kv_store_kernel(const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
                                                       const int32_t *__restrict__ loc, int64_t n, int32_t vec_per_row,
                                                       int64_t slot_bytes, uint8_t *__restrict__ k_pool,
                                                       uint8_t *__restrict__ v_pool,
                                                       int64_t num_slots, float k_scale, float v_scale,
                                                       int32_t *__restrict__ err, uint4 *__restrict__ ctx_k,
                                                       uint4 *__restrict__ ctx_v, const int32_t *__restrict__ ctx_row,
                                                       int64_t ctx_rows) {
    // one warp per token row (K rows of tokens 0..n-1, then their V rows), grid-strided; the
    // row's slot is read once and the lanes stride its vec_per_row 16-byte source vectors,
    // four loads in flight before their stores
    pdl_wait();     // the rows and slots may come from the preceding kernel
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; row < 2 * n; row += nwarps) {
        const bool is_v = row >= n;
        const int64_t tok = is_v ? row - n : row;
        const int32_t slot = __ldg(loc + tok);
        if (slot < 0 || (int64_t)slot >= num_slots) {
            if (lane == 0) set_error(err, DERR_SLOT_RANGE);
            continue;
        }
        const uint4 *src = (is_v ? v_new : k_new) + tok * vec_per_row;
        uint8_t *pool = (is_v ? v_pool : k_pool) + (int64_t)slot * slot_bytes;
        const float s = is_v ? v_scale : k_scale;
        uint4 *cdst = nullptr;
        if constexpr (CTX) {
            const int32_t r = __ldg(ctx_row + tok);
            if (r < 0 || (int64_t)r >= ctx_rows) {
                if (lane == 0) set_error_where(err, DERR_POSITION, (int32_t)tok, r, 0);
            } else {
                cdst = (is_v ? ctx_v : ctx_k) + (int64_t)r * vec_per_row;
            }
        }
        for (int v0 = lane; v0 < vec_per_row; v0 += 4 * 32) {
            uint4 x[4];
#pragma unroll
            for (int k = 0; k < 4; ++k)
                if (v0 + 32 * k < vec_per_row) x[k] = __ldcs(src + v0 + 32 * k);  // streamed once
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int v = v0 + 32 * k;
                if (v >= vec_per_row) continue;
                if constexpr (!FP8) {
                    reinterpret_cast<uint4 *>(pool)[v] = x[k];
                    if (CTX && cdst) cdst[v] = x[k];
                } else {
                    const uint32_t w[4] = {x[k].x, x[k].y, x[k].z, x[k].w};
                    uint16_t c[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        c[i] = f32x2_to_e4m3x2(__fdiv_rn(bf16_lo(w[i]), s), __fdiv_rn(bf16_hi(w[i]), s));
                    uint2 y;
                    y.x = (uint32_t)c[0] | ((uint32_t)c[1] << 16);
                    y.y = (uint32_t)c[2] | ((uint32_t)c[3] << 16);
                    reinterpret_cast<uint2 *>(pool)[v] = y;
                    if (CTX && cdst)
                        cdst[v] = make_uint4(e4m3x2_to_bf16x2(c[0]), e4m3x2_to_bf16x2(c[1]), e4m3x2_to_bf16x2(c[2]),
                                             e4m3x2_to_bf16x2(c[3]));
                }
            }
        }
    }
}

}  // namespace pkv

namespace pkv {

int launch_store(const pkv_pool *pool, const void *k_new, const void *v_new, const int32_t *out_cache_loc, int64_t n,
                 void *workspace, void *ctx_k, void *ctx_v, const int32_t *ctx_row, int64_t ctx_rows, cudaStream_t s) {
    const int64_t row_bytes = (int64_t)pool->num_kv_heads * pool->head_dim * 2;  // bf16 source row
    const int32_t vec_per_row = (int32_t)(row_bytes / 16);
    const int threads = 256;                      // 8 warps, one token row each at a time
    int64_t blocks = (2 * n + 7) / 8;
    const int64_t cap = (int64_t)num_sms() * 8;  // 8 resident blocks of 256 per SM
    if (blocks > cap) blocks = cap;
    const bool fp8 = pool->dtype != PKV_BF16, ctx = ctx_k != nullptr;
    auto kern = fp8 ? (ctx ? kv_store_kernel<true, true> : kv_store_kernel<true, false>)
                    : (ctx ? kv_store_kernel<false, true> : kv_store_kernel<false, false>);
    const cudaError_t e = launch_pdl(kern, dim3((unsigned)blocks), dim3(threads), 0, s, true,
                                     reinterpret_cast<const uint4 *>(k_new), reinterpret_cast<const uint4 *>(v_new),
                                     out_cache_loc, n, vec_per_row, slot_bytes(pool), reinterpret_cast<uint8_t *>(pool->k),
                                     reinterpret_cast<uint8_t *>(pool->v), pool->num_slots, fp8 ? pool->k_scale : 1.f,
                                     fp8 ? pool->v_scale : 1.f, reinterpret_cast<int32_t *>(workspace),
                                     reinterpret_cast<uint4 *>(ctx_k), reinterpret_cast<uint4 *>(ctx_v), ctx_row, ctx_rows);
    return e == cudaSuccess ? PKV_OK : PKV_E_CUDA;
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
    return launch_store(pool, k_new, v_new, out_cache_loc, n, workspace, nullptr, nullptr, nullptr, 0,
                        reinterpret_cast<cudaStream_t>(stream));
}
