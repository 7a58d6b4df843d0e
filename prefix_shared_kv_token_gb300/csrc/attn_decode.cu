// attn_decode: one query token per request over its whole context in the token-indexed
// pool, read through req_to_token, with grouped query heads, split-KV and a shared-prefix
// cascade.
//
// What is computed: for request r with context length L (its just-stored token included)
// and query head h of KV head g = h / G:
//     o[r, h] = sum_{j < L} softmax_j(sm_scale * q[r, h] . K[slot_j, g]) * V[slot_j, g],
//     slot_j = req_to_token[req_pool_indices[r], j].
// The cached prefix is reused rather than recomputed ("Efficiently Programming Large
// Language Models using SGLang" summary, §RadixAttention) and requests whose paths share a
// radix-tree node share its slots ("[SGLang] RadixAttention ...", "Radix Tree 구조도").
//
// GB300 design
//   * One CTA (4 warps) per work item from the host plan.  A *span* item reads a shared
//     node's keys once for up to 64/G member requests (each warp owns 16 query rows =
//     16/G requests x G heads, so the tensor-core M dimension is full); a *tail* item reads
//     one request's unshared keys, and the 4 warps split every key tile.
//   * K/V rows (256 B per head for d = 128) are gathered with 16-byte cp.async into a
//     3-stage shared-memory ring laid out in 128-byte swizzled half-rows (chunk ^ key % 8),
//     so fragment loads and ldmatrix.trans are bank-conflict free.  Slot indices for the
//     tile after next are prefetched into registers while the current tile computes.
//   * QK^T and PV use mma.sync m16n8k16 (bf16 in, fp32 accumulate); the d-order inside each
//     k-step is permuted identically for Q and K so every lane loads 8 contiguous bytes.
//   * Online softmax in the log2 domain; partial states (m, l, acc) of items that cover
//     part of a request go to workspace records and a merge kernel combines them with the
//     log-sum-exp identity.  Tail items combine their 4 warps through shared memory first.
//   * fp8 pools: raw e4m3 tiles land in the ring and are converted exactly to bf16 tiles in
//     shared memory; k_scale folds into the logit scale, v_scale into the output.

#include "../../include/pkv.h"
#include "common.cuh"
#include "launch.h"

namespace pkv {

struct DecodeParams {
    const uint8_t *k_pool;
    const uint8_t *v_pool;
    int64_t num_slots;
    int32_t hkv, hq;
    const int32_t *req_to_token;
    int64_t rt_stride;
    int32_t rt_rows;
    int32_t batch;
    const int32_t *req_pool_indices;
    const int32_t *seq_lens;
    const uint16_t *q;  // bf16 bits [batch][hq][D]
    uint16_t *o;
    float scale_log2;   // sm_scale * k_scale * log2(e)
    float v_scale;
    const DecodeItem *items;
    const int32_t *row_req;
    const int32_t *row_rec;
    float *rec_acc;     // [rec][hq][D]
    float *rec_ml;      // [rec][hq][2]
    int32_t *err;
};

constexpr int kBK = 64;       // keys per tile
constexpr int kStages = 3;
constexpr float kLog2e = 1.4426950408889634f;

// Shared-memory geometry.  Compute tiles hold bf16 rows of 64 keys at a padded stride so that
// the mma.sync fragment loads (8 bytes per lane, K) and ldmatrix.trans (16-byte rows, V) are
// bank-conflict free: K rows at 2D + 32 bytes, V rows at 2D + 16 bytes.  A bf16 pool is
// gathered straight into these tiles; an fp8 pool lands as raw rows of D codes and is
// converted into a separate pair of compute tiles.
template <int D, bool FP8>
struct DLayout {
    static constexpr int kRow = FP8 ? D : 2 * D;          // bytes of one pool row (slot, head)
    static constexpr int kKS = 2 * D + 32;                // compute-tile row strides
    static constexpr int kVS = 2 * D + 16;
    static constexpr int kKTile = kBK * kKS;
    static constexpr int kVTile = kBK * kVS;
    static constexpr int kKRow = FP8 ? D : kKS;           // stage row strides
    static constexpr int kVRow = FP8 ? D : kVS;
    static constexpr int kStageK = kBK * kKRow;           // V rows start here
    static constexpr int kStageBytes = kStageK + kBK * kVRow;
    static constexpr int kConvOff = kStages * kStageBytes;
    static constexpr int kConvBytes = FP8 ? kKTile + kVTile : 0;
    static constexpr int kBarOff = kConvOff + kConvBytes;
    static constexpr int kBytes = kBarOff + 8 * kStages;
};

// Gather of one 64-key tile: thread t < 64 copies key t's K row, thread 64 + t its V row,
// each with one cp.async.bulk (a whole 128- or 256-byte row) completing on the stage's
// mbarrier.  Every thread arrives once per phase (expecting its own bytes, or none when
// the key is past the item or its slot is invalid, in which case it zeroes the row).
template <int D, bool FP8>
struct BulkLoader {
    using L = DLayout<D, FP8>;

    static PKV_DEV int32_t slot(const int32_t *rt, int kpos0, int k1) {
        const int kp = kpos0 + (threadIdx.x & 63);
        return kp < k1 ? __ldg(rt + kp) : -1;
    }

    static PKV_DEV void issue(const DecodeParams &p, uint8_t *stage, uint64_t *bar, int g, int32_t slot) {
        const int t = threadIdx.x;
        const bool is_v = t >= 64;
        const int key = t & 63;
        uint8_t *dst = stage + (is_v ? L::kStageK + key * L::kVRow : key * L::kKRow);
        if (slot >= 0 && (int64_t)slot < p.num_slots) {
            const uint8_t *src = (is_v ? p.v_pool : p.k_pool) + ((int64_t)slot * p.hkv + g) * L::kRow;
            mbar_arrive_expect_tx(bar, L::kRow);
            bulk_copy_g2s(smem_u32(dst), src, L::kRow, bar);
        } else {
            if (slot >= 0) set_error(p.err, DERR_SLOT_RANGE);
#pragma unroll
            for (int i = 0; i < L::kRow / 16; ++i) reinterpret_cast<uint4 *>(dst)[i] = make_uint4(0u, 0u, 0u, 0u);
            fence_proxy_async_smem();  // a later bulk copy rewrites this row
            mbar_arrive(bar);
        }
    }
};

// fp8: convert a raw stage (rows of D codes) into the padded bf16 compute tiles.
template <int D>
PKV_DEV void convert_fp8_stage(const uint8_t *raw, uint8_t *conv) {
    using L = DLayout<D, true>;
    constexpr int kChunks = kBK * D / 16;  // 16 codes per chunk, per tensor
    for (int i = threadIdx.x; i < 2 * kChunks; i += blockDim.x) {
        const int tensor = i / kChunks, ci = i % kChunks;
        const int key = ci / (D / 16), c = ci % (D / 16);
        const uint4 x = *reinterpret_cast<const uint4 *>(raw + tensor * L::kStageK + key * D + c * 16);
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
        uint32_t y[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            y[2 * k] = e4m3x2_to_bf16x2((uint16_t)(w[k] & 0xFFFFu));
            y[2 * k + 1] = e4m3x2_to_bf16x2((uint16_t)(w[k] >> 16));
        }
        uint8_t *dst = conv + (tensor ? L::kKTile + key * L::kVS : key * L::kKS) + c * 32;
        reinterpret_cast<uint4 *>(dst)[0] = make_uint4(y[0], y[1], y[2], y[3]);
        reinterpret_cast<uint4 *>(dst)[1] = make_uint4(y[4], y[5], y[6], y[7]);
    }
}

// Per-warp online-softmax state over 16 query rows (this lane: rows r and r + 8).
template <int D>
struct WarpState {
    float acc[D / 8][4];
    float m[2], l[2];
    uint32_t qf[D / 16][4];
};

// One tile's contribution for this warp: n-tiles [nt0, nt0 + NT) of the key tile.
template <int D, int NT>
PKV_DEV void warp_tile(WarpState<D> &st, const uint8_t *kt, const uint8_t *vt, int nt0, int kpos_tile, int k1,
                       float scale_log2) {
    const int lane = threadIdx.x & 31;
    const int r = lane >> 2, c = lane & 3;
    float s[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int key = (nt0 + nt) * 8 + r;
            const uint2 b2 = *reinterpret_cast<const uint2 *>(kt + key * (2 * D + 32) + (ks * 16 + 4 * c) * 2);
            const uint32_t b[2] = {b2.x, b2.y};
            mma_bf16_16816(s[nt], st.qf[ks], b);
        }
    }
    // mask, scale, running max
    float mt[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int kp = kpos_tile + (nt0 + nt) * 8 + 2 * c + (e & 1);
            const float x = kp < k1 ? s[nt][e] * scale_log2 : -INFINITY;
            s[nt][e] = x;
            mt[e >> 1] = fmaxf(mt[e >> 1], x);
        }
    }
    float alpha[2], mu[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        mt[h] = fmaxf(mt[h], __shfl_xor_sync(0xffffffffu, mt[h], 1));
        mt[h] = fmaxf(mt[h], __shfl_xor_sync(0xffffffffu, mt[h], 2));
        const float mn = fmaxf(st.m[h], mt[h]);
        mu[h] = mn == -INFINITY ? 0.f : mn;
        alpha[h] = ex2(st.m[h] - mu[h]);
        st.m[h] = mn;
    }
    float ls[2] = {0.f, 0.f};
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            // round to the bf16 weight the P.V product uses, and sum exactly that
            const float pv = __bfloat162float(__float2bfloat16_rn(ex2(s[nt][e] - mu[e >> 1])));
            s[nt][e] = pv;
            ls[e >> 1] += pv;
        }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) st.l[h] = st.l[h] * alpha[h] + ls[h];
#pragma unroll
    for (int nd = 0; nd < D / 8; ++nd) {
        st.acc[nd][0] *= alpha[0];
        st.acc[nd][1] *= alpha[0];
        st.acc[nd][2] *= alpha[1];
        st.acc[nd][3] *= alpha[1];
    }
    // O += P V
    const int mat = lane >> 3, mi = lane & 7;
#pragma unroll
    for (int kk = 0; kk < NT / 2; ++kk) {
        uint32_t a[4];
        a[0] = pack_bf16x2(s[2 * kk][0], s[2 * kk][1]);
        a[1] = pack_bf16x2(s[2 * kk][2], s[2 * kk][3]);
        a[2] = pack_bf16x2(s[2 * kk + 1][0], s[2 * kk + 1][1]);
        a[3] = pack_bf16x2(s[2 * kk + 1][2], s[2 * kk + 1][3]);
        const int key = (nt0 + 2 * kk) * 8 + (mat & 1) * 8 + mi;
#pragma unroll
        for (int nd = 0; nd < D / 8; nd += 2) {
            const int dchunk = nd + (mat >> 1);
            uint32_t bv[4];
            ldmatrix_x4_trans(bv, smem_u32(vt) + key * (2 * D + 16) + dchunk * 16);
            mma_bf16_16816(st.acc[nd], a, bv);
            mma_bf16_16816(st.acc[nd + 1], a, bv + 2);
        }
    }
}

template <int D, int G, bool FP8>
__global__ void __launch_bounds__(128, 2) decode_kernel(const DecodeParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    using L = DLayout<D, FP8>;
    using LD = BulkLoader<D, FP8>;
    constexpr int RPW = 16 / G;  // requests per warp in a span item
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kBarOff);

    const DecodeItem it = p.items[blockIdx.x];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = lane >> 2, c = lane & 3;
    const int g = it.g;

    // ---- key source row and range
    const int row = __ldg(p.req_pool_indices + it.src);
    const int k0 = it.k0;
    const int k1 = it.k1 < 0 ? __ldg(p.seq_lens + it.src) : it.k1;
    if (row < 0 || row >= p.rt_rows || k0 < 0 || k1 > p.rt_stride || k1 <= k0) {
        if (threadIdx.x == 0) set_error(p.err, DERR_POSITION);
        return;
    }
    const int32_t *rt = p.req_to_token + (int64_t)row * p.rt_stride;
    const int ntiles = (k1 - k0 + kBK - 1) / kBK;

    // ---- query fragments (rows r and r + 8 of this warp)
    WarpState<D> st;
    int req_of[2] = {-1, -1}, head_of[2] = {0, 0};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int i = r + 8 * h;
        if (it.mode == 0) {
            const int ri = warp * RPW + i / G;
            if (ri < it.nreq) req_of[h] = __ldg(p.row_req + it.row_off + ri);
        } else if (i < G) {
            req_of[h] = __ldg(p.row_req + it.row_off);
        }
        head_of[h] = g * G + (i % G);
        st.m[h] = -INFINITY;
        st.l[h] = 0.f;
    }
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint2 v = make_uint2(0u, 0u);
            if (req_of[h] >= 0)
                v = __ldg(reinterpret_cast<const uint2 *>(p.q + ((int64_t)req_of[h] * p.hq + head_of[h]) * D + ks * 16 +
                                                          4 * c));
            st.qf[ks][h] = v.x;       // k-slots 2c, 2c+1
            st.qf[ks][2 + h] = v.y;   // k-slots 2c+8, 2c+9
        }
    }
#pragma unroll
    for (int nd = 0; nd < D / 8; ++nd) st.acc[nd][0] = st.acc[nd][1] = st.acc[nd][2] = st.acc[nd][3] = 0.f;

    // ---- pipeline: one mbarrier per stage, every thread arrives once per phase
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(&bars[s], blockDim.x);
        fence_mbar_init();
    }
    __syncthreads();
    uint8_t *conv = smem + L::kConvOff;
#pragma unroll
    for (int s = 0; s < kStages - 1; ++s)
        if (s < ntiles) LD::issue(p, smem + s * L::kStageBytes, &bars[s], g, LD::slot(rt, k0 + s * kBK, k1));
    int32_t slot_next = (kStages - 1 < ntiles) ? LD::slot(rt, k0 + (kStages - 1) * kBK, k1) : -1;

    int j = 0;
    bool aborted = false;
    for (; j < ntiles; ++j) {
        const bool ok = mbar_wait(&bars[j % kStages], (j / kStages) & 1);
        if (__syncthreads_or(!ok)) {  // every thread leaves together
            if (threadIdx.x == 0) set_error(p.err, DERR_TIMEOUT | 0x20);
            aborted = true;
            break;
        }
        const int jn = j + kStages - 1;  // refill the stage consumed at j - 1
        if (jn < ntiles) LD::issue(p, smem + (jn % kStages) * L::kStageBytes, &bars[jn % kStages], g, slot_next);
        if (jn + 1 < ntiles) slot_next = LD::slot(rt, k0 + (jn + 1) * kBK, k1);

        const uint8_t *stage = smem + (j % kStages) * L::kStageBytes;
        const uint8_t *kt = stage, *vt = stage + L::kStageK;
        if constexpr (FP8) {
            convert_fp8_stage<D>(stage, conv);
            __syncthreads();
            kt = conv;
            vt = conv + L::kKTile;
        }
        const int kpos_tile = k0 + j * kBK;
        if (it.mode == 0)
            warp_tile<D, 8>(st, kt, vt, 0, kpos_tile, k1, p.scale_log2);
        else
            warp_tile<D, 2>(st, kt, vt, 2 * warp, kpos_tile, k1, p.scale_log2);
        if constexpr (FP8) __syncthreads();  // conv tiles are rewritten next tile
    }
    if (aborted) {
        // let the copies still in flight land (bounded) before the CTA exits
        for (int jj = j; jj < ntiles && jj < j + kStages - 1; ++jj) mbar_wait(&bars[jj % kStages], (jj / kStages) & 1);
        return;
    }

    // ---- epilogue
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        st.l[h] += __shfl_xor_sync(0xffffffffu, st.l[h], 1);
        st.l[h] += __shfl_xor_sync(0xffffffffu, st.l[h], 2);
    }
    if (it.mode == 0) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            if (req_of[h] < 0) continue;
            const int ri = warp * RPW + (r + 8 * h) / G;
            const int rec = __ldg(p.row_rec + it.row_off + ri);
            const int64_t base = (int64_t)req_of[h] * p.hq + head_of[h];
            if (rec < 0) {
                const float inv = p.v_scale / st.l[h];
                uint32_t *dst = reinterpret_cast<uint32_t *>(p.o + base * D);
#pragma unroll
                for (int nd = 0; nd < D / 8; ++nd)
                    dst[(nd * 8 + 2 * c) / 2] = pack_bf16x2(st.acc[nd][2 * h] * inv, st.acc[nd][2 * h + 1] * inv);
            } else {
                const int64_t rb = (int64_t)rec * p.hq + head_of[h];
                float2 *dst = reinterpret_cast<float2 *>(p.rec_acc + rb * D);
#pragma unroll
                for (int nd = 0; nd < D / 8; ++nd)
                    dst[(nd * 8 + 2 * c) / 2] =
                        make_float2(st.acc[nd][2 * h] * p.v_scale, st.acc[nd][2 * h + 1] * p.v_scale);
                if (c == 0) *reinterpret_cast<float2 *>(p.rec_ml + rb * 2) = make_float2(st.m[h], st.l[h]);
            }
        }
        return;
    }
    // tail item: combine the 4 warps (rows 0..G-1 live in lanes with r < G, h = 0)
    __syncthreads();
    float *red_m = reinterpret_cast<float *>(smem);         // [4][8]
    float *red_l = red_m + 32;                              // [4][8]
    float *red_acc = red_l + 32;                            // [4][8][D]
    if (r < G) {
        if (c == 0) {
            red_m[warp * 8 + r] = st.m[0];
            red_l[warp * 8 + r] = st.l[0];
        }
#pragma unroll
        for (int nd = 0; nd < D / 8; ++nd) {
            red_acc[(warp * 8 + r) * D + nd * 8 + 2 * c] = st.acc[nd][0];
            red_acc[(warp * 8 + r) * D + nd * 8 + 2 * c + 1] = st.acc[nd][1];
        }
    }
    __syncthreads();
    const int req = __ldg(p.row_req + it.row_off);
    const int rec = __ldg(p.row_rec + it.row_off);
    for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
        const int i = idx / D, d = idx % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < 4; ++w) M = fmaxf(M, red_m[w * 8 + i]);
        const float Mu = M == -INFINITY ? 0.f : M;
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const float wt = ex2(red_m[w * 8 + i] - Mu);
            L += red_l[w * 8 + i] * wt;
            O += red_acc[(w * 8 + i) * D + d] * wt;
        }
        const int head = g * G + i;
        if (rec < 0) {
            const float v = L > 0.f ? O * p.v_scale / L : 0.f;
            p.o[((int64_t)req * p.hq + head) * D + d] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
        } else {
            const int64_t rb = (int64_t)rec * p.hq + head;
            p.rec_acc[rb * D + d] = O * p.v_scale;
            if (d == 0) *reinterpret_cast<float2 *>(p.rec_ml + rb * 2) = make_float2(M, L);
        }
    }
}

// Combine partial states: o = sum_k 2^(m_k - M) acc_k / sum_k 2^(m_k - M) l_k.
template <int D>
__global__ void __launch_bounds__(256) merge_kernel(const MergeItem *__restrict__ merges, const float *__restrict__ rec_acc,
                                                    const float *__restrict__ rec_ml, uint16_t *__restrict__ o, int hq) {
    const MergeItem mi = merges[blockIdx.x];
    for (int idx = threadIdx.x; idx < hq * D; idx += blockDim.x) {
        const int h = idx / D, d = idx % D;
        float M = -INFINITY;
        for (int k = 0; k < mi.nrec; ++k) {
            const int64_t rb = (int64_t)(mi.rec0 + k * mi.rec_stride) * hq + h;
            M = fmaxf(M, rec_ml[rb * 2]);
        }
        const float Mu = M == -INFINITY ? 0.f : M;
        float L = 0.f, O = 0.f;
        for (int k = 0; k < mi.nrec; ++k) {
            const int64_t rb = (int64_t)(mi.rec0 + k * mi.rec_stride) * hq + h;
            const float2 ml = *reinterpret_cast<const float2 *>(rec_ml + rb * 2);
            const float wt = ex2(ml.x - Mu);
            L += ml.y * wt;
            O += rec_acc[rb * D + d] * wt;
        }
        o[((int64_t)mi.out_row * hq + h) * D + d] = __bfloat16_as_ushort(__float2bfloat16_rn(L > 0.f ? O / L : 0.f));
    }
}

template <int D, int G, bool FP8>
static int launch_decode(const DecodeParams &p, int nitems, cudaStream_t s) {
    constexpr int smem = DLayout<D, FP8>::kBytes;
    static_assert(smem >= (64 + 4 * 8 * D) * 4, "tail reduction must fit in the ring");
    auto kern = decode_kernel<D, G, FP8>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return PKV_E_CUDA;
    kern<<<nitems, 128, smem, s>>>(p);
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_E_CUDA;
}

template <int D>
static int dispatch_g(int G, bool fp8, const DecodeParams &p, int n, cudaStream_t s) {
    switch (G * 2 + (fp8 ? 1 : 0)) {
        case 2: return launch_decode<D, 1, false>(p, n, s);
        case 3: return launch_decode<D, 1, true>(p, n, s);
        case 4: return launch_decode<D, 2, false>(p, n, s);
        case 5: return launch_decode<D, 2, true>(p, n, s);
        case 8: return launch_decode<D, 4, false>(p, n, s);
        case 9: return launch_decode<D, 4, true>(p, n, s);
        case 16: return launch_decode<D, 8, false>(p, n, s);
        case 17: return launch_decode<D, 8, true>(p, n, s);
        default: return PKV_E_UNSUPPORTED;
    }
}

int launch_merge(const pkv_plan_info *info, const void *plan_dev, const float *rec_acc, const float *rec_ml,
                 uint16_t *o, cudaStream_t s) {
    if (info->num_merge == 0) return PKV_OK;
    const MergeItem *m = reinterpret_cast<const MergeItem *>(static_cast<const uint8_t *>(plan_dev) + info->offsets[3]);
    if (info->head_dim == 128)
        merge_kernel<128><<<info->num_merge, 256, 0, s>>>(m, rec_acc, rec_ml, o, info->num_q_heads);
    else
        merge_kernel<64><<<info->num_merge, 256, 0, s>>>(m, rec_acc, rec_ml, o, info->num_q_heads);
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_E_CUDA;
}

int check_call(const pkv_pool *pool, const pkv_batch *batch, const void *q, void *o, const pkv_plan_info *info,
               const void *plan_dev, void *workspace, size_t ws_bytes, int op) {
    int rc = validate_pool(pool);
    if (rc) return rc;
    if (!batch || !q || !o || !info || !plan_dev || !workspace) return PKV_E_INVALID;
    if (!batch->req_to_token || !batch->req_pool_indices || !batch->seq_lens) return PKV_E_INVALID;
    if (info->op != op || info->batch != batch->batch) return PKV_E_PLAN;
    if (info->num_kv_heads != pool->num_kv_heads || info->head_dim != pool->head_dim) return PKV_E_PLAN;
    if (ws_bytes < info->workspace_bytes) return PKV_E_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(plan_dev) & 15) || (reinterpret_cast<uintptr_t>(workspace) & 255))
        return PKV_E_INVALID;
    if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(o)) & 15) return PKV_E_INVALID;
    return PKV_OK;
}

}  // namespace pkv

extern "C" int pkv_attn_decode(const pkv_pool *pool, const pkv_batch *batch, const void *q, void *o, float sm_scale,
                               const pkv_plan_info *info, const void *plan_dev, void *workspace, size_t ws_bytes,
                               void *stream) {
    using namespace pkv;
    int rc = check_call(pool, batch, q, o, info, plan_dev, workspace, ws_bytes, 1);
    if (rc) return rc;
    if (info->num_items == 0) return PKV_OK;
    const uint8_t *plan = static_cast<const uint8_t *>(plan_dev);
    DecodeParams p;
    p.k_pool = static_cast<const uint8_t *>(pool->k);
    p.v_pool = static_cast<const uint8_t *>(pool->v);
    p.num_slots = pool->num_slots;
    p.hkv = pool->num_kv_heads;
    p.hq = info->num_q_heads;
    p.req_to_token = batch->req_to_token;
    p.rt_stride = batch->stride;
    p.rt_rows = batch->num_rows;
    p.batch = batch->batch;
    p.req_pool_indices = batch->req_pool_indices;
    p.seq_lens = batch->seq_lens;
    p.q = static_cast<const uint16_t *>(q);
    p.o = static_cast<uint16_t *>(o);
    const bool fp8 = pool->dtype == PKV_FP8_E4M3;
    p.scale_log2 = sm_scale * (fp8 ? pool->k_scale : 1.f) * kLog2e;
    p.v_scale = fp8 ? pool->v_scale : 1.f;
    p.items = reinterpret_cast<const DecodeItem *>(plan + info->offsets[0]);
    p.row_req = reinterpret_cast<const int32_t *>(plan + info->offsets[1]);
    p.row_rec = reinterpret_cast<const int32_t *>(plan + info->offsets[2]);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    p.err = reinterpret_cast<int32_t *>(ws);
    p.rec_acc = reinterpret_cast<float *>(ws + kWorkspaceHeader);
    p.rec_ml = p.rec_acc + (size_t)info->num_records * info->num_q_heads * info->head_dim;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int G = info->num_q_heads / info->num_kv_heads;
    rc = info->head_dim == 128 ? dispatch_g<128>(G, fp8, p, info->num_items, s)
                               : dispatch_g<64>(G, fp8, p, info->num_items, s);
    if (rc) return rc;
    return launch_merge(info, plan_dev, p.rec_acc, p.rec_ml, p.o, s);
}
