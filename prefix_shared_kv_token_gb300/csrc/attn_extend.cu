// attn_extend: attention for the uncached suffix of each request -- its new query tokens
// against the matched prefix plus the causal part of the suffix -- read through req_to_token.
//
// What is computed: request r extends e new tokens after a p-token matched prefix; query
// token i (position t = p + i) and head h of KV head g = h / G:
//     o[r, i, h] = sum_{j <= t} softmax_j(sm_scale * q . K[slot_j, g]) * V[slot_j, g].
// Only the remainder is prefilled, the prefix K/V are reused ("Efficiently Programming Large
// Language Models using SGLang" summary, §RadixAttention; "SGLang: Treating LLM Interactions
// as Programs ...", §Why this matters in production).
//
// GB300 design (one CTA = one work item: 128 query rows x one KV head x keys [k0, k1))
//   * 128 rows = 128/G query tokens x the G heads that share KV head g, so every K/V row
//     gathered from the pool feeds G query heads.  Q comes in with two 3-D TMA tile loads
//     (box 64 x G x 128/G, 128-byte swizzle).
//   * K and V tiles of 128 keys are gathered straight from the token-indexed pool by three
//     loader warps with 16-byte cp.async (LSU path; lanes of a warp cover whole 256-byte
//     rows), landing in the 128-byte-swizzled K-major layout tcgen05 reads; each loader
//     waits for its own copies and issues fence.proxy.async before arriving on the tile's
//     mbarrier.  Keys past the end of the item are zero-filled.  (TMA tile::gather4 of
//     128-byte rows was measured first: it delivered ~8 B/clk/SM, far below what the tensor
//     core consumes, so the gather runs on the LSU.)
//   * warp 0 issues tcgen05.mma (one thread): S = Q K^T into tensor memory (two S buffers),
//     then O += P V with P taken from tensor memory (the A operand) and V from shared memory
//     as an MN-major operand.  tcgen05.commit signals mbarriers.
//   * warps 4-7 (128 threads, one TMEM lane = one query row each) run the online softmax:
//     tcgen05.ld S, causal mask, exp2, write P (bf16) back over S with tcgen05.st.  O is
//     rescaled in tensor memory only when the running max grows by more than 2^8 (the
//     stale max keeps every p <= 256, exact in fp32 and bf16), so rescales are rare.
//   * fp8 pools: the loaders read e4m3 rows into registers, convert them exactly to bf16
//     and store them into the same swizzled operand layout (generic-proxy writes, then
//     fence.proxy.async before the MMA reads them).
//   * Every wait is bounded (2 s); on expiry the kernel records PKV_DERR_TIMEOUT, lets the
//     other roles time out too, drains in-flight work and frees tensor memory.

#include <algorithm>

#include "../../include/pkv.h"
#include "common.cuh"
#include "launch.h"

namespace pkv {

constexpr int kBM = 128;  // query rows per tile
constexpr int kBN = 128;  // keys per tile
constexpr float kLog2eX = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

struct ExtendParams {
    const uint8_t *k_pool;
    const uint8_t *v_pool;
    const int32_t *req_to_token;
    int64_t rt_stride;
    int32_t rt_rows;
    const int32_t *req_pool_indices;
    int64_t num_slots;
    int32_t hkv, hq;
    uint16_t *o;
    float scale_log2;
    float v_scale;
    const ExtendItem *items;
    float *rec_acc;
    float *rec_ml;
    int32_t *err;
};

template <int D, bool FP8>
struct ExtendCfg {
    static constexpr int kStages = 3;
    static constexpr int kBlk = kBN * 128;              // one 64-column block of a K/V tile
    static constexpr int kTile = kBN * D * 2;           // bf16 K (or V) tile
    static constexpr int kQBytes = kBM * D * 2;
    static constexpr int kQOff = 0;
    static constexpr int kStageOff = kQBytes;
    static constexpr int kSlotOff = kStageOff + kStages * 2 * kTile;  // [2][kBN] int32
    static constexpr int kBarOff = kSlotOff + 2 * kBN * 4;
    static constexpr int kBarBytes = 256;
    static constexpr int kSmem = kBarOff + kBarBytes + 1024;  // + alignment slack
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kColS = 0;                // S buffers at columns 0 and 128
    static constexpr uint32_t kColO = 256;
};

struct Bars {
    uint64_t q;
    uint64_t kfull[3], vfull[3], kvempty[3];
    uint64_t sfull[2], pfull[2];
    uint64_t odone, ofinal, drain;
    uint32_t tmem_base;
    int32_t abort_flag;
};

PKV_DEV bool wait_or_abort(uint64_t *bar, uint32_t parity, Bars *b, int32_t *err, int where) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 0) {
            if (*reinterpret_cast<volatile int32_t *>(&b->abort_flag)) return false;
            if (global_timer_ns() - t0 > kWaitTimeoutNs) {
                set_error(err, DERR_TIMEOUT | where);
                *reinterpret_cast<volatile int32_t *>(&b->abort_flag) = 1;
                return false;
            }
        }
    }
}

template <int D, int G, bool FP8>
__global__ void __launch_bounds__(256, 1)
    extend_kernel(const ExtendParams p, const __grid_constant__ CUtensorMap qmap) {
    using C = ExtendCfg<D, FP8>;
    constexpr int ST = C::kStages;
    constexpr int NBLK = D / 64;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    Bars *bars = reinterpret_cast<Bars *>(smem + C::kBarOff);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // once any CTA of this launch gave up on a wait, the rest exit instead of waiting too
    __shared__ int32_t s_skip;
    if (threadIdx.x == 0) s_skip = (*reinterpret_cast<volatile int32_t *>(p.err) & DERR_TIMEOUT) != 0;
    __syncthreads();
    if (s_skip) return;
    const ExtendItem it = p.items[blockIdx.x];
    const int g = it.g;
    const int row = __ldg(p.req_pool_indices + it.src);
    const int k0 = it.k0, k1 = it.k1;
    if (row < 0 || row >= p.rt_rows || k0 < 0 || k1 > p.rt_stride || k1 <= k0) {
        if (threadIdx.x == 0) set_error(p.err, DERR_POSITION);
        return;
    }
    const int32_t *rt = p.req_to_token + (int64_t)row * p.rt_stride;
    const int ntiles = (k1 - k0 + kBN - 1) / kBN;

    // ---- setup: barriers (thread 0), tensor memory (warp 0)
    if (threadIdx.x == 0) {
        mbar_init(&bars->q, 1);
        for (int s = 0; s < ST; ++s) {
            mbar_init(&bars->kfull[s], 96);  // every loader thread arrives
            mbar_init(&bars->vfull[s], 96);
            mbar_init(&bars->kvempty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars->sfull[b], 1);
            mbar_init(&bars->pfull[b], 128);
        }
        mbar_init(&bars->odone, 1);
        mbar_init(&bars->ofinal, 1);
        mbar_init(&bars->drain, 1);
        bars->abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&bars->tmem_base, C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    if (warp == 0) {
        // ================= MMA issuer =================
        if (lane == 0) {
            constexpr uint32_t idesc_qk = idesc_bf16_f32(kBM, kBN, 0, 0);
            constexpr uint32_t idesc_pv = idesc_bf16_f32(kBM, D, 0, 1);
            const uint32_t q_s = sbase + C::kQOff;
            bool ok = wait_or_abort(&bars->q, 0, bars, p.err, 1);
            auto issue_pv = [&](int i) -> bool {
                const int b = i & 1, s = i % ST;
                if (!wait_or_abort(&bars->pfull[b], (i >> 1) & 1, bars, p.err, 2)) return false;
                if (!wait_or_abort(&bars->vfull[s], (i / ST) & 1, bars, p.err, 3)) return false;
                tc_fence_after();
                const uint32_t v_s = sbase + C::kStageOff + (s * 2 + 1) * C::kTile;
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk) {
                    const uint64_t vdesc = sdesc_sw128(v_s + kk * 16 * 128, C::kBlk, 1024);
                    mma_ts(tmem + C::kColO, tmem + C::kColS + b * kBN + kk * 8, vdesc, idesc_pv,
                           (i > 0 || kk > 0) ? 1u : 0u);
                }
                tc_commit(&bars->kvempty[s]);
                tc_commit(&bars->odone);
                return true;
            };
            for (int j = 0; ok && j < ntiles; ++j) {
                const int s = j % ST, b = j & 1;
                if (!wait_or_abort(&bars->kfull[s], (j / ST) & 1, bars, p.err, 4)) { ok = false; break; }
                tc_fence_after();
                const uint32_t k_s = sbase + C::kStageOff + (s * 2) * C::kTile;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t off = (ks >> 2) * C::kBlk + (ks & 3) * 32;
                    const uint64_t qdesc = sdesc_sw128(q_s + (ks >> 2) * (kBM * 128) + (ks & 3) * 32, 16, 1024);
                    const uint64_t kdesc = sdesc_sw128(k_s + off, 16, 1024);
                    mma_ss(tmem + C::kColS + b * kBN, qdesc, kdesc, idesc_qk, ks > 0 ? 1u : 0u);
                }
                tc_commit(&bars->sfull[b]);
                if (j >= 1 && !issue_pv(j - 1)) { ok = false; break; }
            }
            if (ok) ok = issue_pv(ntiles - 1);
            if (ok) tc_commit(&bars->ofinal);
            // drain: every MMA issued so far has completed before tensor memory is freed
            tc_commit(&bars->drain);
            wait_or_abort(&bars->drain, 0, bars, nullptr, 0);
        }
        __syncwarp();
    } else if (warp < 4) {
        // ================= loaders (warps 1-3, 96 threads) =================
        // Q arrives with one TMA tile load per 64-column block.  K/V: every 16-byte chunk of
        // the tile's key rows is gathered with cp.async (bf16 pool) or loaded, converted
        // e4m3 -> bf16 exactly and stored (fp8 pool), straight into the 128-byte-swizzled
        // K-major layout; lanes of a warp cover contiguous 256-byte rows.  The slot numbers
        // of the next tile are staged in shared memory while the current tile is issued.
        constexpr int NP = 96;
        const int pt = threadIdx.x - 32;  // 0..95
        int32_t *sl = reinterpret_cast<int32_t *>(smem + C::kSlotOff);  // [2][kBN]
        if (pt == 0) {
            prefetch_tmap(&qmap);
            mbar_arrive_expect_tx(&bars->q, kBM * D * 2);
#pragma unroll
            for (int b = 0; b < NBLK; ++b)
                tma_load_3d(sbase + C::kQOff + b * (kBM * 128), &qmap, b * 64, g * G, it.tok0, &bars->q);
        }
        auto load_slots = [&](int j, int buf) {
            for (int k = pt; k < kBN; k += NP) {
                const int kp = k0 + j * kBN + k;
                int32_t slot = -1;
                if (kp < k1) {
                    slot = __ldg(rt + kp);
                    if (slot < 0 || (int64_t)slot >= p.num_slots) {
                        set_error(p.err, DERR_SLOT_RANGE);
                        slot = -1;
                    }
                }
                sl[buf * kBN + k] = slot;  // -1: zero-filled row (past k1 or invalid)
            }
        };
        load_slots(0, 0);
        named_bar_sync(1, NP);
        bool ok = true;
        // bf16: tile j is signalled ST-1 iterations after it was issued, before the stage
        // wait of the current iteration (so the MMA never waits on a tile the loaders hold)
        const int niter = FP8 ? ntiles : ntiles + ST - 1;
        for (int j = 0; j < niter; ++j) {
            if constexpr (!FP8) {
                const int jj = j - (ST - 1);
                if (jj >= 0) {
                    cp_async_wait<2 * ST - 3>();
                    fence_proxy_async_smem();
                    mbar_arrive(&bars->kfull[jj % ST]);
                    cp_async_wait<2 * ST - 4>();
                    fence_proxy_async_smem();
                    mbar_arrive(&bars->vfull[jj % ST]);
                }
            }
            if (j < ntiles) {
                const int s = j % ST;
                if (j >= ST && !wait_or_abort(&bars->kvempty[s], ((j / ST) - 1) & 1, bars, p.err, 5)) {
                    ok = false;
                    break;
                }
                const int32_t *ts = sl + (j & 1) * kBN;
                uint8_t *kdst = smem + C::kStageOff + (s * 2) * C::kTile;
                if constexpr (!FP8) {
                    constexpr int CPR = D / 8;  // 16-byte chunks per row
#pragma unroll
                    for (int tensor = 0; tensor < 2; ++tensor) {
                        const uint8_t *pool = tensor ? p.v_pool : p.k_pool;
                        const uint32_t dst = smem_u32(kdst) + tensor * C::kTile;
                        for (int ci = pt; ci < kBN * CPR; ci += NP) {
                            const int key = ci / CPR, c = ci % CPR;
                            const int32_t slot = ts[key];
                            const uint32_t off = (c >> 3) * C::kBlk + key * 128 + (((c & 7) ^ (key & 7)) << 4);
                            const int64_t src = ((int64_t)(slot < 0 ? 0 : slot) * p.hkv + g) * (D * 2) + c * 16;
                            cp_async_16(dst + off, pool + src, slot < 0 ? 0u : 16u);
                        }
                        cp_async_commit();
                    }
                } else {
                    constexpr int CPR = D / 16;  // 16-code chunks per row
                    constexpr int PER = (kBN * CPR + NP - 1) / NP;
#pragma unroll
                    for (int tensor = 0; tensor < 2; ++tensor) {
                        const uint8_t *pool = tensor ? p.v_pool : p.k_pool;
                        uint8_t *dst = kdst + tensor * C::kTile;
                        uint4 x[PER];
#pragma unroll
                        for (int i = 0; i < PER; ++i) {  // all loads in flight first
                            const int ci = pt + i * NP;
                            x[i] = make_uint4(0u, 0u, 0u, 0u);
                            if (ci < kBN * CPR) {
                                const int32_t slot = ts[ci / CPR];
                                if (slot >= 0)
                                    x[i] = __ldg(reinterpret_cast<const uint4 *>(
                                        pool + ((int64_t)slot * p.hkv + g) * D + (ci % CPR) * 16));
                            }
                        }
#pragma unroll
                        for (int i = 0; i < PER; ++i) {
                            const int ci = pt + i * NP;
                            if (ci >= kBN * CPR) continue;
                            const int key = ci / CPR, c = ci % CPR;
                            const uint32_t w[4] = {x[i].x, x[i].y, x[i].z, x[i].w};
                            uint32_t y[8];
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                y[2 * k] = e4m3x2_to_bf16x2((uint16_t)(w[k] & 0xFFFFu));
                                y[2 * k + 1] = e4m3x2_to_bf16x2((uint16_t)(w[k] >> 16));
                            }
#pragma unroll
                            for (int h = 0; h < 2; ++h) {  // bf16 chunks 2c and 2c+1
                                const int cc = 2 * c + h;
                                const uint32_t off = (cc >> 3) * C::kBlk + key * 128 + (((cc & 7) ^ (key & 7)) << 4);
                                *reinterpret_cast<uint4 *>(dst + off) =
                                    make_uint4(y[4 * h], y[4 * h + 1], y[4 * h + 2], y[4 * h + 3]);
                            }
                        }
                        fence_proxy_async_smem();
                        mbar_arrive(tensor ? &bars->vfull[s] : &bars->kfull[s]);
                    }
                }
                if (j + 1 < ntiles) load_slots(j + 1, (j + 1) & 1);
            } else if constexpr (!FP8) {
                cp_async_commit();  // keep two groups per iteration for the wait counts
                cp_async_commit();
            }
            named_bar_sync(1, NP);
        }
        if (!ok) cp_async_wait<0>();  // abort: let this thread's copies land before exit
    } else {
        // ================= softmax + epilogue (warps 4-7, one query row per thread) ========
        const int r = threadIdx.x - 128;                   // row = TMEM lane
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const int t = r / G;                               // token within the tile
        const int lim = it.qpos0 + t;                      // last visible position
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < ntiles; ++j) {
            const int b = j & 1;
            if (!wait_or_abort(&bars->sfull[b], (j >> 1) & 1, bars, p.err, 8)) { ok = false; break; }
            tc_fence_after();
            uint32_t sv[kBN];
#pragma unroll
            for (int c4 = 0; c4 < kBN / 32; ++c4) tmem_ld32(tmem + lane_base + C::kColS + b * kBN + c4 * 32, sv + c4 * 32);
            tmem_ld_wait();
            const int kp0 = k0 + j * kBN;
            float mt = -INFINITY;
#pragma unroll
            for (int c = 0; c < kBN; ++c) {
                const int kp = kp0 + c;
                const float x = (kp <= lim && kp < k1) ? __uint_as_float(sv[c]) * p.scale_log2 : -INFINITY;
                sv[c] = __float_as_uint(x);
                mt = fmaxf(mt, x);
            }
            const float mn = fmaxf(m, mt);
            float alpha = 1.f;
            bool rescale = false;
            if (mn > m + kRescaleThreshold || m == -INFINITY) {
                alpha = (m == -INFINITY) ? 0.f : ex2(m - mn);
                rescale = (j > 0) && (m != -INFINITY);
                m = mn;
            }
            const float mu = (m == -INFINITY) ? 0.f : m;
            float ls = 0.f;
#pragma unroll
            for (int hbuf = 0; hbuf < 2; ++hbuf) {
                uint32_t pk[32];
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const float p0 = ex2(__uint_as_float(sv[hbuf * 64 + 2 * c]) - mu);
                    const float p1 = ex2(__uint_as_float(sv[hbuf * 64 + 2 * c + 1]) - mu);
                    ls += p0 + p1;
                    pk[c] = pack_bf16x2(p0, p1);
                }
                tmem_st32(tmem + lane_base + C::kColS + b * kBN + hbuf * 32, pk);
            }
            l = l * alpha + ls;
            if (rescale) {
                // O may only be touched once PV of the previous tile has finished
                if (!wait_or_abort(&bars->odone, (j - 1) & 1, bars, p.err, 9)) { ok = false; break; }
                tc_fence_after();
#pragma unroll 1
                for (int c4 = 0; c4 < D / 32; ++c4) {
                    uint32_t ov[32];
                    tmem_ld32(tmem + lane_base + C::kColO + c4 * 32, ov);
                    tmem_ld_wait();
#pragma unroll
                    for (int c = 0; c < 32; ++c) ov[c] = __float_as_uint(__uint_as_float(ov[c]) * alpha);
                    tmem_st32(tmem + lane_base + C::kColO + c4 * 32, ov);
                }
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&bars->pfull[b]);
        }
        if (ok && wait_or_abort(&bars->ofinal, 0, bars, p.err, 10)) {
            tc_fence_after();
            const bool valid = t < it.ntok;
            const int tok = it.tok0 + t;
            const int head = g * G + (r % G);
#pragma unroll 1
            for (int c4 = 0; c4 < D / 32; ++c4) {
                uint32_t ov[32];
                tmem_ld32(tmem + lane_base + C::kColO + c4 * 32, ov);
                tmem_ld_wait();
                if (!valid) continue;
                if (it.rec < 0) {
                    const float inv = l > 0.f ? p.v_scale / l : 0.f;
                    uint4 *dst = reinterpret_cast<uint4 *>(p.o + ((int64_t)tok * p.hq + head) * D + c4 * 32);
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        uint32_t w[4];
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            w[k] = pack_bf16x2(__uint_as_float(ov[v * 8 + 2 * k]) * inv,
                                               __uint_as_float(ov[v * 8 + 2 * k + 1]) * inv);
                        dst[v] = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                } else {
                    const int64_t rb = (int64_t)(it.rec + t) * p.hq + head;
                    float4 *dst = reinterpret_cast<float4 *>(p.rec_acc + rb * D + c4 * 32);
#pragma unroll
                    for (int v = 0; v < 8; ++v)
                        dst[v] = make_float4(__uint_as_float(ov[4 * v]) * p.v_scale,
                                             __uint_as_float(ov[4 * v + 1]) * p.v_scale,
                                             __uint_as_float(ov[4 * v + 2]) * p.v_scale,
                                             __uint_as_float(ov[4 * v + 3]) * p.v_scale);
                    if (c4 == 0) *reinterpret_cast<float2 *>(p.rec_ml + rb * 2) = make_float2(m, l);
                }
            }
        }
    }

    // ---- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

template <int D, int G, bool FP8>
static int launch_extend(const ExtendParams &p, const CUtensorMap &qm, int nitems, cudaStream_t s) {
    constexpr int smem = ExtendCfg<D, FP8>::kSmem;
    static_assert(smem <= 232448, "shared memory budget");
    auto kern = extend_kernel<D, G, FP8>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return PKV_E_CUDA;
    kern<<<nitems, 256, smem, s>>>(p, qm);
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_E_CUDA;
}

template <int D>
static int dispatch_extend(int G, bool fp8, const ExtendParams &p, const CUtensorMap &qm, int n, cudaStream_t s) {
    switch (G * 2 + (fp8 ? 1 : 0)) {
        case 2: return launch_extend<D, 1, false>(p, qm, n, s);
        case 3: return launch_extend<D, 1, true>(p, qm, n, s);
        case 4: return launch_extend<D, 2, false>(p, qm, n, s);
        case 5: return launch_extend<D, 2, true>(p, qm, n, s);
        case 8: return launch_extend<D, 4, false>(p, qm, n, s);
        case 9: return launch_extend<D, 4, true>(p, qm, n, s);
        case 16: return launch_extend<D, 8, false>(p, qm, n, s);
        case 17: return launch_extend<D, 8, true>(p, qm, n, s);
        default: return PKV_E_UNSUPPORTED;
    }
}

int check_call(const pkv_pool *pool, const pkv_batch *batch, const void *q, void *o, const pkv_plan_info *info,
               const void *plan_dev, void *workspace, size_t ws_bytes, int op);
int launch_merge(const pkv_plan_info *info, const void *plan_dev, const float *rec_acc, const float *rec_ml,
                 uint16_t *o, cudaStream_t s);

}  // namespace pkv

extern "C" int pkv_attn_extend(const pkv_pool *pool, const pkv_batch *batch, const void *q, void *o, float sm_scale,
                               const pkv_plan_info *info, const void *plan_dev, void *workspace, size_t ws_bytes,
                               void *stream) {
    using namespace pkv;
    int rc = check_call(pool, batch, q, o, info, plan_dev, workspace, ws_bytes, 2);
    if (rc) return rc;
    if (info->num_items == 0) return PKV_OK;
    const int D = info->head_dim, hq = info->num_q_heads, hkv = info->num_kv_heads, G = hq / hkv;
    const bool fp8 = pool->dtype == PKV_FP8_E4M3;

    // Q as a [T][Hq][D] tensor, box 64 x G x 128/G: one load fills 128 rows (token, head)
    CUtensorMap qm;
    {
        cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)hq, (cuuint64_t)std::max(info->total_q, 1)};
        cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)hq * D * 2};
        cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)(128 / G)};
        if (encode_tiled(&qm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(q), dims, strides, box,
                         CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
            return PKV_E_CUDA;
    }

    const uint8_t *plan = static_cast<const uint8_t *>(plan_dev);
    ExtendParams p;
    p.k_pool = static_cast<const uint8_t *>(pool->k);
    p.v_pool = static_cast<const uint8_t *>(pool->v);
    p.req_to_token = batch->req_to_token;
    p.rt_stride = batch->stride;
    p.rt_rows = batch->num_rows;
    p.req_pool_indices = batch->req_pool_indices;
    p.num_slots = pool->num_slots;
    p.hkv = hkv;
    p.hq = hq;
    p.o = static_cast<uint16_t *>(o);
    p.scale_log2 = sm_scale * (fp8 ? pool->k_scale : 1.f) * kLog2eX;
    p.v_scale = fp8 ? pool->v_scale : 1.f;
    p.items = reinterpret_cast<const ExtendItem *>(plan + info->offsets[0]);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    p.err = reinterpret_cast<int32_t *>(ws);
    p.rec_acc = reinterpret_cast<float *>(ws + kWorkspaceHeader);
    p.rec_ml = p.rec_acc + (size_t)info->num_records * hq * D;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    rc = D == 128 ? dispatch_extend<128>(G, fp8, p, qm, info->num_items, s)
                  : dispatch_extend<64>(G, fp8, p, qm, info->num_items, s);
    if (rc) return rc;
    return launch_merge(info, plan_dev, p.rec_acc, p.rec_ml, p.o, s);
}
