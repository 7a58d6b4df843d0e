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
// GB300 design: gather once, then dense tensor-core attention.
//   1. gather_kernel copies the K/V rows of every key *run* of the plan -- a shared span
//      (a radix-tree node on several requests' paths, read once for all of them) or one
//      request's own remaining positions -- from the token-indexed pool into contiguous
//      workspace laid out [key][Hkv][d] bf16 (fp8 pools are converted exactly here, once
//      per key).  Whole 2 KB slot rows move as 16-byte vectors; a bandwidth-bound kernel.
//   2. extend_kernel: one CTA = two 128-row query tiles (each 128/G tokens x the G heads of
//      KV head g) against one run's keys [0, nkeys), 128 keys per K/V tile.
//        warps 0/2 TMA producers: Q tiles (3-D tile loads of q) and K tiles (warp 0), V
//                 tiles (warp 2) of the gathered run, 128-byte swizzle, into a 2-stage ring;
//        warp 1   tcgen05.mma issuer (one thread): S_q = Q_q K^T into tensor memory, then
//                 O_q += P_q V with P_q read from tensor memory (the A operand) and V as an
//                 MN-major shared-memory operand.  Issue order S0_j S1_j | PV0_j S0_j+1
//                 PV1_j S1_j+1 | ... keeps the tensor core busy while the other tile's
//                 softmax runs;
//        warps 4-7 / 8-11  softmax of Q tile 0 / 1: one thread per row (TMEM lane), causal
//                 mask, exp2, P written over S with tcgen05.st; O_q is rescaled in tensor
//                 memory only when the running max grows by more than 2^8 (p <= 256 stays
//                 exact), and then without waiting: S_q of tile j completing implies PV_q of
//                 tile j-1 completed (tcgen05 ops complete in issue order).
//      An item with one query tile over several key tiles is split: warpgroup 0 takes the
//      even key tiles into S0/O0, warpgroup 1 the odd ones into S1/O1 (both against Q tile
//      0), each with its own running max and sum; the epilogue combines the two states, each
//      warpgroup writing half of the head dimension.
//      The softmax holds a row's 128 scores in registers (one tcgen05.ld pass), takes the
//      row max as a tree, folds scale and max into one FFMA per score and skips the mask on
//      full tiles; the kernel fits the 168-register budget of 384 threads without spilling.
//      Every wait is bounded (the launch's wait limit, 2 s by default); on expiry the CTA
//      records PKV_DERR_TIMEOUT, its roles stop, in-flight work drains and tensor memory is
//      freed.

#include <algorithm>

#include "../../include/pkv.h"
#include "common.cuh"
#include "launch.h"

namespace pkv {

constexpr int kBM = 128;  // query rows per tile
constexpr int kBN = 128;  // keys per K/V tile
constexpr int kXStages = 2;
constexpr float kLog2eX = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr int kBarSplit = 1;               // named barrier of the two softmax warpgroups

struct ExtendParams {
    uint16_t *o;
    int32_t hkv, hq;
    float scale_log2;
    float v_scale;
    const ExtendItem *items;
    int32_t num_items;
    const int32_t *cta_off;   // items of CTA b: [cta_off[b], cta_off[b + 1])
    float *rec_acc;
    float *rec_ml;
    const int32_t *rec_list;  // NULL: token t of an item writes record rec + t; else rec_list[rec + t]
    const PackInfo *packs;    // packed items' segments and row groups (NULL: none)
    int32_t *err;
    WaitPolicy wait;          // pipeline waits (pkv_set_wait_limit_ns)
    int32_t pdl_wait_start;   // 1: wait for the preceding kernel before reading anything (it
                              // wrote this launch's inputs); 0: the inputs were complete
                              // earlier, wait only before exiting
};

template <int D>
struct XCfg {
    static constexpr int kBlkQ = kBM * 128;   // one 64-column block of a Q tile
    static constexpr int kBlkK = kBN * 128;   // one 64-column block of a K/V tile
    static constexpr int kQTile = kBM * D * 2;
    static constexpr int kKTile = kBN * D * 2;
    static constexpr int kQOff = 0;
    static constexpr int kStageOff = 2 * kQTile;
    static constexpr int kBarOff = kStageOff + kXStages * 2 * kKTile;
    static constexpr int kSmem = kBarOff + 256 + 1024;  // + alignment slack
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kColS = 0;     // S_q at q * 128
    static constexpr uint32_t kColO = 256;   // O_q at 256 + q * D
};

struct XBars {
    uint64_t q, qempty;
    uint64_t kfull[kXStages], vfull[kXStages], kvempty[kXStages], kempty[kXStages];
    uint64_t sfull[2], pfull[2], ofinal[2];
    uint64_t drain;
    uint32_t tmem_base;
    int32_t abort_flag;
};

// The launch's first timeout records the wait site (low byte of the code).  (Recording where
// the role was as well -- its item and tile, or only the CTA and the parity waited for -- cost
// the kernel 3 to 3.5 %: the values stay live through every wait.)
PKV_DEV bool xwait(uint64_t *bar, uint32_t parity, XBars *b, int32_t *err, int where, const WaitPolicy &wp) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if (it == 1 || (it & wp.check_mask) == 0) {
            if (*reinterpret_cast<volatile int32_t *>(&b->abort_flag)) return false;
            if (global_timer_ns() - t0 > wp.limit_ns) {
                set_error(err, DERR_TIMEOUT | where);
                *reinterpret_cast<volatile int32_t *>(&b->abort_flag) = 1;
                return false;
            }
        }
    }
}

// ------------------------------------------------------------------------------------------
// gather: run keys -> contiguous bf16 [key][Hkv][D] workspace

struct GatherParams {
    const uint8_t *k_pool;
    const uint8_t *v_pool;
    int64_t slot_bytes;  // from one slot's row to the next
    int64_t num_slots;
    int32_t hkv;
    const int32_t *req_to_token;
    int64_t rt_stride;
    int32_t rt_rows;
    int32_t page_shift;  // 0: token table; else log2 of the page size (page table)
    const int32_t *req_pool_indices;
    const GatherUnit *units;
    int32_t nunits;
    uint16_t *k_out;
    uint16_t *v_out;
    // query rows copied by the CTAs after the units (decode's tensor-core spans; else none):
    // row i of q_out = row q_rows[i] of q_src, q_row_vecs 16-byte vectors each
    const uint4 *q_src;
    uint4 *q_out;
    const int32_t *q_rows;
    int32_t q_batch, q_row_vecs;
    int32_t *err;
    int32_t pdl_wait_start;  // 1: wait for the preceding kernel first; 0: it wrote nothing this
                             // gather reads, wait for it only before exiting
};

// One CTA per unit of <= 32 keys: thread t moves 16-byte pieces of the units' slot rows
// (Hkv * D elements, contiguous in the pool and in the output).
template <int D, bool FP8>
PKV_DEV void gather_body(const GatherParams &p);

template <int D, bool FP8>
__global__ void __launch_bounds__(256) gather_kernel(const GatherParams p) {
    if (p.pdl_wait_start) pdl_wait();  // the pool rows and tables may come from the preceding kernel
    pdl_trigger();
    gather_body<D, FP8>(p);
    if (!p.pdl_wait_start) pdl_wait();  // complete only after the preceding kernel
}

template <int D, bool FP8>
PKV_DEV void gather_body(const GatherParams &p) {
    if ((int)blockIdx.x >= p.nunits) {  // a query row
        const int i = blockIdx.x - p.nunits, r = __ldg(p.q_rows + i);
        if (r < 0 || r >= p.q_batch) {
            if (threadIdx.x == 0) set_error(p.err, DERR_POSITION);
            return;
        }
        for (int v = threadIdx.x; v < p.q_row_vecs; v += blockDim.x)
            p.q_out[(int64_t)i * p.q_row_vecs + v] = __ldg(p.q_src + (int64_t)r * p.q_row_vecs + v);
        return;
    }
    const GatherUnit u = p.units[blockIdx.x];
    const int row = __ldg(p.req_pool_indices + u.src);
    if (row < 0 || row >= p.rt_rows || u.pos0 < 0 || u.pos0 + u.len > (p.rt_stride << p.page_shift)) {
        if (threadIdx.x == 0) set_error(p.err, DERR_POSITION);
        return;
    }
    // the unit's slots, checked once
    __shared__ int32_t s_slot[32];
    if (threadIdx.x < u.len) {
        int32_t slot = table_slot(p.req_to_token + (int64_t)row * p.rt_stride, u.pos0 + threadIdx.x, p.page_shift,
                                  p.num_slots);
        if (slot < 0 || (int64_t)slot >= p.num_slots) {
            set_error(p.err, DERR_SLOT_RANGE);
            slot = -1;  // zero row
        }
        s_slot[threadIdx.x] = slot;
    }
    __syncthreads();
    const int elems = p.hkv * D;                 // per slot row
    const int vec_out = elems / 8;               // 16-byte bf16 vectors per output row
    const bool pow2 = (vec_out & (vec_out - 1)) == 0;
    const int vshift = 31 - __clz(vec_out);
    const int per_tensor = u.len * vec_out;
    constexpr int kInFlight = 4;                 // independent loads per thread before stores
    for (int base = threadIdx.x; base < 2 * per_tensor; base += kInFlight * blockDim.x) {
        uint4 y[kInFlight];
#pragma unroll
        for (int k = 0; k < kInFlight; ++k) {
            const int i = base + k * blockDim.x;
            y[k] = make_uint4(0u, 0u, 0u, 0u);
            if (i >= 2 * per_tensor) continue;
            const int tensor = i >= per_tensor;
            const int rem = i - tensor * per_tensor;
            const int key = pow2 ? rem >> vshift : rem / vec_out, v = rem - key * vec_out;
            const int32_t slot = s_slot[key];
            if (slot < 0) continue;
            const uint8_t *pool = tensor ? p.v_pool : p.k_pool;
            if constexpr (!FP8) {
                y[k] = __ldg(reinterpret_cast<const uint4 *>(pool + (int64_t)slot * p.slot_bytes) + v);
            } else {
                const uint2 x = __ldg(reinterpret_cast<const uint2 *>(pool + (int64_t)slot * p.slot_bytes) + v);
                y[k].x = e4m3x2_to_bf16x2((uint16_t)(x.x & 0xFFFFu));
                y[k].y = e4m3x2_to_bf16x2((uint16_t)(x.x >> 16));
                y[k].z = e4m3x2_to_bf16x2((uint16_t)(x.y & 0xFFFFu));
                y[k].w = e4m3x2_to_bf16x2((uint16_t)(x.y >> 16));
            }
        }
#pragma unroll
        for (int k = 0; k < kInFlight; ++k) {
            const int i = base + k * blockDim.x;
            if (i >= 2 * per_tensor) continue;
            const int tensor = i >= per_tensor;
            const int rem = i - tensor * per_tensor;
            const int key = pow2 ? rem >> vshift : rem / vec_out, v = rem - key * vec_out;
            uint16_t *out = tensor ? p.v_out : p.k_out;
            reinterpret_cast<uint4 *>(out + (int64_t)(u.key0 + key) * elems)[v] = y[k];
        }
    }
}

// p = 2^(s * scale - m) for the 128 scores of one row (masked scores are -inf and give 0),
// packed to bf16 pairs and stored over the row's first 64 S columns in tensor memory.  ls
// accumulates the bf16 weights, so the normalised weights the P.V product uses add up to one
// exactly.  The exponentials run relative to mref = max(m, tile max), so their arguments are
// <= 0 (the bf16x2 exponential's error stays at the bf16 rounding of the weight); when the
// tile max is above the row's lazily kept m, SCALE multiplies by f2 = 2^(mref - m) (<= 2^8,
// bf16).  (Moving part of the exponentials to an FMA-pipe polynomial was measured slower:
// the softmax is bound by instruction issue, not by the MUFU.)
// The precise variant (rows that see few keys, at the very start of a prompt; their items
// run in a separate instantiation of the kernel so the common path keeps its registers):
// fp32 weights p (times f) written as bf16 high parts over S columns [0, 64) and bf16 low
// parts p - high over columns [64, 128); the MMA issuer feeds both to P.V.  ls sums the fp32
// weights.
PKV_DEV void exp_pack_precise(const uint32_t *sv, uint32_t col, float sc, float neg_mref, float f, float *ls) {
#pragma unroll
    for (int part = 0; part < 2; ++part) {
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
            uint32_t pk[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                const float p0 = ex2(fmaf(__uint_as_float(sv[hb * 64 + 2 * c]), sc, neg_mref)) * f;
                const float p1 = ex2(fmaf(__uint_as_float(sv[hb * 64 + 2 * c + 1]), sc, neg_mref)) * f;
                const uint32_t h = pack_bf16x2(p0, p1);
                if (part == 0) {
                    pk[c] = h;
                    ls[0] += p0;
                    ls[1] += p1;
                } else {
                    pk[c] = pack_bf16x2(p0 - bf16_lo(h), p1 - bf16_hi(h));
                }
            }
            tmem_st32(col + part * 64 + hb * 32, pk);
        }
    }
}

template <bool SCALE>
PKV_DEV void exp_pack_regs(const uint32_t *sv, uint32_t col, float sc, float neg_mref, uint32_t f2, float *ls) {
    // packed fp32 pairs: one fma.f32x2 / add.f32x2 per two scores (issue slots are the limit)
    const uint64_t sc2 = f2_pack(sc, sc), mu2 = f2_pack(neg_mref, neg_mref);
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int hb = 0; hb < 2; ++hb) {
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
            const uint64_t x = f2_fma(f2_pack(__uint_as_float(sv[hb * 64 + 2 * c]),
                                              __uint_as_float(sv[hb * 64 + 2 * c + 1])), sc2, mu2);
            float x0, x1;
            f2_unpack(x, x0, x1);
            pk[c] = ex2_bf16x2(pack_bf16x2(x0, x1));  // two weights per MUFU op, already packed
            if constexpr (SCALE) pk[c] = mul_bf16x2(pk[c], f2);
            add_bf16x2_f32(pk[c], acc[(c & 1) * 2], acc[(c & 1) * 2 + 1]);
        }
        tmem_st32(col + hb * 32, pk);
    }
    ls[0] += acc[0] + acc[2];
    ls[1] += acc[1] + acc[3];
}

// ------------------------------------------------------------------------------------------
// dense extend over gathered runs

// Per-item fields every role reads.
struct XItem {
    int32_t g, tok0, ntok, qpos0, pos0, nseg, rec, ntiles, nq;
    bool split;  // one query tile over >= 2 key tiles: both softmax warpgroups take it
    const int32_t *key0, *nkeys;  // segments (the item's own, or its PackInfo's)
    const PackInfo *pk;           // packed item: segments' positions and groups, row groups
};
PKV_DEV XItem load_item(const ExtendItem *itp, int tq, const PackInfo *packs) {
    XItem x;
    x.g = itp->g;
    x.tok0 = itp->tok0;
    x.ntok = itp->ntok;
    x.qpos0 = itp->qpos0;
    x.pos0 = itp->pos0;
    x.pk = (itp->flags & kItemPacked) && packs ? packs + itp->rec : nullptr;
    x.rec = x.pk ? -1 : itp->rec;  // a packed item's rec names its PackInfo; it writes o
    x.nseg = min(max(itp->nseg, 0), x.pk ? kPackSegs : kMaxSegs);
    x.key0 = x.pk ? x.pk->key0 : itp->key0;
    x.nkeys = x.pk ? x.pk->nkeys : itp->nkeys;
    x.ntiles = 0;  // key tiles over all segments (each segment starts a new tile)
    for (int sg = 0; sg < x.nseg; ++sg) x.ntiles += (x.nkeys[sg] + kBN - 1) / kBN;
    x.nq = x.ntok > tq ? 2 : 1;  // query tiles in use
    // split: warpgroup 0 takes the even key tiles and warpgroup 1 the odd ones, each with its
    // own running max, sum and accumulator (S_q, O_q), combined in the epilogue
    x.split = x.nq == 1 && x.ntiles >= 2;
    return x;
}

// Epilogue of one row: 32 accumulator columns [32 c4, 32 c4 + 32) of query token t (global
// token tok, head `head`) -- normalised to bf16 in o, or kept as an fp32 partial record
// (acc, and (m, l) with the first columns).
template <int D>
PKV_DEV void write_out(const ExtendParams &p, const XItem &it, int t, int tok, int head, int c4, const uint32_t *ov,
                       float m, float l) {
    if (it.rec < 0) {
        const float inv = l > 0.f ? p.v_scale / l : 0.f;
        uint4 *dst = reinterpret_cast<uint4 *>(p.o + ((int64_t)tok * p.hq + head) * D + c4 * 32);
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
                w[e] = pack_bf16x2(__uint_as_float(ov[v * 8 + 2 * e]) * inv, __uint_as_float(ov[v * 8 + 2 * e + 1]) * inv);
            dst[v] = make_uint4(w[0], w[1], w[2], w[3]);
        }
    } else {
        const int64_t rb = (int64_t)(p.rec_list ? __ldg(p.rec_list + it.rec + t) : it.rec + t) * p.hq + head;
        float4 *dst = reinterpret_cast<float4 *>(p.rec_acc + rb * D + c4 * 32);
#pragma unroll
        for (int v = 0; v < 8; ++v)
            dst[v] = make_float4(__uint_as_float(ov[4 * v]) * p.v_scale, __uint_as_float(ov[4 * v + 1]) * p.v_scale,
                                 __uint_as_float(ov[4 * v + 2]) * p.v_scale, __uint_as_float(ov[4 * v + 3]) * p.v_scale);
        if (c4 == 0) *reinterpret_cast<float2 *>(p.rec_ml + rb * 2) = make_float2(m, l);
    }
}

// Persistent: one CTA per SM walks its own list of items (the plan deals them longest
// first onto the least loaded CTA).  Tensor memory and barriers live for the whole launch; every
// role keeps its own running phase counters across items.  The next item's Q load waits only
// for the last S MMAs of the current item (qempty), and its first S MMAs may run while the
// softmax warpgroups are still in the current item's epilogue (they read O, not S); the next
// item's first P.V, which overwrites O, needs that warpgroup's next P and so comes after its
// epilogue.
template <int D, int G, bool PRECISE>
__global__ void __launch_bounds__(384, 1)
    extend_kernel(const ExtendParams p, const __grid_constant__ CUtensorMap qmap,
                  const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                  const __grid_constant__ CUtensorMap qmapg) {
    using C = XCfg<D>;
    constexpr int ST = kXStages;
    constexpr int NBLK = D / 64;
    constexpr int TQ = kBM / G;  // tokens per Q tile
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    XBars *bars = reinterpret_cast<XBars *>(smem + C::kBarOff);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (p.pdl_wait_start) pdl_wait();
    pdl_trigger();
    // the plan is read only from here on: with pdl_wait_start it may come from the kernel before
    const int i0 = __ldg(p.cta_off + blockIdx.x), i1 = __ldg(p.cta_off + blockIdx.x + 1);
    // once any CTA of this launch gave up on a wait, the rest exit instead of waiting too
    __shared__ int32_t s_skip;
    __shared__ float2 s_ml[2][kBM];  // split items: each warpgroup's running (max, sum) per row
    if (threadIdx.x == 0) s_skip = (*reinterpret_cast<volatile int32_t *>(p.err) & DERR_TIMEOUT) != 0;
    __syncthreads();
    if (s_skip) {
        if (!p.pdl_wait_start) pdl_wait();
        return;
    }

    if (threadIdx.x == 0) {
        mbar_init(&bars->q, 1);
        mbar_init(&bars->qempty, 1);
        for (int s = 0; s < ST; ++s) {
            mbar_init(&bars->kfull[s], 1);
            mbar_init(&bars->vfull[s], 1);
            mbar_init(&bars->kvempty[s], 1);
            mbar_init(&bars->kempty[s], 1);
        }
        for (int q = 0; q < 2; ++q) {
            mbar_init(&bars->sfull[q], 1);
            mbar_init(&bars->pfull[q], 128);
            mbar_init(&bars->ofinal[q], 1);
        }
        mbar_init(&bars->drain, 1);
        bars->abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&bars->tmem_base, C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    if (warp == 0 || warp == 2) {
        if (lane == 0) {
            // ================= TMA producers =================
            // warp 0 loads Q and the K tiles, warp 2 the V tiles.  A stage is released by
            // kvempty after its last P.V; a split item's tile also releases its K half early
            // (kempty, after its S), so the next K tile loads while the P.V still holds V.
            const bool kside = warp == 0;
            const CUtensorMap *map = kside ? &kmap : &vmap;
            uint64_t *full = kside ? bars->kfull : bars->vfull;
            const uint32_t half = kside ? 0u : (uint32_t)C::kKTile;
            prefetch_tmap(map);
            if (kside) {
                prefetch_tmap(&qmap);
                prefetch_tmap(&qmapg);
            }
            int tp = 0, nql = 0;             // tiles and Q loads issued by this thread
            uint32_t split_mask = 0;         // bit s: stage s's previous tile came from a split item
            uint32_t kpar = 0;               // bit s: parity of the kempty commits due on stage s
            bool ok = true;
            for (int i = i0; ok && i < i1; ++i) {
                const ExtendItem *itp = p.items + i;
                const XItem it = load_item(itp, TQ, p.packs);
                if (kside) {
                    if (nql > 0 && !xwait(&bars->qempty, (nql - 1) & 1, bars, p.err, 6, p.wait)) break;
                    if (it.pk) {
                        // a packed tile: each row group's tokens by their own 32-row box
                        int ng = 0;
                        while (ng < 4 && it.pk->ntok[ng] > 0) ++ng;
                        mbar_arrive_expect_tx(&bars->q, ng * NBLK * 32 * 128);
                        for (int m = 0; m < ng; ++m)
#pragma unroll
                            for (int b = 0; b < NBLK; ++b)
                                tma_load_3d(sbase + C::kQOff + b * C::kBlkQ + m * 32 * 128, &qmapg, b * 64, it.g * G,
                                            it.pk->tok0[m], &bars->q);
                    } else {
                        mbar_arrive_expect_tx(&bars->q, it.nq * C::kQTile);
                        for (int q = 0; q < it.nq; ++q)
#pragma unroll
                            for (int b = 0; b < NBLK; ++b)
                                tma_load_3d(sbase + C::kQOff + q * C::kQTile + b * C::kBlkQ, &qmap, b * 64, it.g * G,
                                            it.tok0 + q * TQ, &bars->q);
                    }
                    ++nql;
                }
                int sg = 0, lt = 0;  // segment and tile within it
                for (int j = 0; j < it.ntiles; ++j, ++tp) {
                    const int s = tp % ST;
                    if (tp >= ST) {
                        const bool early = kside && ((split_mask >> s) & 1u);
                        uint64_t *bar = early ? &bars->kempty[s] : &bars->kvempty[s];
                        const uint32_t par = early ? ((kpar >> s) & 1u) ^ 1u : (uint32_t)((tp / ST) - 1) & 1u;
                        if (!xwait(bar, par, bars, p.err, kside ? 5 : 7, p.wait)) {
                            ok = false;
                            break;
                        }
                    }
                    split_mask = (split_mask & ~(1u << s)) | ((uint32_t)it.split << s);
                    kpar ^= (uint32_t)it.split << s;
                    const uint32_t dst = sbase + C::kStageOff + (s * 2) * C::kKTile + half;
                    const int key = it.key0[sg] + lt * kBN;
                    if (++lt * kBN >= it.nkeys[sg]) {
                        ++sg;
                        lt = 0;
                    }
                    mbar_arrive_expect_tx(&full[s], C::kKTile);
#pragma unroll
                    for (int b = 0; b < NBLK; ++b) tma_load_3d(dst + b * C::kBlkK, map, b * 64, it.g, key, &full[s]);
                }
            }
            // Let every copy this thread issued land before it leaves, whether or not a wait
            // gave up: another role may have stopped waiting (and the CTA may be unwinding)
            // while the last tiles were still in flight.  Each stage's last tile is one of the
            // last ST; earlier tiles were released by the MMAs, so they have landed; no stage
            // is re-armed after its last tile.  In a normal run these phases completed long
            // ago and each wait returns at once.
            if (kside && nql > 0) mbar_wait(&bars->q, (nql - 1) & 1);
            for (int t = tp > ST ? tp - ST : 0; t < tp; ++t) mbar_wait(&full[t % ST], (t / ST) & 1);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ================= MMA issuer =================
            constexpr uint32_t idesc_qk = idesc_bf16_f32(kBM, kBN, 0, 0);
            constexpr uint32_t idesc_pv = idesc_bf16_f32(kBM, D, 0, 1);
            int tm = 0, ip = 0;       // tiles and items before the current one
            uint32_t cpar = 0;        // bit q: parity of the next phase to consume on pfull[q]
            bool ok = true;
            for (int i = i0; ok && i < i1; ++i, ++ip) {
                const XItem it = load_item(p.items + i, TQ, p.packs);
                if (!xwait(&bars->q, ip & 1, bars, p.err, 1, p.wait)) break;
                if (!it.split) {
                    auto issue_s = [&](int q, int j) -> bool {
                        const int tg = tm + j, s = tg % ST;
                        if (q == 0 && !xwait(&bars->kfull[s], (tg / ST) & 1, bars, p.err, 4, p.wait)) return false;
                        tc_fence_after();
                        const uint32_t q_s = sbase + C::kQOff + q * C::kQTile;
                        const uint32_t k_s = sbase + C::kStageOff + (s * 2) * C::kKTile;
#pragma unroll
                        for (int ks = 0; ks < D / 16; ++ks) {
                            const uint64_t qd = sdesc_sw128(q_s + (ks >> 2) * C::kBlkQ + (ks & 3) * 32, 16, 1024);
                            const uint64_t kd = sdesc_sw128(k_s + (ks >> 2) * C::kBlkK + (ks & 3) * 32, 16, 1024);
                            mma_ss(tmem + C::kColS + q * kBN, qd, kd, idesc_qk, ks > 0 ? 1u : 0u);
                        }
                        tc_commit(&bars->sfull[q]);
                        if (j == it.ntiles - 1 && q == it.nq - 1) tc_commit(&bars->qempty);  // Q no longer read
                        return true;
                    };
                    auto issue_pv = [&](int q, int j) -> bool {
                        const int tg = tm + j, s = tg % ST;
                        if (!xwait(&bars->pfull[q], (cpar >> q) & 1u, bars, p.err, 2, p.wait)) return false;
                        cpar ^= 1u << q;
                        if (q == 0 && !xwait(&bars->vfull[s], (tg / ST) & 1, bars, p.err, 3, p.wait)) return false;
                        tc_fence_after();
                        const uint32_t v_s = sbase + C::kStageOff + (s * 2 + 1) * C::kKTile;
#pragma unroll
                        for (int kk = 0; kk < kBN / 16; ++kk) {
                            const uint64_t vd = sdesc_sw128(v_s + kk * 16 * 128, C::kBlkK, 1024);
                            mma_ts(tmem + C::kColO + q * D, tmem + C::kColS + q * kBN + kk * 8, vd, idesc_pv,
                                   (j > 0 || kk > 0) ? 1u : 0u);
                        }
                        if constexpr (PRECISE) {  // + the weights' bf16 low parts, columns [64, 128) of S
#pragma unroll
                            for (int kk = 0; kk < kBN / 16; ++kk) {
                                const uint64_t vd = sdesc_sw128(v_s + kk * 16 * 128, C::kBlkK, 1024);
                                mma_ts(tmem + C::kColO + q * D, tmem + C::kColS + q * kBN + 64 + kk * 8, vd, idesc_pv,
                                       1u);
                            }
                        }
                        if (q == it.nq - 1) tc_commit(&bars->kvempty[s]);
                        if (j == it.ntiles - 1) tc_commit(&bars->ofinal[q]);
                        return true;
                    };
                    ok = issue_s(0, 0) && (it.nq < 2 || issue_s(1, 0));
                    for (int j = 0; ok && j < it.ntiles; ++j) {
                        if (!issue_pv(0, j)) { ok = false; break; }
                        if (j + 1 < it.ntiles && !issue_s(0, j + 1)) { ok = false; break; }
                        if (it.nq > 1) {
                            if (!issue_pv(1, j)) { ok = false; break; }
                            if (j + 1 < it.ntiles && !issue_s(1, j + 1)) { ok = false; break; }
                        }
                    }
                } else {
                    // split item: key tile j goes to S_{j&1} / O_{j&1}, all with Q tile 0.  Order
                    // S(0) S(1) | PV(0) S(2) | PV(1) S(3) | ... -- the same ping-pong as above.
                    // Each tile has a stage of its own, so its K half is released (kempty) once
                    // its S is done and the next K tile loads while this one's P.V still waits.
                    auto split_s = [&](int j) -> bool {
                        const int q = j & 1, tg = tm + j, s = tg % ST;
                        if (!xwait(&bars->kfull[s], (tg / ST) & 1, bars, p.err, 4, p.wait)) return false;
                        tc_fence_after();
                        const uint32_t q_s = sbase + C::kQOff;
                        const uint32_t k_s = sbase + C::kStageOff + (s * 2) * C::kKTile;
#pragma unroll
                        for (int ks = 0; ks < D / 16; ++ks) {
                            const uint64_t qd = sdesc_sw128(q_s + (ks >> 2) * C::kBlkQ + (ks & 3) * 32, 16, 1024);
                            const uint64_t kd = sdesc_sw128(k_s + (ks >> 2) * C::kBlkK + (ks & 3) * 32, 16, 1024);
                            mma_ss(tmem + C::kColS + q * kBN, qd, kd, idesc_qk, ks > 0 ? 1u : 0u);
                        }
                        tc_commit(&bars->sfull[q]);
                        tc_commit(&bars->kempty[s]);
                        if (j == it.ntiles - 1) tc_commit(&bars->qempty);
                        return true;
                    };
                    auto split_pv = [&](int j) -> bool {
                        const int q = j & 1, tg = tm + j, s = tg % ST;
                        if (!xwait(&bars->pfull[q], (cpar >> q) & 1u, bars, p.err, 2, p.wait)) return false;
                        cpar ^= 1u << q;
                        if (!xwait(&bars->vfull[s], (tg / ST) & 1, bars, p.err, 3, p.wait)) return false;
                        tc_fence_after();
                        const uint32_t v_s = sbase + C::kStageOff + (s * 2 + 1) * C::kKTile;
#pragma unroll
                        for (int kk = 0; kk < kBN / 16; ++kk) {
                            const uint64_t vd = sdesc_sw128(v_s + kk * 16 * 128, C::kBlkK, 1024);
                            mma_ts(tmem + C::kColO + q * D, tmem + C::kColS + q * kBN + kk * 8, vd, idesc_pv,
                                   (j > 1 || kk > 0) ? 1u : 0u);
                        }
                        if constexpr (PRECISE) {
#pragma unroll
                            for (int kk = 0; kk < kBN / 16; ++kk) {
                                const uint64_t vd = sdesc_sw128(v_s + kk * 16 * 128, C::kBlkK, 1024);
                                mma_ts(tmem + C::kColO + q * D, tmem + C::kColS + q * kBN + 64 + kk * 8, vd, idesc_pv,
                                       1u);
                            }
                        }
                        tc_commit(&bars->kvempty[s]);
                        if (j + 2 >= it.ntiles) tc_commit(&bars->ofinal[q]);  // O_q's last tile
                        return true;
                    };
                    ok = split_s(0) && split_s(1);
                    for (int j = 0; ok && j < it.ntiles; ++j)
                        ok = split_pv(j) && (j + 2 >= it.ntiles || split_s(j + 2));
                }
                tm += it.ntiles;
            }
            // every MMA issued so far completes before tensor memory is freed
            tc_commit(&bars->drain);
            mbar_wait(&bars->drain, 0);
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ================= softmax + epilogue: query tile q, or in a split item the key
        // tiles of parity q =================
        const int q = (warp - 4) >> 2;
        const int r = threadIdx.x - 128 - q * 128;              // row = TMEM lane
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t colS = tmem + lane_base + C::kColS + q * kBN;
        const uint32_t colO = tmem + lane_base + C::kColO + q * D;
        int cw = 0, co = 0;  // phases consumed on sfull[q] and ofinal[q]
        bool alive = true;   // false after a failed wait; the remaining items are skipped
        for (int i = i0; i < i1; ++i) {
            const ExtendItem *itp = p.items + i;
            const XItem it = load_item(itp, TQ, p.packs);
            if (!it.split && q >= it.nq) continue;
            if (!alive) {
                // the other warpgroup meets the same barrier on every split item
                if (it.split) named_bar_and(kBarSplit, 256, false);
                continue;
            }
            // token of this row within the item (packed: within its row group r / 32) and the
            // last position it sees
            const int t = it.pk ? (r & 31) / G : (it.split ? 0 : q * TQ) + r / G;
            const int lim = (it.pk ? it.pk->qpos0[r >> 5] : it.qpos0) + t;
            float m = -INFINITY, l = 0.f;
            bool ok = true;
            int sg = 0, lt = 0, segpos = it.pos0;  // segment, tile within it, its first position
            const int jsecond = it.split ? 2 : 1;  // this warpgroup's second tile and later rescale O
            for (int j = 0; j < it.ntiles; ++j) {
                if (it.split && (j & 1) != q) {  // the other warpgroup's tile: move the cursor only
                    if (++lt * kBN >= it.nkeys[sg]) {
                        segpos += it.nkeys[sg];
                        ++sg;
                        lt = 0;
                    }
                    continue;
                }
                // lanes leave together: a split warp must not reach the .sync.aligned tcgen05 ops
                if (!__all_sync(0xffffffffu, xwait(&bars->sfull[q], cw & 1, bars, p.err, 8, p.wait))) {
                    ok = false;
                    break;
                }
                ++cw;
                tc_fence_after();
                const int kl0 = lt * kBN;                       // key index of column 0 in the segment
                const int kp0 = (it.pk ? it.pk->spos[sg] : segpos) + kl0;  // its context position
                const int nvalid = min(kBN, it.nkeys[sg] - kl0);
                // packed: a member's own keys are hidden from the other row groups (warp-uniform)
                const bool seen = !it.pk || it.pk->sgrp[sg] < 0 || it.pk->sgrp[sg] == (r >> 5);
                if (++lt * kBN >= it.nkeys[sg]) {
                    segpos += it.nkeys[sg];
                    ++sg;
                    lt = 0;
                }
                const int ncaus = lim - kp0 + 1;                // columns <= lim
                const int lastc = seen ? min(nvalid, ncaus) : 0;  // columns [0, lastc) visible
                // warp-uniform: the tcgen05.ld/st below are .sync.aligned, so every lane of
                // the warp must take the same path (lastc differs between rows of a causal tile)
                const bool full = __all_sync(0xffffffffu, lastc >= kBN);
                uint32_t sv[kBN];
#pragma unroll
                for (int c4 = 0; c4 < kBN / 32; ++c4) tmem_ld32(colS + c4 * 32, sv + c4 * 32);
                tmem_ld_wait();
                if (!full) {
#pragma unroll
                    for (int c = 0; c < kBN; ++c) if (c >= lastc) sv[c] = __float_as_uint(-INFINITY);
                }
                float mx[4];  // 3-input max: two new scores per instruction, 4 chains
#pragma unroll
                for (int c = 0; c < 4; ++c) mx[c] = __uint_as_float(sv[c]);
#pragma unroll
                for (int c = 4; c < kBN; c += 2)
                    mx[(c >> 1) & 3] = fmax3(mx[(c >> 1) & 3], __uint_as_float(sv[c]), __uint_as_float(sv[c + 1]));
                const float mt = fmaxf(fmax3(mx[0], mx[1], mx[2]), mx[3]) * p.scale_log2;
                float alpha = 1.f;
                bool rescale = false;
                if (mt > m + kRescaleThreshold || m == -INFINITY) {
                    alpha = (m == -INFINITY) ? 0.f : ex2(m - mt);
                    rescale = (j >= jsecond) && (m != -INFINITY);
                    m = mt;
                }
                // exponent reference: the larger of m and the tile max (arguments <= 0)
                const float mref = fmaxf(m, mt);
                const float neg_mref = (mref == -INFINITY) ? 0.f : -mref;
                float ls[4] = {0.f, 0.f, 0.f, 0.f};
                if constexpr (PRECISE) {
                    exp_pack_precise(sv, colS, p.scale_log2, neg_mref, mt > m ? ex2(mt - m) : 1.f, ls);
                } else if (__any_sync(0xffffffffu, mt > m)) {
                    const float f = mt > m ? ex2(mt - m) : 1.f;  // <= 2^8 (m is then finite)
                    exp_pack_regs<true>(sv, colS, p.scale_log2, neg_mref, pack_bf16x2(f, f), ls);
                } else {
                    exp_pack_regs<false>(sv, colS, p.scale_log2, neg_mref, 0u, ls);
                }
                const float ls0 = ls[0] + ls[2], ls1 = ls[1] + ls[3];
                l = l * alpha + (ls0 + ls1);
                // this warpgroup's previous P.V is complete: its S of this tile was issued
                // after it.  The whole warp rescales when any of its rows must
                // (.sync.aligned), the others by 1.
                if (__any_sync(0xffffffffu, rescale)) {
                    const float f = rescale ? alpha : 1.f;
#pragma unroll 1
                    for (int c4 = 0; c4 < D / 32; ++c4) {
                        uint32_t ov[32];
                        tmem_ld32(colO + c4 * 32, ov);
                        tmem_ld_wait();
#pragma unroll
                        for (int c = 0; c < 32; ++c) ov[c] = __float_as_uint(__uint_as_float(ov[c]) * f);
                        tmem_st32(colO + c4 * 32, ov);
                    }
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(&bars->pfull[q]);
            }
            bool fin = __all_sync(0xffffffffu, ok && xwait(&bars->ofinal[q], co & 1, bars, p.err, 10, p.wait));
            if (it.split) {
                // exchange the row's running max and sum with the other warpgroup; both
                // warpgroups leave together when either gave up on a wait
                s_ml[q][r] = make_float2(m, l);
                tc_fence_before();
                fin = named_bar_and(kBarSplit, 256, fin);
            }
            if (!fin) {
                alive = false;
                continue;
            }
            ++co;
            tc_fence_after();
            const bool valid = t < (it.pk ? it.pk->ntok[r >> 5] : it.ntok);
            const int tok = (it.pk ? it.pk->tok0[r >> 5] : it.tok0) + t;
            const int head = it.g * G + (r % G);
            if (!it.split) {
#pragma unroll 1
                for (int c4 = 0; c4 < D / 32; ++c4) {
                    uint32_t ov[32];
                    tmem_ld32(colO + c4 * 32, ov);
                    tmem_ld_wait();
                    if (!valid) continue;
                    write_out<D>(p, it, t, tok, head, c4, ov, m, l);
                }
            } else {
                // O = O_0 f_0 + O_1 f_1 over the common max; warpgroup q writes the columns
                // [q D / 2, (q + 1) D / 2)
                const float2 other = s_ml[q ^ 1][r];
                const float mm = fmaxf(m, other.x);
                const float fs = m == -INFINITY ? 0.f : ex2(m - mm);
                const float fo = other.x == -INFINITY ? 0.f : ex2(other.x - mm);
                const float f0 = q == 0 ? fs : fo, f1 = q == 0 ? fo : fs;
                l = l * fs + other.y * fo;
                m = mm;
                const uint32_t colO0 = tmem + lane_base + C::kColO;
#pragma unroll 1
                for (int c4 = q * (D / 64); c4 < (q + 1) * (D / 64); ++c4) {
                    uint32_t ov[32], ov1[32];
                    tmem_ld32(colO0 + c4 * 32, ov);
                    tmem_ld32(colO0 + D + c4 * 32, ov1);
                    tmem_ld_wait();
#pragma unroll
                    for (int c = 0; c < 32; ++c)
                        ov[c] = __float_as_uint(fmaf(__uint_as_float(ov[c]), f0, __uint_as_float(ov1[c]) * f1));
                    if (!valid) continue;
                    write_out<D>(p, it, t, tok, head, c4, ov, m, l);
                }
            }
            tc_fence_before();  // the next item's first P.V overwrites O after our next arrive
            // split: both warpgroups have read O_0 and O_1 before either arrives on the next item
            if (it.split) named_bar_sync(kBarSplit, 256);
        }
    }

    // ---- teardown: every copy has landed (consumed, or drained by the producer after an
    // abort) and every MMA has completed (drained by the issuer)
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
    if (!p.pdl_wait_start) pdl_wait();  // complete only after the preceding kernel
}

// The kernel's tensor maps: Q tiles, K and V boxes, and Q row groups (packed items).
struct XMaps {
    CUtensorMap q, k, v, qg;
};

template <int D, int G, bool PRECISE>
static int launch_extend(const ExtendParams &p, const XMaps &mp, int nctas, cudaStream_t s, bool pdl) {
    constexpr int smem = XCfg<D>::kSmem;
    static_assert(smem <= 232448, "shared memory budget");
    auto kern = extend_kernel<D, G, PRECISE>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return PKV_E_CUDA;
    // persistent: the plan's CTA lists
    return launch_pdl(kern, dim3(nctas), dim3(384), smem, s, pdl, p, mp.q, mp.k, mp.v, mp.qg) == cudaSuccess ? PKV_OK
                                                                                                     : PKV_E_CUDA;
}

template <int D, bool PRECISE>
static int dispatch_g(int G, const ExtendParams &p, const XMaps &mp, int n, cudaStream_t s, bool pdl) {
    switch (G) {
        case 1: return launch_extend<D, 1, PRECISE>(p, mp, n, s, pdl);
        case 2: return launch_extend<D, 2, PRECISE>(p, mp, n, s, pdl);
        case 4: return launch_extend<D, 4, PRECISE>(p, mp, n, s, pdl);
        case 8: return launch_extend<D, 8, PRECISE>(p, mp, n, s, pdl);
        default: return PKV_E_UNSUPPORTED;
    }
}

template <int D>
static int dispatch_extend(int G, const ExtendParams &p, const XMaps &mp, int n, cudaStream_t s, bool precise,
                           bool pdl) {
    return precise ? dispatch_g<D, true>(G, p, mp, n, s, pdl) : dispatch_g<D, false>(G, p, mp, n, s, pdl);
}

template <int D>
static int launch_gather(const GatherParams &p, bool fp8, int nunits, cudaStream_t s) {
    return launch_pdl(fp8 ? gather_kernel<D, true> : gather_kernel<D, false>, dim3(nunits), dim3(256), 0, s, true, p) ==
                   cudaSuccess
               ? PKV_OK
               : PKV_E_CUDA;
}

int check_call(const pkv_pool *pool, const pkv_batch *batch, const void *q, void *o, const pkv_plan_info *info,
               const void *plan_dev, void *workspace, size_t ws_bytes, int op);
int launch_merge(const pkv_plan_info *info, const void *plan_dev, const float *rec_acc, const float *rec_ml,
                 uint16_t *o, cudaStream_t s);

// Tensor maps: Q as [rows][Hq][D] (box 64 x G x 128/G, and 64 x G x 32/G for one row group
// of a packed tile); gathered K/V as [keys][Hkv][D] (box 64 x 1 x 128): every box lands as
// 128 (or 32) rows of 128 bytes, 128-byte swizzled.
static int make_maps(const void *q, int64_t qrows, const uint16_t *kg, const uint16_t *vg, int64_t nkeys, int D,
                     int hq, int hkv, XMaps *mp) {
    const int G = hq / hkv;
    CUtensorMap *qm = &mp->q, *km = &mp->k, *vm = &mp->v;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)hq, (cuuint64_t)std::max<int64_t>(qrows, 1)};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)hq * D * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)(128 / G)};
    if (encode_tiled(qm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(q), dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
        return PKV_E_CUDA;
    cuuint32_t gbox[3] = {64, (cuuint32_t)G, (cuuint32_t)(32 / G)};
    if (encode_tiled(&mp->qg, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(q), dims, strides, gbox,
                     CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
        return PKV_E_CUDA;
    cuuint64_t kdims[3] = {(cuuint64_t)D, (cuuint64_t)hkv, (cuuint64_t)std::max<int64_t>(nkeys, 1)};
    cuuint64_t kstrides[2] = {(cuuint64_t)D * 2, (cuuint64_t)hkv * D * 2};
    cuuint32_t kbox[3] = {64, 1, 128};
    if (encode_tiled(km, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t *>(kg), kdims, kstrides, kbox,
                     CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS ||
        encode_tiled(vm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t *>(vg), kdims, kstrides, kbox,
                     CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
        return PKV_E_CUDA;
    return PKV_OK;
}

// Decode over shared spans with many members, on the tensor cores: the plan's spans are
// gathered once into the workspace (bf16 [key][Hkv][D]), the member requests' query rows
// are gathered next to them, and extend-kernel items (two 128-row query tiles of 128/G
// members x G heads, one KV head, a chunk of the span; no mask: every query comes after
// the span) write each member's partial record for the chunk.
struct SpanBufs {
    uint16_t *kg, *vg, *qg;
    int64_t nunits, nkeys, nq, nx;
};
static SpanBufs span_bufs(const pkv_plan_info *info, uint8_t *ws) {
    SpanBufs b;
    b.nx = info->offsets[8];
    b.nunits = info->offsets[10];
    b.nkeys = info->offsets[11];
    b.nq = info->offsets[13];
    const int D = info->head_dim, hkv = info->num_kv_heads;
    b.kg = reinterpret_cast<uint16_t *>(ws + info->offsets[15]);
    b.vg = b.kg + (size_t)b.nkeys * hkv * D;
    const size_t qoff = ((size_t)info->offsets[15] + 2 * (size_t)b.nkeys * hkv * D * 2 + 255) & ~size_t(255);
    b.qg = reinterpret_cast<uint16_t *>(ws + qoff);
    return b;
}

int decode_span_gather(const pkv_pool *pool, const pkv_batch *batch, const void *q, const pkv_plan_info *info,
                       const uint8_t *plan, uint8_t *ws, cudaStream_t s) {
    const SpanBufs b = span_bufs(info, ws);
    if (b.nx == 0) return PKV_OK;
    const int D = info->head_dim, hq = info->num_q_heads, hkv = info->num_kv_heads;
    GatherParams gp;
    gp.k_pool = static_cast<const uint8_t *>(pool->k);
    gp.v_pool = static_cast<const uint8_t *>(pool->v);
    gp.slot_bytes = slot_bytes(pool);
    gp.num_slots = pool->num_slots;
    gp.hkv = hkv;
    gp.req_to_token = batch->req_to_token;
    gp.rt_stride = batch->stride;
    gp.rt_rows = batch->num_rows;
    gp.page_shift = page_shift_of(batch);
    gp.req_pool_indices = batch->req_pool_indices;
    gp.units = reinterpret_cast<const GatherUnit *>(plan + info->offsets[9]);
    gp.k_out = b.kg;
    gp.v_out = b.vg;
    gp.err = reinterpret_cast<int32_t *>(ws);
    gp.pdl_wait_start = 1;
    // one launch: the span keys, then the member query rows
    gp.nunits = (int32_t)b.nunits;
    gp.q_src = static_cast<const uint4 *>(q);
    gp.q_out = reinterpret_cast<uint4 *>(b.qg);
    gp.q_rows = reinterpret_cast<const int32_t *>(plan + info->offsets[12]);
    gp.q_batch = batch->batch;
    gp.q_row_vecs = hq * D / 8;
    const bool fp8 = pool->dtype == PKV_FP8_E4M3;
    return D == 128 ? launch_gather<128>(gp, fp8, (int)(b.nunits + b.nq), s)
                    : launch_gather<64>(gp, fp8, (int)(b.nunits + b.nq), s);
}

int decode_span_attend(const pkv_pool *pool, const void *q, float sm_scale, const pkv_plan_info *info,
                       const uint8_t *plan, uint8_t *ws, float *rec_acc, float *rec_ml, cudaStream_t s,
                       bool after_decode) {
    (void)q;
    const SpanBufs b = span_bufs(info, ws);
    if (b.nx == 0) return PKV_OK;
    const int D = info->head_dim, hq = info->num_q_heads, hkv = info->num_kv_heads, G = hq / hkv;
    const bool fp8 = pool->dtype == PKV_FP8_E4M3;
    XMaps mp;
    int rc = make_maps(b.qg, b.nq, b.kg, b.vg, b.nkeys, D, hq, hkv, &mp);
    if (rc) return rc;
    ExtendParams p;
    p.o = nullptr;  // every item writes records
    p.hkv = hkv;
    p.hq = hq;
    p.scale_log2 = sm_scale * (fp8 ? pool->k_scale : 1.f) * kLog2eX;
    p.v_scale = fp8 ? pool->v_scale : 1.f;
    p.items = reinterpret_cast<const ExtendItem *>(plan + info->offsets[7]);
    p.num_items = (int32_t)b.nx;
    p.err = reinterpret_cast<int32_t *>(ws);
    p.rec_acc = rec_acc;
    p.rec_ml = rec_ml;
    p.rec_list = reinterpret_cast<const int32_t *>(plan + info->offsets[14]);
    p.packs = nullptr;
    p.wait = wait_policy(wait_limit_ns());
    // Right after the gather, wait for it first; after the decode kernel (which itself waited
    // for the gather), read the gathered rows at once and wait for the decode kernel only
    // before exiting, so the merge that follows sees every record.
    p.pdl_wait_start = after_decode ? 0 : 1;
    // the spans' items, then the short requests' items (precise weights)
    const ExtendItem *items = reinterpret_cast<const ExtendItem *>(plan + info->offsets[7]);
    const int64_t nprec = info->offsets[18];
    for (int part = 0; part < 2; ++part) {
        const int64_t n = part == 0 ? b.nx - nprec : nprec;
        if (n == 0) continue;
        p.items = items + (part == 0 ? 0 : b.nx - nprec);
        p.num_items = (int32_t)n;
        p.cta_off = reinterpret_cast<const int32_t *>(plan + info->offsets[part == 0 ? 16 : 19]);
        const int64_t nctas = info->offsets[part == 0 ? 17 : 20];
        if (nctas < 1 || nctas > n || nprec > b.nx) return PKV_E_PLAN;
        rc = D == 128 ? dispatch_extend<128>(G, p, mp, (int)nctas, s, part == 1, true)
                      : dispatch_extend<64>(G, p, mp, (int)nctas, s, part == 1, true);
        if (rc) return rc;
    }
    return PKV_OK;
}

}  // namespace pkv

namespace pkv {

int launch_store(const pkv_pool *pool, const void *k_new, const void *v_new, const int32_t *out_cache_loc, int64_t n,
                 void *workspace, void *ctx_k, void *ctx_v, const int32_t *ctx_row, int64_t ctx_rows, cudaStream_t s);

// The extend items of a plan over keys already laid out as bf16 [key][Hkv][D] arrays (the
// workspace's gathered runs, or a caller's context arrays), then the merge.
static int extend_items(const pkv_pool *pool, const void *q, void *o, float sm_scale, const pkv_plan_info *info,
                        const void *plan_dev, uint8_t *ws, const uint16_t *kg, const uint16_t *vg, int64_t nkeys,
                        cudaStream_t s) {
    const int D = info->head_dim, hq = info->num_q_heads, hkv = info->num_kv_heads, G = hq / hkv;
    const bool fp8 = pool->dtype == PKV_FP8_E4M3;
    const uint8_t *plan = static_cast<const uint8_t *>(plan_dev);
    float *rec_acc = reinterpret_cast<float *>(ws + kWorkspaceHeader);
    float *rec_ml = rec_acc + (size_t)info->num_records * hq * D;
    XMaps mp;
    int rc = make_maps(q, info->total_q, kg, vg, nkeys, D, hq, hkv, &mp);
    if (rc) return rc;

    ExtendParams p;
    p.o = static_cast<uint16_t *>(o);
    p.hkv = hkv;
    p.hq = hq;
    p.scale_log2 = sm_scale * (fp8 ? pool->k_scale : 1.f) * kLog2eX;
    p.v_scale = fp8 ? pool->v_scale : 1.f;
    p.items = reinterpret_cast<const ExtendItem *>(plan + info->offsets[0]);
    p.num_items = info->num_items;
    p.err = reinterpret_cast<int32_t *>(ws);
    p.rec_acc = rec_acc;
    p.rec_ml = rec_ml;
    p.rec_list = nullptr;
    p.wait = wait_policy(wait_limit_ns());
    // The extend kernels of an extend call are ordinary stream launches: they start once the
    // store / gather before them has completed.  (Launched programmatically, so that their
    // CTAs took SMs while the store was still running, the serving loop's prefill calls
    // intermittently found a K/V tile row of another CTA written over a CTA's pipeline
    // barriers, and the pipeline timed out; with ordinary launches it never did.)
    p.pdl_wait_start = 1;  // the gather (or the store) just before wrote the keys
    p.packs = info->offsets[14] > 0 ? reinterpret_cast<const PackInfo *>(plan + info->offsets[13]) : nullptr;
    void *ev0 = g_kernel_events[0], *ev1 = g_kernel_events[1];
    g_kernel_events[0] = g_kernel_events[1] = nullptr;
    if (ev0 && cudaEventRecord(static_cast<cudaEvent_t>(ev0), s) != cudaSuccess) return PKV_E_CUDA;
    // the main item list, then (if any) the items whose rows see few keys (precise weights)
    for (int part = 0; part < 2; ++part) {
        const int64_t nitems = part == 0 ? info->num_items - info->offsets[10] : info->offsets[10];
        if (nitems == 0) continue;
        p.items = reinterpret_cast<const ExtendItem *>(plan + info->offsets[part == 0 ? 0 : 9]);
        p.num_items = (int32_t)nitems;
        p.cta_off = reinterpret_cast<const int32_t *>(plan + info->offsets[part == 0 ? 7 : 11]);
        const int64_t nctas = info->offsets[part == 0 ? 8 : 12];
        if (nctas < 1 || nctas > nitems) return PKV_E_PLAN;
        rc = D == 128 ? dispatch_extend<128>(G, p, mp, (int)nctas, s, part == 1, false)
                      : dispatch_extend<64>(G, p, mp, (int)nctas, s, part == 1, false);
        if (rc) return rc;
    }
    if (ev1 && cudaEventRecord(static_cast<cudaEvent_t>(ev1), s) != cudaSuccess) return PKV_E_CUDA;
    return launch_merge(info, plan_dev, rec_acc, rec_ml, p.o, s);
}

}  // namespace pkv

namespace pkv {

// pkv_attn_extend, and with `store` (a fused-store plan) the store of the new tokens first:
// into the pool and straight into their gathered rows; the gather (cached positions only)
// then runs beside the store and waits for it only before exiting.
static int extend_call(const pkv_pool *pool, const pkv_batch *batch, const void *q, void *o, float sm_scale,
                       const void *k_new, const void *v_new, const int32_t *out_cache_loc, bool store,
                       const pkv_plan_info *info, const void *plan_dev, void *workspace, size_t ws_bytes,
                       void *stream) {
    int rc = check_call(pool, batch, q, o, info, plan_dev, workspace, ws_bytes, 2);
    if (rc) return rc;
    if (info->offsets[16] != (store ? 2 : 0)) return PKV_E_PLAN;
    if (store) {
        if (info->total_q > 0 && (!k_new || !v_new || !out_cache_loc)) return PKV_E_INVALID;
        if ((reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new)) & 15) return PKV_E_INVALID;
    }
    if (info->num_items == 0 && !(store && info->total_q > 0)) return PKV_OK;
    const int D = info->head_dim, hq = info->num_q_heads, hkv = info->num_kv_heads;
    const bool fp8 = pool->dtype == PKV_FP8_E4M3;
    const uint8_t *plan = static_cast<const uint8_t *>(plan_dev);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

    // workspace: header | records (acc, ml) | gathered K | gathered V
    const size_t rec_bytes = (size_t)info->num_records * hq * (D + 2) * 4;
    uint16_t *kg = reinterpret_cast<uint16_t *>(ws + kWorkspaceHeader + ((rec_bytes + 255) & ~size_t(255)));
    const int64_t nkeys = info->offsets[6];  // gathered keys
    uint16_t *vg = kg + (size_t)nkeys * hkv * D;

    GatherParams gp;
    gp.k_pool = static_cast<const uint8_t *>(pool->k);
    gp.v_pool = static_cast<const uint8_t *>(pool->v);
    gp.slot_bytes = slot_bytes(pool);
    gp.num_slots = pool->num_slots;
    gp.hkv = hkv;
    gp.req_to_token = batch->req_to_token;
    gp.rt_stride = batch->stride;
    gp.rt_rows = batch->num_rows;
    gp.page_shift = page_shift_of(batch);
    gp.req_pool_indices = batch->req_pool_indices;
    gp.units = reinterpret_cast<const GatherUnit *>(plan + info->offsets[4]);
    gp.k_out = kg;
    gp.v_out = vg;
    gp.err = reinterpret_cast<int32_t *>(ws);
    gp.pdl_wait_start = 1;
    const int nunits = (int)info->offsets[5];
    gp.nunits = nunits;  // no query rows to copy
    gp.q_src = nullptr;
    gp.q_out = nullptr;
    gp.q_rows = nullptr;
    gp.q_batch = gp.q_row_vecs = 0;
    if (store && info->total_q > 0) {
        rc = launch_store(pool, k_new, v_new, out_cache_loc, info->total_q, ws, kg, vg,
                          reinterpret_cast<const int32_t *>(plan + info->offsets[15]), nkeys, s);
        if (rc) return rc;
        gp.pdl_wait_start = 0;  // it reads no row the store writes
    }
    if (nunits > 0) {
        rc = D == 128 ? launch_gather<128>(gp, fp8, nunits, s) : launch_gather<64>(gp, fp8, nunits, s);
        if (rc) return rc;
    }
    if (info->num_items == 0) return PKV_OK;
    return extend_items(pool, q, o, sm_scale, info, plan_dev, ws, kg, vg, nkeys, s);
}

}  // namespace pkv

extern "C" int pkv_attn_extend(const pkv_pool *pool, const pkv_batch *batch, const void *q, void *o, float sm_scale,
                               const pkv_plan_info *info, const void *plan_dev, void *workspace, size_t ws_bytes,
                               void *stream) {
    return pkv::extend_call(pool, batch, q, o, sm_scale, nullptr, nullptr, nullptr, false, info, plan_dev, workspace,
                            ws_bytes, stream);
}

extern "C" int pkv_attn_extend_store(const pkv_pool *pool, const pkv_batch *batch, const void *q, void *o,
                                     float sm_scale, const void *k_new, const void *v_new,
                                     const int32_t *out_cache_loc, const pkv_plan_info *info, const void *plan_dev,
                                     void *workspace, size_t ws_bytes, void *stream) {
    return pkv::extend_call(pool, batch, q, o, sm_scale, k_new, v_new, out_cache_loc, true, info, plan_dev, workspace,
                            ws_bytes, stream);
}

extern "C" int pkv_attn_extend_ctx(const pkv_pool *pool, const void *q, void *o, float sm_scale, const void *k_new,
                                   const void *v_new, const int32_t *out_cache_loc, void *ctx_k, void *ctx_v,
                                   int64_t ctx_rows, const pkv_plan_info *info, const void *plan_dev,
                                   void *workspace, size_t ws_bytes, void *stream) {
    using namespace pkv;
    int rc = validate_pool(pool);
    if (rc) return rc;
    if (!q || !o || !info || !plan_dev || !workspace || !ctx_k || !ctx_v) return PKV_E_INVALID;
    if (info->op != 2 || info->offsets[16] != 1 || info->offsets[6] != ctx_rows) return PKV_E_PLAN;
    if (info->num_kv_heads != pool->num_kv_heads || info->head_dim != pool->head_dim) return PKV_E_PLAN;
    if (ws_bytes < info->workspace_bytes) return PKV_E_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(plan_dev) & 15) || (reinterpret_cast<uintptr_t>(workspace) & 255))
        return PKV_E_INVALID;
    if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(o) | reinterpret_cast<uintptr_t>(ctx_k) |
         reinterpret_cast<uintptr_t>(ctx_v)) & 15)
        return PKV_E_INVALID;
    const int64_t n = info->total_q;
    if (n == 0) return PKV_OK;
    if (!k_new || !v_new || !out_cache_loc) return PKV_E_INVALID;
    if ((reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new)) & 15) return PKV_E_INVALID;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const uint8_t *plan = static_cast<const uint8_t *>(plan_dev);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    // the new tokens into the pool and, as the pool now holds them, into their context rows
    rc = launch_store(pool, k_new, v_new, out_cache_loc, n, ws, ctx_k, ctx_v,
                      reinterpret_cast<const int32_t *>(plan + info->offsets[15]), ctx_rows, s);
    if (rc) return rc;
    if (info->num_items == 0) return PKV_OK;
    return extend_items(pool, q, o, sm_scale, info, plan_dev, ws, static_cast<const uint16_t *>(ctx_k),
                        static_cast<const uint16_t *>(ctx_v), ctx_rows, s);
}
