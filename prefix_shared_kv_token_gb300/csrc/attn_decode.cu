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
// GB300 design: decode is a stream of K/V bytes, so the kernel is built to keep HBM busy.
//   * Persistent CTAs (the plan sizes the grid to the SMs) each walk a fixed, load-balanced
//     list of work items.  An item is (shared span chunk x up to 16/G member requests) or
//     (one request's unshared key chunk), over a *head group* of hg <= 8 KV heads.
//   * One producer warp streams 16-key tiles through a shared-memory ring without pausing
//     between items: for each key it issues one cp.async.bulk of the slot's whole head-group
//     row (hg * d elements, contiguous in the pool: 2 KB for 8 bf16 heads of 128) for K and
//     one for V, completing as transaction bytes on the stage's mbarrier.  Rows land at a
//     padded stride so the fragment loads below are bank-conflict free.
//   * Consumer warp w owns KV head g0 + w: its 16 MMA rows are the item's requests x G query
//     heads.  QK^T and PV use mma.sync m16n8k16 (bf16 in, fp32 accumulate; the d-order in
//     each k-step is permuted identically for Q and K so every lane loads 8 contiguous
//     bytes), with an online softmax in the log2 domain.  The next item's query fragments
//     are fetched while the current item runs.
//   * An item that covers part of a request writes a partial record (m, l, acc); a merge
//     kernel combines a request's records with the log-sum-exp identity.  An item that
//     covers a whole request writes its output directly.
//   * fp8 pools: raw e4m3 rows land in the ring and each warp converts its own head's rows
//     exactly to bf16 in a private tile (releasing the stage at once); k_scale folds into
//     the logit scale, v_scale into the output.
//   * Every wait is bounded (the launch's wait limit, 2 s by default); on expiry the CTA
//     records PKV_DERR_TIMEOUT, its warps stop, and the producer lets every copy it issued
//     land before it exits.

#include "../../include/pkv.h"
#include "common.cuh"
#include "launch.h"

// persistent decode CTAs per SM for a head group of hg KV heads (the planner's rule)
int decode_ctas_per_sm(int32_t hg, int32_t d);

namespace pkv {

struct DecodeParams {
    const uint8_t *k_pool;
    const uint8_t *v_pool;
    int64_t num_slots;
    int32_t hkv, hq;
    int32_t hg;         // KV heads per item = consumer warps
    const int32_t *req_to_token;
    int64_t rt_stride;
    int32_t rt_rows;
    int32_t page_shift;  // 0: token table; else log2 of the page size (page table)
    int32_t batch;
    const int32_t *req_pool_indices;
    const int32_t *seq_lens;
    const uint16_t *q;  // bf16 bits [batch][hq][D]
    uint16_t *o;
    float scale_log2;   // sm_scale * k_scale * log2(e)
    float v_scale;
    const DecodeItem *items;
    const int32_t *cta_off;  // items of CTA b: [cta_off[b], cta_off[b + 1])
    const int32_t *row_req;
    const int32_t *row_rec;
    int64_t slot_bytes;  // from one slot's pool row to the next
    int32_t joint;       // one copy per key brings its K and V rows (interleaved pool, hg == hkv)
    float *rec_acc;     // [rec][hq][D]
    float *rec_ml;      // [rec][hq][2]
    int32_t *err;
    WaitPolicy wait;    // pipeline waits (pkv_set_wait_limit_ns)
    int32_t late_wait;  // 1: the kernel before (the span gather) wrote nothing this one reads; an
                        // extra warp waits for it and then releases the next kernel, the others
                        // start at once
};

constexpr int kBK = 16;       // keys per tile
constexpr int kHdr = 256;     // barriers, abort flag, per-stage tile info
constexpr float kLog2e = 1.4426950408889634f;

// Per-stage description written by the producer before it arms the stage.
struct TileInfo {
    int32_t kpos;   // position of the tile's first key
    int32_t k1;     // one past the item's last key
    int32_t item;   // plan item
    int32_t flags;  // kFirst | kLast, or kEnd (no keys: the CTA's list is done)
};
constexpr int32_t kFirst = 1, kLast = 2, kEnd = 4;

// Shared-memory geometry for a head group of hg KV heads.  bf16: K rows at a stride of
// 32 (mod 128) bytes, V rows at 16 (mod 128), so the 8-byte K fragment loads and the
// 16-byte ldmatrix.trans rows of a warp hit distinct banks.  fp8: raw rows of hg * D codes;
// each consumer warp converts its head into a private bf16 tile with those strides.
// Joint layout (an interleaved pool read by a head group that covers every KV head): each
// key's K row and V row arrive together by one copy, [K row | V row] at a stride of 2 rowb + 32
// (bf16: the K loads stay conflict-free; the V rows share that stride).
template <int D, bool FP8>
struct DGeo {
    static constexpr int kStages = FP8 ? 4 : 3;
    static constexpr int kConvK = 2 * D + 32, kConvV = 2 * D + 16;
    static constexpr int kConvBytes = kBK * (kConvK + kConvV);  // per consumer warp
    int rowb;     // pool bytes of one key's head-group row, per tensor
    int kstride;  // stage offset of key j's K row: j * kstride
    int vbase, vstride;  // of key j's V row: vbase + j * vstride
    int stage;    // bytes per stage
    int conv;     // offset of the conversion tiles (fp8)
    int bytes;    // dynamic shared memory
    __host__ __device__ DGeo(int hg, bool joint) {
        rowb = hg * D * (FP8 ? 1 : 2);
        if (joint) {
            kstride = vstride = 2 * rowb + (FP8 ? 0 : 32);
            vbase = rowb;
            stage = kBK * kstride;
        } else {
            kstride = FP8 ? rowb : rowb + 32;
            vstride = FP8 ? rowb : rowb + 16;
            vbase = kBK * kstride;
            stage = kBK * (kstride + vstride);
        }
        conv = kHdr + kStages * stage;
        bytes = conv + (FP8 ? hg * kConvBytes : 0);
    }
};

// QUICK launches (a short wait limit) poll with test_wait and read the timer on every try;
// the others try_wait and read it every 256 retries.
template <bool QUICK>
PKV_DEV bool dwait(uint64_t *bar, uint32_t parity, int32_t *abort_flag, int32_t *err, int where,
                   const WaitPolicy &wp) {
    if (QUICK ? mbar_test_wait(bar, parity) : mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (QUICK ? mbar_test_wait(bar, parity) : mbar_try_wait(bar, parity)) return true;
        if (QUICK || (it & 255u) == 0) {
            if (*reinterpret_cast<volatile int32_t *>(abort_flag)) return false;
            if (global_timer_ns() - t0 > wp.limit_ns) {
                set_error(err, DERR_TIMEOUT | where);
                *reinterpret_cast<volatile int32_t *>(abort_flag) = 1;
                return false;
            }
        }
    }
}

// Query fragments of one item for consumer warp w: rows i = r and r + 8 of the 16-row tile
// (request i / G of the item, query head (g0 + w) * G + i % G); rows past nreq * G are zero.
template <int D, int G>
struct ItemRows {
    uint32_t qf[D / 16][4];
    int32_t req[2];
    int32_t g0, row_off;
};

template <int D, int G>
PKV_DEV void load_rows(const DecodeParams &p, int item, int w, ItemRows<D, G> &x) {
    const int lane = threadIdx.x & 31, r = lane >> 2, c = lane & 3;
    const DecodeItem it = p.items[item];
    x.g0 = it.g0;
    x.row_off = it.row_off;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int i = r + 8 * h;
        x.req[h] = i < it.nreq * G ? __ldg(p.row_req + it.row_off + i / G) : -1;
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int head = (it.g0 + w) * G + (r + 8 * h) % G;
        const uint16_t *qrow = p.q + ((int64_t)(x.req[h] < 0 ? 0 : x.req[h]) * p.hq + head) * D + 4 * c;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            uint2 v = make_uint2(0u, 0u);
            if (x.req[h] >= 0) v = __ldg(reinterpret_cast<const uint2 *>(qrow + ks * 16));
            x.qf[ks][h] = v.x;       // k-slots 2c, 2c+1
            x.qf[ks][2 + h] = v.y;   // k-slots 2c+8, 2c+9
        }
    }
}

// fp8: convert this warp's head (codes at column `col` of each raw row) into its bf16 tiles.
template <int D>
PKV_DEV void convert_head(const uint8_t *raw, const DGeo<D, true> &geo, int col, uint8_t *conv) {
    using Gm = DGeo<D, true>;
    const int lane = threadIdx.x & 31;
    constexpr int kChunks = kBK * D / 16;  // 16 codes per chunk, per tensor
#pragma unroll 2
    for (int i = lane; i < 2 * kChunks; i += 32) {
        const int tensor = i >= kChunks, ci = i - tensor * kChunks;
        const int key = ci / (D / 16), cc = ci % (D / 16);
        const int row = tensor ? geo.vbase + key * geo.vstride : key * geo.kstride;
        const uint4 x = *reinterpret_cast<const uint4 *>(raw + row + col + cc * 16);
        const uint32_t wd[4] = {x.x, x.y, x.z, x.w};
        uint32_t y[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            y[2 * k] = e4m3x2_to_bf16x2((uint16_t)(wd[k] & 0xFFFFu));
            y[2 * k + 1] = e4m3x2_to_bf16x2((uint16_t)(wd[k] >> 16));
        }
        uint8_t *dst = conv + (tensor ? kBK * Gm::kConvK + key * Gm::kConvV : key * Gm::kConvK) + cc * 32;
        reinterpret_cast<uint4 *>(dst)[0] = make_uint4(y[0], y[1], y[2], y[3]);
        reinterpret_cast<uint4 *>(dst)[1] = make_uint4(y[4], y[5], y[6], y[7]);
    }
}

// Online-softmax state of one warp over its 16 rows (this lane: rows r and r + 8).
template <int D>
struct WarpState {
    float acc[D / 8][4];
    float m[2], l[2];
};

// One 16-key tile for this warp.  kt / vt point at key 0 of the warp's head; sk / sv are
// the row strides.  Keys at positions >= k1 are masked.
template <int D>
PKV_DEV void tile16(WarpState<D> &st, const uint32_t (&qf)[D / 16][4], const uint8_t *kt, int sk, const uint8_t *vt,
                    int sv, int kpos, int k1, float scale_log2) {
    const int lane = threadIdx.x & 31;
    const int r = lane >> 2, c = lane & 3;
    float s[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const uint2 b2 = *reinterpret_cast<const uint2 *>(kt + (nt * 8 + r) * sk + (ks * 16 + 4 * c) * 2);
            const uint32_t b[2] = {b2.x, b2.y};
            mma_bf16_16816(s[nt], qf[ks], b);
        }
    }
    // scale, mask (only an item's last tile can hold keys past k1), running max
    const bool ragged = kpos + kBK > k1;
    float mt[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            float x = s[nt][e] * scale_log2;
            if (ragged && kpos + nt * 8 + 2 * c + (e & 1) >= k1) x = -INFINITY;
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
    // weights rounded to the bf16 the P.V product uses; the row sums add exactly those
    uint32_t a[4];  // A fragment: row r keys 0-7, row r+8 keys 0-7, row r keys 8-15, row r+8 keys 8-15
    float ls[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const uint32_t pk = pack_bf16x2(ex2(s[nt][2 * hh] - mu[hh]), ex2(s[nt][2 * hh + 1] - mu[hh]));
            add_bf16x2_f32(pk, ls[hh][0], ls[hh][1]);
            a[2 * nt + hh] = pk;
        }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) st.l[h] = st.l[h] * alpha[h] + (ls[h][0] + ls[h][1]);
#pragma unroll
    for (int nd = 0; nd < D / 8; ++nd) {
        st.acc[nd][0] *= alpha[0];
        st.acc[nd][1] *= alpha[0];
        st.acc[nd][2] *= alpha[1];
        st.acc[nd][3] *= alpha[1];
    }
    // O += P V: V rows are keys; ldmatrix.trans yields the k-major B fragments
    const int mat = lane >> 3, mi = lane & 7;
    const uint32_t vrow = smem_u32(vt) + ((mat & 1) * 8 + mi) * sv;
#pragma unroll
    for (int nd = 0; nd < D / 8; nd += 2) {
        uint32_t bv[4];
        ldmatrix_x4_trans(bv, vrow + (nd + (mat >> 1)) * 16);
        mma_bf16_16816(st.acc[nd], a, bv);
        mma_bf16_16816(st.acc[nd + 1], a, bv + 2);
    }
}

// The producer's walk over its CTA's tiles: items [c0, c1) in order (an item whose
// positions are out of range is reported and skipped), each item's tiles cyclically from
// its start tile.  next_tile() returns the next tile with this lane's slot load issued, or a
// tile flagged kEnd after the last one.
struct TileCursor {
    int i, j, nt, jj, k0, k1, g0;
    const int32_t *rt;
};
struct TileSlot {
    TileInfo info;
    int32_t slot;  // this lane's key (lane & 15) of the tile; -1 past the item's end
    int32_t g0;
};

PKV_DEV TileSlot next_tile(const DecodeParams &p, TileCursor &cur, int c1, int key) {
    TileSlot e;
    while (cur.j >= cur.nt) {
        if (cur.i + 1 >= c1) {
            cur.i = c1;
            e.info.kpos = e.info.k1 = 0;
            e.info.item = -1;
            e.info.flags = kEnd;
            e.slot = -1;
            e.g0 = 0;
            return e;
        }
        ++cur.i;
        const DecodeItem it = p.items[cur.i];
        const int row = __ldg(p.req_pool_indices + it.src);
        const int k1 = it.k1 < 0 ? __ldg(p.seq_lens + it.src) : it.k1;
        if (row < 0 || row >= p.rt_rows || it.k0 < 0 || k1 > (p.rt_stride << p.page_shift) || k1 <= it.k0) {
            if ((threadIdx.x & 31) == 0) set_error(p.err, DERR_POSITION);
            continue;
        }
        cur.k0 = it.k0;
        cur.k1 = k1;
        cur.g0 = it.g0;
        cur.nt = (k1 - it.k0 + kBK - 1) / kBK;
        cur.j = 0;
        cur.jj = it.rot > 0 ? it.rot % cur.nt : 0;  // the softmax does not depend on key order
        cur.rt = p.req_to_token + (int64_t)row * p.rt_stride;
    }
    e.info.kpos = cur.k0 + cur.jj * kBK;
    e.info.k1 = cur.k1;
    e.info.item = cur.i;
    e.info.flags = (cur.j == 0 ? kFirst : 0) | (cur.j == cur.nt - 1 ? kLast : 0);
    e.g0 = cur.g0;
    const int kp = e.info.kpos + key;
    e.slot = kp < cur.k1 ? table_slot(cur.rt, kp, p.page_shift, p.num_slots) : -1;
    ++cur.j;
    cur.jj = cur.jj + 1 == cur.nt ? 0 : cur.jj + 1;
    return e;
}

template <int D, int G, bool FP8, bool QUICK>
__global__ void __launch_bounds__((D == 64 ? 288 : 320), (D == 64 ? 2 : 1)) decode_kernel(const DecodeParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    using Gm = DGeo<D, FP8>;
    constexpr int S = Gm::kStages;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *empty = full + 4;
    int32_t *abort_flag = reinterpret_cast<int32_t *>(smem + 64);
    TileInfo *tinfo = reinterpret_cast<TileInfo *>(smem + 128);
    uint8_t *ring = smem + kHdr;
    const Gm geo(p.hg, p.joint != 0);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool late = p.late_wait != 0;
    if (!late) {
        pdl_wait();     // the query tokens' K/V were stored just before
        pdl_trigger();  // the span pass may take SMs as this kernel's CTAs finish
    }
    const int c0 = __ldg(p.cta_off + blockIdx.x), c1 = __ldg(p.cta_off + blockIdx.x + 1);

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], p.hg);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (late && warp == p.hg + 1) {
        // After the span gather, which reads the pool but writes only its own rows, the other
        // warps stream at once: what they read (pool, tables, queries, plan) was complete
        // before the gather started, since the gather waited for the kernel before it.  This
        // warp waits for the gather, then lets the span pass (which reads the gather's rows)
        // be scheduled; the CTA completes only after the gather has.
        if (lane == 0) {
            pdl_wait();
            pdl_trigger();
        }
        return;
    }

    if (warp == p.hg) {
        // ------------------------------------------------------------------ producer warp
        // lanes 0-15: K row of key `lane` of the tile; lanes 16-31: V row of key `lane - 16`.
        // Joint layout: lanes 0-15 each bring key `lane`'s K and V rows with one copy.
        const int key = lane & 15;
        const bool joint = p.joint != 0;
        const bool is_v = !joint && lane >= 16;
        const bool issuer = !joint || lane < 16;
        const uint8_t *pool = is_v ? p.v_pool : p.k_pool;
        const int64_t head_bytes = (int64_t)D * (FP8 ? 1 : 2);
        const uint32_t copy_bytes = (uint32_t)geo.rowb * (joint ? 2u : 1u);
        // the slots of the next 4 tiles are in flight while the current tile is issued
        TileCursor cur;
        cur.i = c0 - 1;
        cur.j = cur.nt = 0;
        TileSlot e0 = next_tile(p, cur, c1, key), e1 = next_tile(p, cur, c1, key);
        TileSlot e2 = next_tile(p, cur, c1, key), e3 = next_tile(p, cur, c1, key);
        int t = 0;
        bool ended = false;  // the list ran out (tile t carries kEnd) rather than a wait giving up
        for (;; ++t) {
            const int s = t % S;
            if (t >= S && !__all_sync(0xffffffffu, dwait<QUICK>(&empty[s], ((t / S) - 1) & 1, abort_flag, p.err, 0x31, p.wait)))
                break;  // warp-uniform: every lane leaves together
            if (e0.info.flags & kEnd) {
                if (lane == 0) {
                    tinfo[s].flags = kEnd;
                    mbar_arrive(&full[s]);
                }
                ended = true;
                break;
            }
            const int kp = e0.info.kpos + key;
            const bool in = issuer && kp < e0.info.k1;
            const bool valid = in && e0.slot >= 0 && (int64_t)e0.slot < p.num_slots;
            if (in && !valid) set_error(p.err, DERR_SLOT_RANGE);
            uint8_t *dst = ring + s * geo.stage + (is_v ? geo.vbase + key * geo.vstride : key * geo.kstride);
            // no copy: a V row past the item's end, or either row of a bad slot, reads as zeros
            // (keys past the end are masked, so their K rows are left as they are; in the joint
            // layout the K row past the end is cleared with its V row)
            if (issuer && !valid && (in || is_v || joint)) {
                for (uint32_t b = 0; b < copy_bytes; b += 16) *reinterpret_cast<uint4 *>(dst + b) = make_uint4(0u, 0u, 0u, 0u);
                fence_proxy_async_smem();  // a later bulk copy rewrites this row
            }
            const uint32_t nvalid = __popc(__ballot_sync(0xffffffffu, valid));
            __syncwarp();
            if (lane == 0) {
                tinfo[s] = e0.info;
                mbar_arrive_expect_tx(&full[s], nvalid * copy_bytes);
            }
            __syncwarp();
            if (valid)
                bulk_copy_g2s(smem_u32(dst), pool + (int64_t)e0.slot * p.slot_bytes + (int64_t)e0.g0 * head_bytes,
                              copy_bytes, &full[s]);
            e0 = e1;
            e1 = e2;
            e2 = e3;
            e3 = next_tile(p, cur, c1, key);
        }
        // Let every copy this warp issued land before it leaves: the consumers may have given
        // up on a wait (and returned) while the last tiles were still in flight.  Tile t was
        // not issued; tiles before t - S were released by the consumers, so they have landed,
        // and so has tile t - S when the list ran out (its stage was released for the kEnd
        // tile, which re-armed that stage: its barrier must not be waited on again).  In a
        // normal run the remaining phases completed long ago and each wait returns at once.
        for (int u = max(0, t - S + (ended ? 1 : 0)); u < t; ++u) mbar_wait(&full[u % S], (u / S) & 1);
        return;
    }

    // ---------------------------------------------------------------------- consumer warps
    const int w = warp;
    const int r = lane >> 2, c = lane & 3;
    WarpState<D> st;
    ItemRows<D, G> cur, nxt;
    int nxt_item = -1;
    if (c0 < c1) {
        load_rows<D, G>(p, c0, w, nxt);
        nxt_item = c0;
    }
    int32_t rec[2] = {-1, -1};
    uint8_t *conv = smem + geo.conv + w * Gm::kConvBytes;
    for (int t = 0;; ++t) {
        const int s = t % S;
        if (!__all_sync(0xffffffffu, dwait<QUICK>(&full[s], (t / S) & 1, abort_flag, p.err, 0x33, p.wait))) return;
        const TileInfo ti = tinfo[s];
        if (ti.flags & kEnd) return;
        if (ti.flags & kFirst) {
            if (nxt_item == ti.item)
                cur = nxt;
            else
                load_rows<D, G>(p, ti.item, w, cur);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                rec[h] = cur.req[h] >= 0 ? __ldg(p.row_rec + cur.row_off + (r + 8 * h) / G) : -1;
                st.m[h] = -INFINITY;
                st.l[h] = 0.f;
            }
#pragma unroll
            for (int nd = 0; nd < D / 8; ++nd) st.acc[nd][0] = st.acc[nd][1] = st.acc[nd][2] = st.acc[nd][3] = 0.f;
            // fetch the next item's rows while this one runs
            nxt_item = ti.item + 1 < c1 ? ti.item + 1 : -1;
            if (nxt_item >= 0) load_rows<D, G>(p, nxt_item, w, nxt);
        }
        const uint8_t *stage = ring + s * geo.stage;
        if constexpr (FP8) {
            convert_head<D>(stage, geo, w * D, conv);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
            tile16<D>(st, cur.qf, conv, Gm::kConvK, conv + kBK * Gm::kConvK, Gm::kConvV, ti.kpos, ti.k1, p.scale_log2);
            __syncwarp();  // the conversion tiles are rewritten for the next tile
        } else {
            const int col = w * D * 2;
            tile16<D>(st, cur.qf, stage + col, geo.kstride, stage + geo.vbase + col, geo.vstride, ti.kpos, ti.k1,
                      p.scale_log2);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
        if (ti.flags & kLast) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                st.l[h] += __shfl_xor_sync(0xffffffffu, st.l[h], 1);
                st.l[h] += __shfl_xor_sync(0xffffffffu, st.l[h], 2);
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                if (cur.req[h] < 0) continue;
                const int head = (cur.g0 + w) * G + (r + 8 * h) % G;
                if (rec[h] < 0) {
                    const float inv = p.v_scale / st.l[h];
                    uint32_t *dst = reinterpret_cast<uint32_t *>(p.o + ((int64_t)cur.req[h] * p.hq + head) * D);
#pragma unroll
                    for (int nd = 0; nd < D / 8; ++nd)
                        dst[(nd * 8 + 2 * c) / 2] = pack_bf16x2(st.acc[nd][2 * h] * inv, st.acc[nd][2 * h + 1] * inv);
                } else {
                    const int64_t rb = (int64_t)rec[h] * p.hq + head;
                    float2 *dst = reinterpret_cast<float2 *>(p.rec_acc + rb * D);
#pragma unroll
                    for (int nd = 0; nd < D / 8; ++nd)
                        dst[(nd * 8 + 2 * c) / 2] =
                            make_float2(st.acc[nd][2 * h] * p.v_scale, st.acc[nd][2 * h + 1] * p.v_scale);
                    if (c == 0) *reinterpret_cast<float2 *>(p.rec_ml + rb * 2) = make_float2(st.m[h], st.l[h]);
                }
            }
        }
    }
}

// Combine partial states: o = sum_k 2^(m_k - M) acc_k / sum_k 2^(m_k - M) l_k.  One warp per
// (row, query head); each lane owns D / 32 consecutive elements.  One pass over the records,
// four at a time with all their loads in flight, rescaling the running sums when the
// maximum grows.
template <int D>
__global__ void __launch_bounds__(256) merge_kernel(const MergeItem *__restrict__ merges, const float *__restrict__ rec_acc,
                                                    const float *__restrict__ rec_ml, uint16_t *__restrict__ o, int hq) {
    // the merge list is plan data, complete before the call: read it while the kernel before
    // is still running, then wait for the records
    const MergeItem mi = merges[blockIdx.x];
    pdl_wait();  // every record of the call has been written
    pdl_trigger();
    const int h = blockIdx.y * 8 + (threadIdx.x >> 5);
    if (h >= hq) return;
    const int lane = threadIdx.x & 31;
    constexpr int V = D / 32, B = 4;
    float M = -INFINITY, L = 0.f, O[V];
#pragma unroll
    for (int v = 0; v < V; ++v) O[v] = 0.f;
    for (int k0 = 0; k0 < mi.nrec; k0 += B) {
        float2 ml[B];
        float a[B][V];
#pragma unroll
        for (int j = 0; j < B; ++j) {
            ml[j] = make_float2(-INFINITY, 0.f);
#pragma unroll
            for (int v = 0; v < V; ++v) a[j][v] = 0.f;
            if (k0 + j < mi.nrec) {
                const int64_t rb = (int64_t)(mi.rec0 + (k0 + j) * mi.rec_stride) * hq + h;
                ml[j] = __ldg(reinterpret_cast<const float2 *>(rec_ml + rb * 2));
                if constexpr (V == 4) {
                    const float4 x = __ldg(reinterpret_cast<const float4 *>(rec_acc + rb * D + lane * 4));
                    a[j][0] = x.x;
                    a[j][1] = x.y;
                    a[j][2] = x.z;
                    a[j][3] = x.w;
                } else {
                    const float2 x = __ldg(reinterpret_cast<const float2 *>(rec_acc + rb * D + lane * 2));
                    a[j][0] = x.x;
                    a[j][1] = x.y;
                }
            }
        }
        float mb = M;
#pragma unroll
        for (int j = 0; j < B; ++j) mb = fmaxf(mb, ml[j].x);
        if (mb == -INFINITY) continue;  // nothing seen yet (records of empty ranges)
        const float alpha = ex2(M - mb);  // 0 when M is -inf
        L *= alpha;
#pragma unroll
        for (int v = 0; v < V; ++v) O[v] *= alpha;
#pragma unroll
        for (int j = 0; j < B; ++j) {
            const float wt = ex2(ml[j].x - mb);  // 0 for padding entries
            L += ml[j].y * wt;
#pragma unroll
            for (int v = 0; v < V; ++v) O[v] += a[j][v] * wt;
        }
        M = mb;
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    uint32_t *dst = reinterpret_cast<uint32_t *>(o + ((int64_t)mi.out_row * hq + h) * D + lane * V);
#pragma unroll
    for (int v = 0; v < V; v += 2) dst[v / 2] = pack_bf16x2(O[v] * inv, O[v + 1] * inv);
}

template <int D, int G, bool FP8>
static int launch_decode(const DecodeParams &p, int nctas, cudaStream_t s) {
    const DGeo<D, FP8> geo(p.hg, p.joint != 0);
    auto kern = p.wait.quick ? decode_kernel<D, G, FP8, true> : decode_kernel<D, G, FP8, false>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, geo.bytes) != cudaSuccess)
        return PKV_E_CUDA;
    const int warps = p.hg + 1 + (p.late_wait ? 1 : 0);
    return launch_pdl(kern, dim3(nctas), dim3(32 * warps), geo.bytes, s, true, p) == cudaSuccess ? PKV_OK : PKV_E_CUDA;
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
    const dim3 grid((unsigned)info->num_merge, (unsigned)((info->num_q_heads + 7) / 8));
    const cudaError_t e = launch_pdl(info->head_dim == 128 ? merge_kernel<128> : merge_kernel<64>, grid, dim3(256), 0,
                                     s, true, m, rec_acc, rec_ml, o, (int)info->num_q_heads);
    return e == cudaSuccess ? PKV_OK : PKV_E_CUDA;
}

int check_call(const pkv_pool *pool, const pkv_batch *batch, const void *q, void *o, const pkv_plan_info *info,
               const void *plan_dev, void *workspace, size_t ws_bytes, int op) {
    int rc = validate_pool(pool);
    if (rc) return rc;
    if (!batch || !q || !o || !info || !plan_dev || !workspace) return PKV_E_INVALID;
    if (!batch->req_to_token || !batch->req_pool_indices || !batch->seq_lens) return PKV_E_INVALID;
    if (page_shift_of(batch) < 0) return PKV_E_INVALID;
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
    if (info->num_items == 0 && info->offsets[8] == 0) return PKV_OK;
    const int64_t nctas = info->offsets[SEC_NUM_CTAS], hg = info->offsets[SEC_HEAD_GROUP];
    if (nctas < 1 || (info->num_items > 0 && nctas > info->num_items) || (hg != 1 && hg != 2 && hg != 4 && hg != 8) ||
        pool->num_kv_heads % hg)
        return PKV_E_PLAN;
    const uint8_t *plan = static_cast<const uint8_t *>(plan_dev);
    DecodeParams p;
    p.k_pool = static_cast<const uint8_t *>(pool->k);
    p.v_pool = static_cast<const uint8_t *>(pool->v);
    p.num_slots = pool->num_slots;
    p.hkv = pool->num_kv_heads;
    p.hq = info->num_q_heads;
    p.hg = (int32_t)hg;
    p.req_to_token = batch->req_to_token;
    p.rt_stride = batch->stride;
    p.rt_rows = batch->num_rows;
    p.page_shift = page_shift_of(batch);
    p.batch = batch->batch;
    p.req_pool_indices = batch->req_pool_indices;
    p.seq_lens = batch->seq_lens;
    p.q = static_cast<const uint16_t *>(q);
    p.o = static_cast<uint16_t *>(o);
    const bool fp8 = pool->dtype == PKV_FP8_E4M3;
    p.scale_log2 = sm_scale * (fp8 ? pool->k_scale : 1.f) * kLog2e;
    p.v_scale = fp8 ? pool->v_scale : 1.f;
    p.items = reinterpret_cast<const DecodeItem *>(plan + info->offsets[SEC_ITEMS]);
    p.cta_off = reinterpret_cast<const int32_t *>(plan + info->offsets[SEC_CTA_OFF]);
    p.row_req = reinterpret_cast<const int32_t *>(plan + info->offsets[SEC_ROW_REQ]);
    p.row_rec = reinterpret_cast<const int32_t *>(plan + info->offsets[SEC_ROW_REC]);
    p.slot_bytes = slot_bytes(pool);
    p.joint = kv_interleaved(pool) && hg == pool->num_kv_heads ? 1 : 0;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    p.err = reinterpret_cast<int32_t *>(ws);
    p.wait = wait_policy(wait_limit_ns());
    p.rec_acc = reinterpret_cast<float *>(ws + kWorkspaceHeader);
    p.rec_ml = p.rec_acc + (size_t)info->num_records * info->num_q_heads * info->head_dim;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // The gather of the widely shared spans (and their members' query rows), the decode
    // kernel over everything else, the spans on the tensor cores, the merge.  The span pass
    // reads only what the gather wrote, so it takes SMs as decode CTAs finish instead of
    // waiting for the whole decode kernel, and its records are the freshest in L2 when the
    // merge reads them.
    rc = decode_span_gather(pool, batch, q, info, plan, ws, s);
    if (rc) return rc;
    // After a span gather the decode kernel streams from its start and one extra warp waits
    // for the gather, where that warp does not cost the kernel a CTA per SM (d = 128: 12 warps
    // of 168 registers fit an SM; at most 10 warps a CTA).
    const int per_sm = decode_ctas_per_sm((int32_t)hg, info->head_dim);
    p.late_wait = (info->offsets[8] > 0 && info->head_dim == 128 && hg + 2 <= 10 && per_sm * (hg + 2) <= 12) ? 1 : 0;
    if (info->num_items > 0) {
        const int G = info->num_q_heads / info->num_kv_heads;
        rc = info->head_dim == 128 ? dispatch_g<128>(G, fp8, p, (int)nctas, s)
                                   : dispatch_g<64>(G, fp8, p, (int)nctas, s);
        if (rc) return rc;
    }
    rc = decode_span_attend(pool, q, sm_scale, info, plan, ws, p.rec_acc, p.rec_ml, s, info->num_items > 0);
    if (rc) return rc;
    return launch_merge(info, plan_dev, p.rec_acc, p.rec_ml, p.o, s);
}
