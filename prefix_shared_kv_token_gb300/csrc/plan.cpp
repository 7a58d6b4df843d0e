// Host planner: turns one attention call (batch tables + optional shared-prefix cascade)
// into a flat list of work items for the kernels, the partial-state records they write and
// the merges that combine those records.
//
// Decode ([SG] summary §RadixAttention: each running request decodes over its whole cached
// context): work = (shared span chunk x up to 16/G member requests, or one request's
// unshared key chunk) x head group of <= 8 KV heads.  A span item reads the span's slots
// once for a group of its member requests (a radix-tree node on several paths: "Radix Tree
// 구조도" -- the two branches under [1,2,3] share its KV); a tail item reads one request's
// remaining positions.  Every (request, span chunk) and (request, tail chunk) owns one
// partial record (m, l, acc) unless the request has a single item, which then writes its
// output directly.  The kernel's CTAs are persistent: the planner deals the items to them
// longest first onto the least loaded CTA (LPT), and each CTA walks its own list.
//
// Extend (only the uncached remainder is prefilled, [SG] §RadixAttention): work = tile of
// up to 128/G query tokens x KV head over keys [k0, k1), causal within the request.  With a
// cascade, span items cover the contiguous query tokens of the span's members against the
// span (no mask needed: every query comes after the span) and the per-request items cover
// the rest of the context causally; one record per (query token, part), merged per token.

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <numeric>
#include <queue>
#include <utility>
#include <vector>

#include "../../include/pkv.h"

namespace {

struct DecodeItem { int32_t g0, mode, nreq, row_off, src, k0, k1, rot; };
constexpr int kMaxSegs = 4;
struct ExtendItem { int32_t g, tok0, ntok, qpos0, pos0, nseg, rec, flags, key0[kMaxSegs], nkeys[kMaxSegs]; };
// rows seeing fewer keys than this get bf16 high + low weights in the kernels (see common.cuh)
constexpr int32_t kPreciseKeys = 32;
struct GatherUnit { int32_t src, pos0, len, key0; };
struct MergeItem { int32_t out_row, rec0, nrec, rec_stride; };
// a packed extend item (flags & kItemPacked): up to four requests' last few tokens in one
// query tile, a 32-row group each, over shared segments (sgrp -1) and each one's own tail
constexpr int32_t kItemPacked = 4;
constexpr int32_t kPackSegs = 5;
struct PackInfo {
    int32_t key0[kPackSegs], nkeys[kPackSegs], spos[kPackSegs], sgrp[kPackSegs];
    int32_t tok0[4], ntok[4], qpos0[4];
};
static_assert(sizeof(DecodeItem) == 32 && sizeof(ExtendItem) == 64 && sizeof(MergeItem) == 16 &&
                  sizeof(PackInfo) == 128, "layout");

constexpr size_t kHeader = 256;
// decode: a shared span goes to the tensor-core path from this many member requests and keys
constexpr int32_t kTensorMinMembers = 12;
constexpr int32_t kTensorMinKeys = 256;
// decode: a batch whose contexts are all this short (and that has a CTA per request) gets one
// item per request and no merge
constexpr int32_t kFlatMaxLen = 128;
size_t align16(size_t x) { return (x + 15) & ~size_t(15); }

// Persistent CTAs: deal items longest-processing-time-first onto the least loaded of nctas
// CTAs (ties: lowest index); each CTA then runs its items in that (descending) order.
// Returns the items CTA-major and the CTA ranges cta_off[nctas + 1].
template <class T>
void lpt_deal(const std::vector<T> &items, const std::vector<int64_t> &cost, int32_t nctas, std::vector<T> *placed,
              std::vector<int32_t> *cta_off) {
    const int32_t n = (int32_t)items.size();
    std::vector<int32_t> order(n);
    std::iota(order.begin(), order.end(), 0);
    std::stable_sort(order.begin(), order.end(), [&](int32_t x, int32_t y) { return cost[x] > cost[y]; });
    std::vector<std::vector<int32_t>> per_cta(nctas);
    using Slot = std::pair<int64_t, int32_t>;  // (load, cta)
    std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> heap;
    for (int32_t b = 0; b < nctas; ++b) heap.push({0, b});
    for (int32_t x : order) {
        Slot sl = heap.top();
        heap.pop();
        per_cta[sl.second].push_back(x);
        sl.first += cost[x];
        heap.push(sl);
    }
    placed->clear();
    placed->reserve(items.size());
    cta_off->assign(1, 0);
    for (int32_t b = 0; b < nctas; ++b) {
        for (int32_t x : per_cta[b]) placed->push_back(items[x]);
        cta_off->push_back((int32_t)placed->size());
    }
}

// Extend-kernel item weight, in half key-tile steps of a two-query-tile item (6 per key tile):
// a two-tile item overlaps one tile's softmax with the other's MMAs; a one-tile item over
// several key tiles splits them between the two softmax warpgroups (about half the cost of
// a two-tile item); a one-tile item over one key tile runs serially.
int64_t extend_item_cost(const ExtendItem &x, int32_t tq, const std::vector<PackInfo> *packs = nullptr) {
    int64_t tiles = 0;
    const bool packed = (x.flags & kItemPacked) && packs;
    const int32_t *nk = packed ? (*packs)[(size_t)x.rec].nkeys : x.nkeys;
    for (int32_t i = 0; i < std::min(x.nseg, packed ? kPackSegs : kMaxSegs); ++i) tiles += (nk[i] + 127) / 128;
    const int64_t per = x.ntok > tq ? 6 : (tiles >= 2 ? 3 : 4);
    return tiles * per + 4;
}

// Keys per gather unit (one CTA each): up to 32, fewer when the gather is small, so that it
// still spreads over about 4 CTAs per SM.
int32_t gather_unit_keys(int64_t total_keys, int32_t num_sms) {
    const int64_t per = (total_keys + 4 * (int64_t)num_sms - 1) / (4 * (int64_t)num_sms);
    return (int32_t)std::min<int64_t>(32, std::max<int64_t>(4, per));
}

int check_heads(int32_t hq, int32_t hkv, int32_t d) {
    if (hq <= 0 || hkv <= 0 || hq % hkv) return PKV_E_INVALID;
    int32_t G = hq / hkv;
    if (G != 1 && G != 2 && G != 4 && G != 8) return PKV_E_UNSUPPORTED;
    if (d != 64 && d != 128) return PKV_E_UNSUPPORTED;
    return PKV_OK;
}

// Per-request ordered span lists from the cascade; fills tail_start.  Validates that the
// spans of every member tile [0, tail_start) in order and stay inside the context.
int spans_per_request(const pkv_cascade *c, int32_t batch, const int32_t *seq_lens,
                      std::vector<std::vector<int32_t>> *per_req, std::vector<int32_t> *tail_start) {
    per_req->assign((size_t)batch, {});
    tail_start->assign((size_t)batch, 0);
    if (!c || c->num_spans == 0) return PKV_OK;
    if (c->num_spans < 0 || !c->span_req || !c->span_start || !c->span_len || !c->grp_indptr || !c->grp_req)
        return PKV_E_INVALID;
    if (c->grp_indptr[0] != 0) return PKV_E_INVALID;
    for (int32_t s = 0; s < c->num_spans; ++s) {
        if (c->span_len[s] <= 0 || c->span_start[s] < 0) return PKV_E_INVALID;
        if (c->grp_indptr[s + 1] < c->grp_indptr[s]) return PKV_E_INVALID;
        if (c->span_req[s] < 0 || c->span_req[s] >= batch) return PKV_E_INVALID;
        bool src_is_member = false;
        for (int32_t i = c->grp_indptr[s]; i < c->grp_indptr[s + 1]; ++i) {
            int32_t r = c->grp_req[i];
            if (r < 0 || r >= batch) return PKV_E_INVALID;
            (*per_req)[r].push_back(s);
            src_is_member |= (r == c->span_req[s]);
        }
        if (!src_is_member) return PKV_E_INVALID;
    }
    for (int32_t r = 0; r < batch; ++r) {
        auto &v = (*per_req)[r];
        std::sort(v.begin(), v.end(), [&](int32_t a, int32_t b) { return c->span_start[a] < c->span_start[b]; });
        int32_t pos = 0;
        for (int32_t s : v) {
            if (c->span_start[s] != pos) return PKV_E_INVALID;
            pos += c->span_len[s];
        }
        if (pos > seq_lens[r]) return PKV_E_INVALID;
        (*tail_start)[r] = pos;
    }
    return PKV_OK;
}

template <class T>
void put(std::vector<uint8_t> &blob, size_t off, const std::vector<T> &v) {
    if (!v.empty()) std::memcpy(blob.data() + off, v.data(), v.size() * sizeof(T));
}

int emit(const std::vector<uint8_t> &blob, void *plan, size_t plan_cap, pkv_plan_info *info) {
    info->plan_bytes = blob.size();
    if (!plan) return PKV_OK;
    if (plan_cap < blob.size()) return PKV_E_WORKSPACE;
    std::memcpy(plan, blob.data(), blob.size());
    return PKV_OK;
}

}  // namespace

// Persistent decode CTAs per SM for a head group of hg KV heads: the kernel runs hg + 1
// warps with a 3-stage ring of 16-key tiles (bf16 layout, the larger one).  Registers are
// allocated per warp from each of the 4 sub-partitions' 16,384; the kernel is compiled for
// 168 registers a thread at d = 128 and 96 at d = 64.
int decode_ctas_per_sm(int32_t hg, int32_t d) {
    const int64_t warps = hg + 1;
    const int64_t smem = 256 + 3 * 16 * (4 * (int64_t)hg * d + 48) + 1024;
    const int64_t warps_per_sm = 4 * (16384 / (32 * (d == 128 ? 168 : 96)));
    int64_t n = std::min<int64_t>({232448 / smem, warps_per_sm / warps, 64 / warps, 8});
    return (int)std::max<int64_t>(n, 1);
}

extern "C" int pkv_plan_decode(int32_t batch, const int32_t *seq_lens, int32_t num_q_heads,
                               int32_t num_kv_heads, int32_t head_dim, const pkv_cascade *cascade,
                               const pkv_plan_opts *opts, void *plan, size_t plan_cap,
                               pkv_plan_info *info) {
    if (!info || batch < 0 || (batch > 0 && !seq_lens)) return PKV_E_INVALID;
    int rc = check_heads(num_q_heads, num_kv_heads, head_dim);
    if (rc) return rc;
    for (int32_t r = 0; r < batch; ++r)
        if (seq_lens[r] < 1) return PKV_E_INVALID;
    const int32_t G = num_q_heads / num_kv_heads;
    int32_t chunk = (opts && opts->chunk_keys > 0) ? opts->chunk_keys : 256;
    int32_t span_chunk = (opts && opts->span_chunk > 0) ? opts->span_chunk : 1024;
    const int32_t num_sms = (opts && opts->num_sms > 0) ? opts->num_sms : 152;
    const bool dyn_tail = opts && opts->dynamic_tail;
    const int32_t R = 16 / G;  // requests per span item: one 16-row MMA tile per KV head
    const int32_t TQ2 = 2 * (128 / G);  // requests per tensor-core span item (two 128-row tiles)
    // head group: KV heads read together per key (one contiguous pool row), <= 8
    int32_t hg = 8;
    while (num_kv_heads % hg) hg /= 2;

    std::vector<std::vector<int32_t>> spans_of;
    std::vector<int32_t> tail_start;
    rc = spans_per_request(cascade, batch, seq_lens, &spans_of, &tail_start);
    if (rc) return rc;

    // A tiny batch -- every context at most kFlatMaxLen keys, a CTA for every request -- is
    // bound by latency, not bytes: each request becomes one item over its whole context that
    // writes its output directly (no span items, no records, no merge launch), whatever the
    // cascade says.  Explicit chunk options keep the general plan.
    bool flat_plan = false;
    {
        int32_t max_len = 0;
        for (int32_t r = 0; r < batch; ++r) max_len = std::max(max_len, seq_lens[r]);
        flat_plan = !(opts && (opts->chunk_keys > 0 || opts->span_chunk > 0)) && batch <= num_sms &&
                    max_len <= kFlatMaxLen;
        if (flat_plan) {
            cascade = nullptr;
            spans_of.assign((size_t)batch, {});
            tail_start.assign((size_t)batch, 0);
            chunk = std::max<int32_t>(max_len, 1);
        }
    }

    // Shared spans with many member requests go to the tensor-core path: the span's keys
    // are gathered once into the workspace and attended as a dense block by 2 x 128/G of its
    // member requests per item (extend kernel), instead of re-reading the span per group of
    // 16/G requests.  Key chunks are sized for about one item per SM, at least 512 keys.
    const int32_t nspans = cascade ? cascade->num_spans : 0;
    std::vector<int32_t> sp_chunk(nspans, span_chunk);
    std::vector<char> sp_tensor(nspans, 0);
    std::vector<char> in_tensor(batch, 0);
    // The tensor-core span pass runs beside the decode kernel on span_sms SMs when it is small
    // next to it (opts->span_sms: 0 = decide here, < 0 = never, > 0 = that many SMs).  The
    // estimate, in SM-microseconds at the rates measured on GB300: a decode-kernel key moves
    // its head group's K and V rows at ~40 KB per us per SM; a tensor-core span item costs
    // ~2.3 us per 128-key tile for two 128-row query tiles, plus ~5 us to start.  Beside the
    // decode kernel the pass gets about 1.25x its share of the SMs, at least 12; it stays after
    // the decode kernel when its share is above a fifth.
    int32_t span_sms = (opts && opts->span_sms != 0) ? std::max(opts->span_sms, 0) : -1;
    if (span_sms < 0 && nspans > 0) {
        const double elem = 2.0;  // bytes of a pool element the decode kernel moves (bf16 rows)
        double dec = 0.0, spn = 0.0;
        for (int32_t r = 0; r < batch; ++r) dec += (double)(seq_lens[r] - tail_start[r]);
        for (int32_t s = 0; s < nspans; ++s) {
            const int32_t m = cascade->grp_indptr[s + 1] - cascade->grp_indptr[s], len = cascade->span_len[s];
            if (m >= kTensorMinMembers && len >= kTensorMinKeys)
                spn += (double)((m + TQ2 - 1) / TQ2) * num_kv_heads * (((len + 127) / 128) * 2.3 + 5.0);
            else
                dec += (double)len * ((m + R - 1) / R);
        }
        dec *= (double)num_kv_heads * head_dim * elem * 2.0 / 40000.0;  // SM-us
        const double share = spn / std::max(spn + dec, 1.0);
        span_sms = (spn > 0.0 && share <= 0.2) ? std::max<int32_t>(12, (int32_t)(1.25 * share * num_sms + 0.5)) : 0;
    }
    span_sms = std::min(std::max(span_sms, 0), num_sms - 1);
    for (int32_t s = 0; s < nspans; ++s) {
        const int32_t m = cascade->grp_indptr[s + 1] - cascade->grp_indptr[s], len = cascade->span_len[s];
        if (m < kTensorMinMembers || len < kTensorMinKeys) continue;
        sp_tensor[s] = 1;
        // Beside the decode kernel (span_sms option) the pass has few SMs and time to spare:
        // about two long items per SM there (fewer records, less set-up per key); else about
        // one item per SM.
        const int64_t per_chunk = (int64_t)((m + TQ2 - 1) / TQ2) * num_kv_heads;
        const int64_t want = span_sms > 0 ? (2 * (int64_t)span_sms + per_chunk / 2) / per_chunk
                                          : (num_sms + per_chunk - 1) / per_chunk;
        const int32_t nch = (int32_t)std::max<int64_t>(1, std::min<int64_t>(want, (len + 511) / 512));
        sp_chunk[s] = ((len + nch - 1) / nch + 127) / 128 * 128;
        for (int32_t i = cascade->grp_indptr[s]; i < cascade->grp_indptr[s + 1]; ++i) in_tensor[cascade->grp_req[i]] = 1;
    }

    // Requests whose whole context is shorter than kPreciseKeys keys leave the decode kernel:
    // each becomes one tensor-core item over its own gathered context with precise (bf16
    // high + low) weights, and takes no part in span items.
    std::vector<char> short_req(batch, 0);
    for (int32_t r = 0; r < batch; ++r)
        if (seq_lens[r] < kPreciseKeys) short_req[r] = in_tensor[r] = 1;

    // A small batch is cut finer (default chunk sizes only): the decode kernel's keys, span
    // re-reads included, are split into about two items per persistent CTA, at least 64
    // keys each.
    {
        int64_t work = 0;
        for (int32_t r = 0; r < batch; ++r)
            if (!short_req[r]) work += seq_lens[r] - tail_start[r];
        for (int32_t s = 0; s < nspans; ++s)
            if (!sp_tensor[s])
                work += (int64_t)cascade->span_len[s] *
                        ((cascade->grp_indptr[s + 1] - cascade->grp_indptr[s] + R - 1) / R);
        const int64_t target = 2 * (int64_t)num_sms * decode_ctas_per_sm(hg, head_dim) / (num_kv_heads / hg);
        const int32_t fine = (int32_t)std::max<int64_t>(64, ((work + target - 1) / std::max<int64_t>(target, 1) + 15) / 16 * 16);
        if (!(opts && opts->chunk_keys > 0) && !flat_plan) chunk = std::min(chunk, fine);
        if (!(opts && opts->span_chunk > 0))
            for (int32_t s = 0; s < nspans; ++s)
                if (!sp_tensor[s]) sp_chunk[s] = std::min(span_chunk, fine);
    }

    // records per request: its span chunks (in path order), then its tail chunks
    auto nchunks = [](int32_t len, int32_t c) { return len <= 0 ? 0 : (len + c - 1) / c; };
    std::vector<int32_t> nrec(batch, 0), rec_base(batch, 0);
    for (int32_t r = 0; r < batch; ++r) {
        int32_t n = 0;
        for (int32_t s : spans_of[r]) n += nchunks(cascade->span_len[s], sp_chunk[s]);
        n += nchunks(seq_lens[r] - tail_start[r], chunk);
        nrec[r] = short_req[r] ? 1 : n;
    }
    int32_t num_records = 0;
    for (int32_t r = 0; r < batch; ++r) {
        if (nrec[r] >= 2 || in_tensor[r]) {  // tensor-core items always write records
            rec_base[r] = num_records;
            num_records += nrec[r];
        } else {
            rec_base[r] = -1;  // single item: direct output
        }
    }
    // per-request running index into its own records
    std::vector<int32_t> next_rec(batch, 0);

    std::vector<DecodeItem> items;
    std::vector<int64_t> cost;  // load-balancing weight: 5 per key (a span's later member
                                // groups cost as much per key as its first: measured per-CTA
                                // times follow the tile count, not L2 reuse)
    std::vector<int32_t> row_req, row_rec;
    std::vector<MergeItem> merges;
    int32_t num_span_items = 0;
    constexpr int64_t kItemOverhead = 40;  // in fifths of a key

    // tensor-core span items (extend-kernel layout), their gathered keys and query rows
    std::vector<ExtendItem> xitems;
    std::vector<GatherUnit> units;
    std::vector<int32_t> qsrc, rec_list;
    int64_t nkeys = 0;

    if (cascade) {
        for (int32_t s = 0; s < cascade->num_spans; ++s) {
            const int32_t st = cascade->span_start[s], len = cascade->span_len[s];
            const int32_t m0 = cascade->grp_indptr[s], m1 = cascade->grp_indptr[s + 1];
            if (sp_tensor[s]) {
                const int32_t key0 = (int32_t)nkeys, q0 = (int32_t)qsrc.size();
                units.push_back({cascade->span_req[s], st, len, key0});  // split into units below
                nkeys += len;
                for (int32_t i = m0; i < m1; ++i) qsrc.push_back(cascade->grp_req[i]);
                for (int32_t c0 = 0; c0 < len; c0 += sp_chunk[s]) {
                    const int32_t c1 = std::min(len, c0 + sp_chunk[s]);
                    for (int32_t a = m0; a < m1; a += TQ2) {
                        const int32_t b = std::min(m1, a + TQ2);
                        const int32_t roff = (int32_t)rec_list.size();
                        for (int32_t i = a; i < b; ++i) {
                            const int32_t r = cascade->grp_req[i];
                            rec_list.push_back(rec_base[r] + next_rec[r]);
                            next_rec[r] += 1;
                        }
                        for (int32_t g = 0; g < num_kv_heads; ++g) {
                            ExtendItem it{};
                            it.g = g;
                            it.tok0 = q0 + (a - m0);
                            it.ntok = b - a;
                            it.qpos0 = 1 << 30;  // every query comes after the span: no mask
                            it.pos0 = st + c0;
                            it.nseg = 1;
                            it.rec = roff;
                            it.key0[0] = key0 + c0;
                            it.nkeys[0] = c1 - c0;
                            xitems.push_back(it);
                            ++num_span_items;
                        }
                    }
                }
                continue;
            }
            std::vector<int32_t> mem;  // members read through the decode kernel
            for (int32_t i = m0; i < m1; ++i)
                if (!short_req[cascade->grp_req[i]]) mem.push_back(cascade->grp_req[i]);
            const int32_t nm = (int32_t)mem.size();
            for (int32_t c0 = 0; c0 < len && nm > 0; c0 += sp_chunk[s]) {
                const int32_t c1 = std::min(len, c0 + sp_chunk[s]);
                for (int32_t a = 0; a < nm; a += R) {
                    const int32_t b = std::min(nm, a + R);
                    const int32_t off = (int32_t)row_req.size();
                    for (int32_t i = a; i < b; ++i) {
                        const int32_t r = mem[i];
                        row_req.push_back(r);
                        row_rec.push_back(rec_base[r] < 0 ? -1 : rec_base[r] + next_rec[r]);
                        next_rec[r] += 1;
                    }
                    // every member group reads the chunk from its first tile: groups of one
                    // chunk have equal cost, sit next to each other in the deal and run at
                    // about the same time, so all but the first find the chunk in L2.  (Start
                    // tiles staggered over the chunk made the reads of one tile too far apart
                    // in time: on the multi-turn workload the kernel read 1.23 GB from DRAM
                    // for 0.94 GB of unique K/V; in order it reads 0.95 GB.)
                    for (int32_t g0 = 0; g0 < num_kv_heads; g0 += hg) {
                        items.push_back({g0, 0, b - a, off, cascade->span_req[s], st + c0, st + c1, 0});
                        cost.push_back((int64_t)(c1 - c0) * 5 + kItemOverhead);
                        ++num_span_items;
                    }
                }
            }
        }
    }
    for (int32_t r = 0; r < batch; ++r) {
        const int32_t t0 = tail_start[r], L = seq_lens[r];
        for (int32_t k0 = t0; k0 < L && !short_req[r]; k0 += chunk) {
            const int32_t k1 = std::min(L, k0 + chunk);
            const int32_t off = (int32_t)row_req.size();
            row_req.push_back(r);
            row_rec.push_back(rec_base[r] < 0 ? -1 : rec_base[r] + next_rec[r]);
            next_rec[r] += 1;
            const bool last = k1 == L;
            for (int32_t g0 = 0; g0 < num_kv_heads; g0 += hg) {
                items.push_back({g0, 1, 1, off, r, k0, (last && dyn_tail) ? -1 : k1, 0});
                cost.push_back((int64_t)(k1 - k0) * 5 + kItemOverhead);
            }
        }
    }
    // short requests: one precise tensor-core item per KV head over the whole context
    std::vector<ExtendItem> xprecise;
    for (int32_t r = 0; r < batch; ++r) {
        if (!short_req[r]) continue;
        const int32_t L = seq_lens[r], key0 = (int32_t)nkeys, q0 = (int32_t)qsrc.size(), roff = (int32_t)rec_list.size();
        units.push_back({r, 0, L, key0});  // split into units below
        nkeys += L;
        qsrc.push_back(r);
        rec_list.push_back(rec_base[r]);
        next_rec[r] += 1;
        for (int32_t g = 0; g < num_kv_heads; ++g) {
            ExtendItem it{};
            it.g = g;
            it.tok0 = q0;
            it.ntok = 1;
            it.qpos0 = L - 1;
            it.pos0 = 0;
            it.nseg = 1;
            it.rec = roff;
            it.flags = 1;  // precise weights
            it.key0[0] = key0;
            it.nkeys[0] = L;
            xprecise.push_back(it);
        }
    }
    for (int32_t r = 0; r < batch; ++r)
        if (rec_base[r] >= 0) merges.push_back({r, rec_base[r], nrec[r], 1});

    // persistent CTAs: longest-processing-time-first onto the least loaded CTA
    const int32_t n_items = (int32_t)items.size();
    // SMs left to the tensor-core span pass, which then runs beside the decode kernel
    if (xitems.empty() || n_items == 0) span_sms = 0;
    const int32_t nctas = std::max<int32_t>(
        1, std::min<int64_t>(n_items, (int64_t)(num_sms - span_sms) * decode_ctas_per_sm(hg, head_dim)));
    std::vector<DecodeItem> placed;
    std::vector<int32_t> cta_off;
    lpt_deal(items, cost, nctas, &placed, &cta_off);
    if (n_items == 0) cta_off.push_back(0);

    if (nkeys >= ((int64_t)1 << 31)) return PKV_E_UNSUPPORTED;
    {
        const int32_t uk = gather_unit_keys(nkeys, num_sms);
        std::vector<GatherUnit> runs;
        runs.swap(units);
        for (const GatherUnit &R : runs)
            for (int32_t c = 0; c < R.len; c += uk) units.push_back({R.src, R.pos0 + c, std::min(uk, R.len - c), R.key0 + c});
    }
    // tensor-core items: the spans' list, then the short requests' (precise) list, back to
    // back, each dealt onto its own persistent CTAs
    std::vector<ExtendItem> xplaced, xplaced_p;
    std::vector<int32_t> xcta_off, xcta_off_p;
    auto xdeal = [&](const std::vector<ExtendItem> &v, std::vector<ExtendItem> *out, std::vector<int32_t> *off,
                     int32_t sms) {
        if (v.empty()) return 0;
        const int32_t n = std::max<int32_t>(1, std::min<int32_t>((int32_t)v.size(), sms));
        std::vector<int64_t> xcost;
        for (const ExtendItem &x : v) xcost.push_back(extend_item_cost(x, TQ2 / 2));
        lpt_deal(v, xcost, n, out, off);
        return n;
    };
    const int32_t xctas = xdeal(xitems, &xplaced, &xcta_off, span_sms > 0 ? span_sms : num_sms);
    const int32_t xctas_p = xdeal(xprecise, &xplaced_p, &xcta_off_p, num_sms);
    xplaced.insert(xplaced.end(), xplaced_p.begin(), xplaced_p.end());

    std::memset(info, 0, sizeof(*info));
    info->op = 1;
    info->batch = batch;
    info->num_q_heads = num_q_heads;
    info->num_kv_heads = num_kv_heads;
    info->head_dim = head_dim;
    info->num_items = n_items;
    info->num_span_items = num_span_items;
    info->num_records = num_records;
    info->num_merge = (int32_t)merges.size();
    info->total_q = batch;
    size_t off = 0;
    info->offsets[0] = (int64_t)off; off = align16(off + placed.size() * sizeof(DecodeItem));
    info->offsets[1] = (int64_t)off; off = align16(off + row_req.size() * sizeof(int32_t));
    info->offsets[2] = (int64_t)off; off = align16(off + row_rec.size() * sizeof(int32_t));
    info->offsets[3] = (int64_t)off; off = align16(off + merges.size() * sizeof(MergeItem));
    info->offsets[4] = (int64_t)off; off = align16(off + cta_off.size() * sizeof(int32_t));
    info->offsets[5] = nctas;
    info->offsets[6] = hg;
    info->offsets[7] = (int64_t)off; off = align16(off + xplaced.size() * sizeof(ExtendItem));
    info->offsets[8] = (int64_t)xplaced.size();
    info->offsets[9] = (int64_t)off; off = align16(off + units.size() * sizeof(GatherUnit));
    info->offsets[10] = (int64_t)units.size();
    info->offsets[11] = nkeys;
    info->offsets[12] = (int64_t)off; off = align16(off + qsrc.size() * sizeof(int32_t));
    info->offsets[13] = (int64_t)qsrc.size();
    info->offsets[14] = (int64_t)off; off = align16(off + rec_list.size() * sizeof(int32_t));
    info->offsets[16] = (int64_t)off; off = align16(off + xcta_off.size() * sizeof(int32_t));
    info->offsets[17] = xctas;
    info->offsets[18] = (int64_t)xplaced_p.size();
    info->offsets[19] = (int64_t)off; off = align16(off + xcta_off_p.size() * sizeof(int32_t));
    info->offsets[20] = xctas_p;
    std::vector<uint8_t> blob(std::max<size_t>(off, 16), 0);
    put(blob, (size_t)info->offsets[0], placed);
    put(blob, (size_t)info->offsets[1], row_req);
    put(blob, (size_t)info->offsets[2], row_rec);
    put(blob, (size_t)info->offsets[3], merges);
    put(blob, (size_t)info->offsets[4], cta_off);
    put(blob, (size_t)info->offsets[7], xplaced);
    put(blob, (size_t)info->offsets[16], xcta_off);
    put(blob, (size_t)info->offsets[19], xcta_off_p);
    put(blob, (size_t)info->offsets[9], units);
    put(blob, (size_t)info->offsets[12], qsrc);
    put(blob, (size_t)info->offsets[14], rec_list);
    // workspace: header | records (acc, ml) | gathered K | gathered V | gathered query rows
    auto align256 = [](size_t x) { return (x + 255) & ~size_t(255); };
    size_t ws = align256(kHeader + (size_t)num_records * num_q_heads * (head_dim + 2) * 4);
    info->offsets[15] = (int64_t)ws;
    ws += 2 * (size_t)nkeys * num_kv_heads * head_dim * 2;
    ws = align256(ws) + qsrc.size() * (size_t)num_q_heads * head_dim * 2;
    info->workspace_bytes = ws;
    return emit(blob, plan, plan_cap, info);
}

// Extend plans.  ctx_row0 == NULL: the call gathers its key runs (shared spans, each
// request's own positions) from the pool into the workspace.  ctx_row0 != NULL (context-
// buffer plans, chunked prefill): request r's context positions [0, seq_lens[r]) live in the
// caller's bf16 context arrays at rows ctx_row0[r] + position; earlier calls wrote the rows of
// its earlier positions, and this call writes the rows of its new tokens while it stores them
// into the pool, so nothing is gathered (no cascade).
static int plan_extend_impl(int32_t batch, const int32_t *seq_lens, const int32_t *extend_lens,
                            const int32_t *qo_indptr, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                            const pkv_cascade *cascade, const pkv_plan_opts *opts, const int32_t *ctx_row0,
                            int64_t ctx_rows, void *plan, size_t plan_cap, pkv_plan_info *info) {
    const int32_t num_sms = (opts && opts->num_sms > 0) ? opts->num_sms : 152;
    if (!info || batch < 0 || (batch > 0 && (!seq_lens || !extend_lens || !qo_indptr))) return PKV_E_INVALID;
    int rc = check_heads(num_q_heads, num_kv_heads, head_dim);
    if (rc) return rc;
    if (qo_indptr[0] != 0) return PKV_E_INVALID;
    for (int32_t r = 0; r < batch; ++r) {
        if (extend_lens[r] < 1 || extend_lens[r] > seq_lens[r]) return PKV_E_INVALID;
        if (qo_indptr[r + 1] - qo_indptr[r] != extend_lens[r]) return PKV_E_INVALID;
    }
    const bool ctx = ctx_row0 != nullptr;
    if (ctx) {
        if (cascade || ctx_rows <= 0 || ctx_rows >= ((int64_t)1 << 31)) return PKV_E_INVALID;
        // each request's rows inside the arrays, no two requests' rows overlapping
        std::vector<std::pair<int64_t, int64_t>> rows;
        for (int32_t r = 0; r < batch; ++r) {
            if (ctx_row0[r] < 0 || (int64_t)ctx_row0[r] + seq_lens[r] > ctx_rows) return PKV_E_INVALID;
            rows.push_back({ctx_row0[r], (int64_t)ctx_row0[r] + seq_lens[r]});
        }
        std::sort(rows.begin(), rows.end());
        for (size_t i = 1; i < rows.size(); ++i)
            if (rows[i].first < rows[i - 1].second) return PKV_E_INVALID;
    }
    const int32_t G = num_q_heads / num_kv_heads;
    const int32_t TQ2 = 2 * (128 / G);  // query tokens per item (two 128-row tiles)
    const int32_t total_q = qo_indptr[batch];

    std::vector<std::vector<int32_t>> spans_of;
    std::vector<int32_t> tail_start;
    rc = spans_per_request(cascade, batch, seq_lens, &spans_of, &tail_start);
    if (rc) return rc;
    // a span must lie inside the cached prefix of each member (queries come after it)
    for (int32_t r = 0; r < batch; ++r)
        if (tail_start[r] > seq_lens[r] - extend_lens[r]) return PKV_E_INVALID;

    // key runs, gathered once each into the workspace: every span, then every request's
    // remaining positions [tail_start, seq_len).  A request whose path has more shared
    // spans than an item holds segments gathers its whole context as one run instead.
    struct Run { int32_t src, pos0, len, key0; };
    std::vector<Run> runs;
    int64_t nkeys = 0;
    auto add_run = [&](int32_t src, int32_t pos0, int32_t len) {
        runs.push_back({src, pos0, len, (int32_t)nkeys});
        nkeys += len;
        return (int32_t)runs.size() - 1;
    };
    std::vector<int32_t> span_run;
    if (cascade)
        for (int32_t s = 0; s < cascade->num_spans; ++s)
            span_run.push_back(add_run(cascade->span_req[s], cascade->span_start[s], cascade->span_len[s]));
    if (ctx) nkeys = ctx_rows;  // keys are rows of the caller's context arrays
    // segments per request: (run, keys used), in context order.  The last shared span is cut
    // to a multiple of the 128-key tile and its remainder joins the request's own gathered
    // tail, so no key tile is spent on a few leftover span keys.
    struct Seg { int32_t run, len; };
    std::vector<std::vector<Seg>> segs_of(batch);
    // fused store (pkv_attn_extend_store): the call's store writes each new token's K/V to
    // the pool and straight to its gathered row, so the gather covers cached positions only
    const bool fuse = !ctx && opts && opts->fuse_store;
    for (int32_t r = 0; r < batch; ++r) {
        const int32_t ns = (int32_t)spans_of[r].size();
        if (ctx) {
            runs.push_back({r, 0, seq_lens[r], ctx_row0[r]});
            segs_of[r].push_back({(int32_t)runs.size() - 1, seq_lens[r]});
        } else if (ns + 1 <= kMaxSegs) {
            int32_t rem = 0;
            for (int32_t k = 0; k < ns; ++k) {
                const int32_t sp = spans_of[r][k];
                int32_t len = cascade->span_len[sp];
                if (k == ns - 1) {
                    rem = len % 128;
                    len -= rem;
                }
                if (len > 0) segs_of[r].push_back({span_run[sp], len});
            }
            const int32_t t0 = tail_start[r] - rem;
            segs_of[r].push_back({add_run(r, t0, seq_lens[r] - t0), seq_lens[r] - t0});
        } else {
            segs_of[r].push_back({add_run(r, 0, seq_lens[r]), seq_lens[r]});
        }
    }
    if (nkeys >= ((int64_t)1 << 31)) return PKV_E_UNSUPPORTED;
    std::vector<GatherUnit> units;
    const int32_t uk = gather_unit_keys(nkeys, num_sms);
    // each request's own run (its last segment) holds its new positions [seq - ext, seq)
    std::vector<int32_t> own_run_of(runs.size(), -1);
    for (int32_t r = 0; r < batch; ++r) own_run_of[(size_t)segs_of[r].back().run] = r;
    if (!ctx)
        for (size_t j = 0; j < runs.size(); ++j) {
            const Run &R = runs[j];
            const int32_t r = own_run_of[j];
            const int32_t len = (fuse && r >= 0) ? seq_lens[r] - extend_lens[r] - R.pos0 : R.len;
            for (int32_t c = 0; c < len; c += uk) units.push_back({R.src, R.pos0 + c, std::min(uk, len - c), R.key0 + c});
        }
    // the row of every new token (in q order) that the store writes: in the caller's context
    // arrays (context-buffer plans) or among the gathered rows (fused-store plans)
    std::vector<int32_t> tok_row;
    if (ctx || fuse)
        for (int32_t r = 0; r < batch; ++r) {
            const Run &R = runs[(size_t)segs_of[r].back().run];
            for (int32_t i = 0; i < extend_lens[r]; ++i)
                tok_row.push_back(R.key0 + seq_lens[r] - extend_lens[r] + i - R.pos0);
        }

    // items: up to 2 x 128/G query tokens of one request x one KV head, over its segments;
    // the last segment is cut at the last query token's position (causal)
    std::vector<ExtendItem> items;
    std::vector<MergeItem> merges;
    int32_t num_span_items = 0;
    // A request's last few tokens (at most one 32-row group: 32/G tokens) after shared spans
    // are set aside: such chunks with the same shared spans share one query tile, a row
    // group each, over those spans plus each one's own tail (a packed item).
    const int32_t RG = 32 / G;  // tokens per 32-row group
    std::vector<ExtendItem> leftovers;
    for (int32_t r = 0; r < batch; ++r) {
        const int32_t e = extend_lens[r], p = seq_lens[r] - e;
        const auto &sg = segs_of[r];
        for (int32_t i0 = 0; i0 < e; i0 += TQ2) {
            const int32_t n = std::min(TQ2, e - i0);
            ExtendItem it{};
            it.tok0 = qo_indptr[r] + i0;
            it.ntok = n;
            it.qpos0 = p + i0;
            it.flags = p + i0 + 1 < kPreciseKeys ? 1 : 0;  // its first row sees p + i0 + 1 keys
            it.pos0 = runs[sg[0].run].pos0;
            it.nseg = (int32_t)sg.size();
            it.rec = -1;
            int32_t end = p + i0 + n;  // one past the last visible position
            for (size_t k = 0; k < sg.size(); ++k) {
                const Run &R = runs[sg[k].run];
                it.key0[k] = R.key0;
                it.nkeys[k] = k + 1 == sg.size() ? end - R.pos0 : sg[k].len;
            }
            if (it.nseg > 1) ++num_span_items;
            if (n <= RG && it.nseg > 1 && !(it.flags & 1)) {
                leftovers.push_back(it);
                continue;
            }
            for (int32_t g = 0; g < num_kv_heads; ++g) {
                it.g = g;
                items.push_back(it);
            }
        }
    }
    // pack the set-aside chunks: same shared segments (runs, lengths, start), up to 4 groups
    // and kPackSegs segments per tile; a chunk left alone is an ordinary item
    std::vector<PackInfo> packs;
    {
        auto same_shared = [](const ExtendItem &a, const ExtendItem &b) {
            if (a.nseg != b.nseg || a.pos0 != b.pos0) return false;
            for (int32_t k = 0; k + 1 < a.nseg; ++k)
                if (a.key0[k] != b.key0[k] || a.nkeys[k] != b.nkeys[k]) return false;
            return true;
        };
        std::vector<char> used(leftovers.size(), 0);
        for (size_t a = 0; a < leftovers.size(); ++a) {
            if (used[a]) continue;
            const ExtendItem &lead = leftovers[a];
            const int32_t nshared = lead.nseg - 1;
            const int32_t cap = std::min<int32_t>(4, kPackSegs - nshared);
            std::vector<size_t> grp{a};
            used[a] = 1;
            for (size_t b = a + 1; b < leftovers.size() && (int32_t)grp.size() < cap; ++b)
                if (!used[b] && same_shared(lead, leftovers[b])) {
                    grp.push_back(b);
                    used[b] = 1;
                }
            if (grp.size() == 1) {
                ExtendItem it = lead;
                for (int32_t g = 0; g < num_kv_heads; ++g) {
                    it.g = g;
                    items.push_back(it);
                }
                continue;
            }
            PackInfo pk{};
            int32_t pos = lead.pos0;
            for (int32_t k = 0; k < nshared; ++k) {
                pk.key0[k] = lead.key0[k];
                pk.nkeys[k] = lead.nkeys[k];
                pk.spos[k] = pos;
                pk.sgrp[k] = -1;
                pos += lead.nkeys[k];
            }
            for (size_t m = 0; m < grp.size(); ++m) {
                const ExtendItem &x = leftovers[grp[m]];
                const int32_t k = nshared + (int32_t)m;
                pk.key0[k] = x.key0[x.nseg - 1];
                pk.nkeys[k] = x.nkeys[x.nseg - 1];
                pk.spos[k] = pos;  // every member's own tail starts right after the shared part
                pk.sgrp[k] = (int32_t)m;
                pk.tok0[m] = x.tok0;
                pk.ntok[m] = x.ntok;
                pk.qpos0[m] = x.qpos0;
            }
            ExtendItem it{};
            it.tok0 = lead.tok0;
            it.ntok = TQ2 / 2;  // one query tile
            it.qpos0 = lead.qpos0;
            it.pos0 = lead.pos0;
            it.nseg = nshared + (int32_t)grp.size();
            it.rec = (int32_t)packs.size();
            it.flags = kItemPacked;
            for (int32_t k = 0; k < std::min(it.nseg, kMaxSegs); ++k) {
                it.key0[k] = pk.key0[k];
                it.nkeys[k] = pk.nkeys[k];
            }
            packs.push_back(pk);
            for (int32_t g = 0; g < num_kv_heads; ++g) {
                it.g = g;
                items.push_back(it);
            }
        }
    }
    // two lists, each dealt onto its own persistent CTAs: the common items, then the items
    // holding rows that see few keys (a separate launch with precise weights); stored back to
    // back, so items [0, num_items) cover both
    std::vector<ExtendItem> placed, placed_x;
    std::vector<int32_t> cta_off, cta_off_x;
    int32_t nctas = 1, nctas_x = 0;
    {
        std::vector<ExtendItem> common, precise;
        for (const ExtendItem &x : items) (x.flags & 1 ? precise : common).push_back(x);
        auto deal = [&](const std::vector<ExtendItem> &v, std::vector<ExtendItem> *out, std::vector<int32_t> *off) {
            const int32_t n = std::max<int32_t>(1, std::min<int32_t>((int32_t)v.size(), num_sms));
            std::vector<int64_t> cost;
            for (const ExtendItem &x : v) cost.push_back(extend_item_cost(x, TQ2 / 2, &packs));
            lpt_deal(v, cost, n, out, off);
            return n;
        };
        nctas = deal(common, &placed, &cta_off);
        if (!precise.empty()) nctas_x = deal(precise, &placed_x, &cta_off_x);
    }
    const int32_t n_main = (int32_t)placed.size();
    placed.insert(placed.end(), placed_x.begin(), placed_x.end());
    const bool cascaded = false;
    const int32_t kmax = 1;

    std::memset(info, 0, sizeof(*info));
    info->op = 2;
    info->batch = batch;
    info->num_q_heads = num_q_heads;
    info->num_kv_heads = num_kv_heads;
    info->head_dim = head_dim;
    info->num_items = (int32_t)items.size();
    info->num_span_items = num_span_items;
    info->num_records = cascaded ? kmax * total_q : 0;
    info->num_merge = (int32_t)merges.size();
    info->total_q = total_q;
    size_t off = 0;
    info->offsets[0] = (int64_t)off; off = align16(off + placed.size() * sizeof(ExtendItem));
    info->offsets[3] = (int64_t)off; off = align16(off + merges.size() * sizeof(MergeItem));
    info->offsets[4] = (int64_t)off; off = align16(off + units.size() * sizeof(GatherUnit));
    info->offsets[5] = (int64_t)units.size();
    info->offsets[6] = nkeys;
    info->offsets[7] = (int64_t)off; off = align16(off + cta_off.size() * sizeof(int32_t));
    info->offsets[8] = nctas;
    info->offsets[9] = info->offsets[0] + (int64_t)n_main * (int64_t)sizeof(ExtendItem);
    info->offsets[10] = (int64_t)placed_x.size();
    info->offsets[11] = (int64_t)off; off = align16(off + cta_off_x.size() * sizeof(int32_t));
    info->offsets[12] = nctas_x;
    info->offsets[13] = (int64_t)off; off = align16(off + packs.size() * sizeof(PackInfo));
    info->offsets[14] = (int64_t)packs.size();
    info->offsets[15] = (int64_t)off; off = align16(off + tok_row.size() * sizeof(int32_t));
    info->offsets[16] = ctx ? 1 : (fuse ? 2 : 0);
    std::vector<uint8_t> blob(std::max<size_t>(off, 16), 0);
    put(blob, (size_t)info->offsets[0], placed);
    put(blob, (size_t)info->offsets[13], packs);
    put(blob, (size_t)info->offsets[7], cta_off);
    put(blob, (size_t)info->offsets[11], cta_off_x);
    put(blob, (size_t)info->offsets[3], merges);
    put(blob, (size_t)info->offsets[4], units);
    put(blob, (size_t)info->offsets[15], tok_row);
    const size_t rec_bytes = (size_t)info->num_records * num_q_heads * (head_dim + 2) * 4;
    info->workspace_bytes = kHeader + ((rec_bytes + 255) & ~size_t(255)) +
                            (ctx ? 0 : 2 * (size_t)nkeys * num_kv_heads * head_dim * 2);
    return emit(blob, plan, plan_cap, info);
}

extern "C" int pkv_plan_extend(int32_t batch, const int32_t *seq_lens, const int32_t *extend_lens,
                               const int32_t *qo_indptr, int32_t num_q_heads, int32_t num_kv_heads,
                               int32_t head_dim, const pkv_cascade *cascade, const pkv_plan_opts *opts,
                               void *plan, size_t plan_cap, pkv_plan_info *info) {
    return plan_extend_impl(batch, seq_lens, extend_lens, qo_indptr, num_q_heads, num_kv_heads, head_dim, cascade,
                            opts, nullptr, 0, plan, plan_cap, info);
}

extern "C" int pkv_plan_extend_ctx(int32_t batch, const int32_t *seq_lens, const int32_t *extend_lens,
                                   const int32_t *qo_indptr, const int32_t *ctx_row0, int64_t ctx_rows,
                                   int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                   const pkv_plan_opts *opts, void *plan, size_t plan_cap, pkv_plan_info *info) {
    if (!ctx_row0 && batch > 0) return PKV_E_INVALID;
    static const int32_t none = 0;
    return plan_extend_impl(batch, seq_lens, extend_lens, qo_indptr, num_q_heads, num_kv_heads, head_dim, nullptr,
                            opts, ctx_row0 ? ctx_row0 : &none, ctx_rows, plan, plan_cap, info);
}
