/*
 * pkv.h -- C ABI of the prefix-shared, token-indexed KV attention library (libpkv.so).
 *
 * One KV pool indexed per token: K_pool[num_slots][num_kv_heads][head_dim] and the same for
 * V.  A host-side radix tree of token prefixes maps each cached token to its pool slot, so
 * requests that share a prefix share its slots.  Sources for what each call computes:
 *
 *   [RC]  "[SGLang] RadixAttention: Radix Tree 기반 프리픽스 캐싱의 핵심"
 *         (blog.secrett2633.cloud/opensource/sglang/radix-cache) -- sections
 *         "Radix Tree 구조도", "핵심 자료구조: TreeNode", "프리픽스 매칭", "노드 분할",
 *         "삽입", "Eviction 전략", "참조 카운트: lock_ref".
 *   [SG]  "Efficiently Programming Large Language Models using SGLang" (summary,
 *         0h-n0.github.io/posts/paper-2312-07910) -- §RadixAttention (match length,
 *         "only the remainder is prefilled"), §LRU Evictionポリシー.
 *   [PR]  "SGLang: Treating LLM Interactions as Programs for High-Throughput Inference"
 *         (codethepapers.com) -- §Key Algorithmic Steps (prefix reuse, forked branches
 *         sharing the prefix cache), §Why this matters in production.
 *   [RT]  "SGLang后端运行时优化细节" (highthink.cn) -- §显存分级管理机制, the fp8_e4m3 KV
 *         cache dtype.
 *
 * Conventions for every function below
 *   - Returns PKV_OK (0) or a negative PKV_E_* code; pkv_strerror() names it.
 *   - "device" pointers are CUDA device memory owned by the caller; "host" pointers are
 *     ordinary host memory owned by the caller.  The library allocates no device memory and
 *     never synchronises a stream, except pkv_get_device_error() and
 *     pkv_get_noalloc_device_error(), which synchronise.
 *   - Device calls are asynchronous on the given stream (a cudaStream_t passed as void*;
 *     NULL is the legacy default stream).  Argument errors are reported before anything is
 *     enqueued; launch errors come back as PKV_E_CUDA.
 *   - bf16 is IEEE bfloat16 (raw 16-bit patterns); e4m3 is OCP FP8 E4M3 (bias 7, max 448).
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------------------------------ */
/* status                                                                                */

#define PKV_OK             0
#define PKV_E_INVALID     -1  /* null pointer, negative size, inconsistent arguments      */
#define PKV_E_UNSUPPORTED -2  /* head_dim / group size / dtype combination not built       */
#define PKV_E_WORKSPACE   -3  /* workspace or plan buffer too small                        */
#define PKV_E_CUDA        -4  /* a CUDA runtime call or kernel launch failed               */
#define PKV_E_NOSPACE     -5  /* allocator: fewer free slots than requested                */
#define PKV_E_NOTFOUND    -6  /* tree: unknown node id                                     */
#define PKV_E_DEVICE      -7  /* a kernel recorded an error in the workspace error word    */
#define PKV_E_PLAN        -8  /* plan blob does not match the call                         */

/* values a kernel may leave in the workspace error word (first error wins) */
#define PKV_DERR_SLOT_RANGE 0x100  /* a slot read from a table was outside [0, num_slots)     */
#define PKV_DERR_TIMEOUT    0x200  /* a bounded wait inside a kernel gave up (low byte: which) */
#define PKV_DERR_POSITION   0x400  /* a work item addressed positions outside its row         */

const char *pkv_strerror(int code);
int pkv_version(void);  /* major*10000 + minor*100 + patch */

/* ------------------------------------------------------------------------------------ */
/* the KV pool                                                                          */

typedef enum { PKV_BF16 = 0, PKV_FP8_E4M3 = 1 } pkv_dtype;

typedef struct pkv_pool {
    void   *k;             /* device, slot s's K row of [num_kv_heads][head_dim] elements at */
                           /* element s * slot_stride                                       */
    void   *v;             /* device, the same for V; bf16 (2 B) or e4m3 (1 B) elements     */
    int64_t num_slots;     /* num_slots * num_kv_heads must be < 2^31                     */
    int32_t num_kv_heads;
    int32_t head_dim;      /* 64 or 128                                                   */
    int32_t dtype;         /* pkv_dtype                                                   */
    float   k_scale;       /* fp8 only: stored code = e4m3(x / k_scale), value = code*k_scale */
    float   v_scale;
    /* Elements from one slot's row to the next, in k and in v; 0 means num_kv_heads *
     * head_dim (two dense arrays).  2 * num_kv_heads * head_dim with v = k + num_kv_heads *
     * head_dim is the interleaved layout [num_slots][K row | V row]: a slot's K and V are one
     * contiguous run, which decode reads with a single copy per key.  The stride in bytes
     * must be a multiple of 16. */
    int64_t slot_stride;
} pkv_pool;

/* ------------------------------------------------------------------------------------ */
/* kv_store: write the K/V rows of newly computed tokens into their pool slots.          */
/*                                                                                      */
/* Pool values are per-token KV indices held by the radix tree ([RC] "Radix Tree 구조도",  */
/* TreeNode.value); tokens not yet cached get fresh slots (out_cache_loc) from the       */
/* allocator and their K/V are written there before attention reads them ([PR] "compute  */
/* missing KV tensors -> insert node").                                                  */
/*   k_new, v_new   device, bf16 [n][num_kv_heads][head_dim], row-major                   */
/*   out_cache_loc  device, int32 [n]; slot of token i; entries must be distinct and in   */
/*                  [0, num_slots) (a duplicate makes the result of that slot undefined;  */
/*                  pkv_check_out_cache_loc below detects it on the host)                 */
/*   workspace      device error word (4 bytes, 4-aligned) or NULL; a slot outside         */
/*                  [0, num_slots) is never written and sets PKV_DERR_SLOT_RANGE there     */
/* bf16 pool: bit-exact copy.  fp8 pool: e4m3_rn_satfinite(float(x) / scale) per element  */
/* (IEEE fp32 division).  n == 0 is a no-op.                                              */
int pkv_kv_store(const pkv_pool *pool, const void *k_new, const void *v_new,
                 const int32_t *out_cache_loc, int64_t n, void *workspace, void *stream);

/* Host check of kv_store's precondition (opt-in: the allocator hands out distinct slots, so a
 * caller runs this only on its checked path).  New tokens get slots from the allocator's free
 * list ([RC] "Eviction 전략": evicted slots go back through token_to_kv_pool_allocator.free),
 * so within one call no two tokens may name the same slot.
 *   out_cache_loc  host int32 [n]
 *   bad            host, may be NULL: index of the first entry that is out of [0, num_slots)
 *                  or repeats an earlier entry's slot; -1 when there is none
 * PKV_OK when every entry is in range and distinct, else PKV_E_INVALID.  Nothing is enqueued. */
int pkv_check_out_cache_loc(const int32_t *out_cache_loc, int64_t n, int64_t num_slots, int64_t *bad);

/* ------------------------------------------------------------------------------------ */
/* batch tables consumed by the attention calls (all device memory)                     */

typedef struct pkv_batch {
    const int32_t *req_to_token;      /* [num_rows][stride]: slot of each context position, */
                                      /* or with page_size > 1 the page of each block       */
    int64_t        stride;            /* entries per row: >= longest context (in blocks)    */
    int32_t        num_rows;
    const int32_t *req_pool_indices;  /* [batch]: row of request r in req_to_token          */
    const int32_t *seq_lens;          /* [batch]: context length of r, new tokens included  */
    int32_t        batch;
    /* 0 or 1: a token table (above).  P > 1, a power of two <= 4096: a paged pool whose page
     * k holds slots [k P, k P + P); req_to_token[row][b] is the page of positions
     * [b P, b P + P), so position t reads slot req_to_token[row][t / P] * P + t % P ([SG]
     * §Technical Details: the KV is referred to by 16-token block).  Any other value:
     * PKV_E_INVALID.  A page whose slots fall outside the pool reads as zero K/V rows and
     * sets PKV_DERR_SLOT_RANGE. */
    int32_t        page_size;
} pkv_batch;

/* A shared-prefix cascade, in host memory.  Span s is a run of positions
 * [span_start[s], span_start[s] + span_len[s]) whose slots are identical in the rows of all
 * its member requests grp_req[grp_indptr[s] .. grp_indptr[s+1]) (a radix-tree node, or a
 * chain of nodes, on the path of >= 2 requests of the batch: [RC] "Radix Tree 구조도" -- the
 * two branches under [1,2,3] share its KV).  span_req[s] is one member whose row is read.
 * For every request the spans it belongs to must tile [0, t) for some t, in order; the
 * attention kernels read each span once per group and merge partial softmax states.
 * pkv_tree_cascade() produces this description from the tree.                             */
typedef struct pkv_cascade {
    int32_t        num_spans;
    const int32_t *span_req;
    const int32_t *span_start;
    const int32_t *span_len;
    const int32_t *grp_indptr;        /* [num_spans + 1] */
    const int32_t *grp_req;           /* batch indices   */
} pkv_cascade;

/* Planner knobs (NULL = defaults). */
typedef struct pkv_plan_opts {
    int32_t chunk_keys;    /* decode: keys per unshared work item (0 = 256, cut finer for a */
                           /* small batch so each persistent CTA gets about two items)      */
    int32_t span_chunk;    /* decode: keys per shared-span work item (0 = 1024, cut finer   */
                           /* the same way; tensor-core spans are sized for ~one item per SM) */
    int32_t num_sms;       /* SMs of the target GPU for load balancing (0 = 152)             */
    int32_t dynamic_tail;  /* decode: last item of each request reads its end from seq_lens  */
                           /* on the device, so the plan stays valid while tails grow by     */
                           /* whole decode steps inside the same chunk                        */
    int32_t span_sms;      /* decode: SMs left to the tensor-core pass over widely shared     */
                           /* spans, which then runs beside the decode kernel (whose CTAs     */
                           /* take the other SMs); 0 = decided by the planner, < 0 = the pass */
                           /* always runs after the decode kernel                             */
    int32_t fuse_store;    /* extend: a plan for pkv_attn_extend_store, which stores the new  */
                           /* tokens itself (pool and gathered rows in one pass)              */
} pkv_plan_opts;

/* Host description of a plan; pass it, with a device copy of the plan blob, to the device
 * call.  Filled by pkv_plan_decode / pkv_plan_extend. */
typedef struct pkv_plan_info {
    int32_t op;                /* 1 = decode, 2 = extend                                   */
    int32_t batch;
    int32_t num_q_heads, num_kv_heads, head_dim;
    int32_t num_items;         /* attention work items                                      */
    int32_t num_span_items;    /* of which read a shared span (cascade)                     */
    int32_t num_records;       /* partial (m, l, acc) records written for merging            */
    int32_t num_merge;         /* requests (decode) or query tokens (extend) to merge        */
    int32_t total_q;           /* query tokens in the call                                  */
    size_t  plan_bytes;        /* size of the plan blob                                     */
    size_t  workspace_bytes;   /* device workspace the call needs (>= 256)                  */
    int64_t offsets[24];       /* byte offsets and counts of the blob's sections (internal) */
} pkv_plan_info;

/* Decode plan: one query token per request, at position seq_lens[r] - 1, attending to the
 * whole context [0, seq_lens[r]) including its own just-stored token.  Work is split over
 * (request or shared span) x KV head x key chunk (split-KV); partial states are merged.
 *   seq_lens  host int32 [batch], each >= 1
 *   cascade   host, may be NULL (every request reads its whole row)
 *   plan      host buffer of plan_cap bytes, or NULL to only size the plan in *info        */
int pkv_plan_decode(int32_t batch, const int32_t *seq_lens, int32_t num_q_heads,
                    int32_t num_kv_heads, int32_t head_dim, const pkv_cascade *cascade,
                    const pkv_plan_opts *opts, void *plan, size_t plan_cap,
                    pkv_plan_info *info);

/* Extend plan: request r queries its extend_lens[r] new tokens at positions
 * seq_lens[r] - extend_lens[r] + i; query token i attends causally to positions
 * [0, seq_lens[r] - extend_lens[r] + i] -- the matched prefix plus its own suffix ([SG]
 * §RadixAttention: only the unmatched remainder is prefilled).
 *   seq_lens, extend_lens  host int32 [batch], 1 <= extend_lens[r] <= seq_lens[r]
 *   qo_indptr              host int32 [batch + 1]: query tokens of r are rows
 *                          qo_indptr[r] .. qo_indptr[r+1]-1 of q and o
 *   cascade                host, may be NULL                                            */
int pkv_plan_extend(int32_t batch, const int32_t *seq_lens, const int32_t *extend_lens,
                    const int32_t *qo_indptr, int32_t num_q_heads, int32_t num_kv_heads,
                    int32_t head_dim, const pkv_cascade *cascade, const pkv_plan_opts *opts,
                    void *plan, size_t plan_cap, pkv_plan_info *info);

/* Attention over the pool, read through req_to_token (see the two plan calls for the
 * positions each query sees).  Head h uses KV head h / (num_q_heads / num_kv_heads).
 *   q          device, bf16 [total_q][num_q_heads][head_dim]
 *   o          device, bf16 [total_q][num_q_heads][head_dim], fully overwritten
 *   sm_scale   logit scale, usually 1/sqrt(head_dim)
 *   info       host, from the matching pkv_plan_* call
 *   plan_dev   device copy of the plan blob (info->plan_bytes bytes, 16-byte aligned)
 *   workspace  device, >= info->workspace_bytes, 256-byte aligned; its first 4 bytes are
 *              the error word (zero it once; kernels only ever set it)
 * Accumulation is fp32; softmax probabilities enter the P*V product as bf16.  For an fp8
 * pool the codes are converted exactly to bf16 and the scales are applied in fp32.     */
int pkv_attn_decode(const pkv_pool *pool, const pkv_batch *batch, const void *q, void *o,
                    float sm_scale, const pkv_plan_info *info, const void *plan_dev,
                    void *workspace, size_t ws_bytes, void *stream);

int pkv_attn_extend(const pkv_pool *pool, const pkv_batch *batch, const void *q, void *o,
                    float sm_scale, const pkv_plan_info *info, const void *plan_dev,
                    void *workspace, size_t ws_bytes, void *stream);

/* Store + extend in one call (a plan from pkv_plan_extend with opts->fuse_store set): the new
 * tokens' K/V go into the pool exactly as pkv_kv_store writes them and, as the pool now holds
 * them, straight into the call's gathered rows, so the key gather reads only cached
 * positions -- the rows just stored are not read back from the pool ([PR] "compute missing
 * KV tensors -> insert node": the missing K/V are computed once and reused).
 *   k_new, v_new, out_cache_loc  the new tokens' rows and slots in q order (total_q rows),
 *                                as pkv_kv_store takes them
 * Everything else as pkv_attn_extend; slot-range errors of the store go to the workspace
 * error word, and so does a context row outside the plan's gathered rows (PKV_DERR_POSITION,
 * header words 1-2 = the token and the row; that copy is skipped).  pkv_attn_extend rejects
 * a fused-store plan and this call any other. */
int pkv_attn_extend_store(const pkv_pool *pool, const pkv_batch *batch, const void *q, void *o, float sm_scale,
                          const void *k_new, const void *v_new, const int32_t *out_cache_loc,
                          const pkv_plan_info *info, const void *plan_dev, void *workspace, size_t ws_bytes,
                          void *stream);

/* Chunked prefill over a context buffer kept by the caller ("SGLang后端运行时优化细节",
 * §RadixAttention KV缓存复用的底层逻辑, 3 开发者需关注的配置项: --chunked-prefill-size prefills a
 * long prompt a chunk at a time, each chunk over the chunks cached before it).  The caller
 * keeps, for every request being prefilled this way, a run of rows in two device arrays
 * ctx_k, ctx_v of bf16 [ctx_rows][num_kv_heads][head_dim]: context position t of request r
 * lives at row ctx_row0[r] + t.  Each chunk's call stores its new tokens' K/V into the pool
 * (exactly as pkv_kv_store) and, in the same pass, into their context rows as the pool now
 * holds them (bf16 bits; for an fp8 pool the stored code converted exactly to bf16, unscaled);
 * its attention then reads the context rows directly.  Rows of earlier positions must hold
 * what the earlier calls (or the caller) wrote there: nothing is gathered or re-read from the
 * pool.  Positions and masks are those of pkv_plan_extend; there is no cascade.
 *   ctx_row0   host int32 [batch]; rows [ctx_row0[r], ctx_row0[r] + seq_lens[r]) inside
 *              [0, ctx_rows) and disjoint between requests (else PKV_E_INVALID)
 * The plan's workspace_bytes does not include the context arrays (the caller owns them). */
int pkv_plan_extend_ctx(int32_t batch, const int32_t *seq_lens, const int32_t *extend_lens,
                        const int32_t *qo_indptr, const int32_t *ctx_row0, int64_t ctx_rows,
                        int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                        const pkv_plan_opts *opts, void *plan, size_t plan_cap, pkv_plan_info *info);

/* The store + attention of one chunk (a plan from pkv_plan_extend_ctx).
 *   q, o                      as pkv_attn_extend ([total_q][num_q_heads][head_dim] bf16)
 *   k_new, v_new, out_cache_loc  the new tokens' K/V rows and pool slots, in q order, as
 *                             pkv_kv_store takes them (total_q rows)
 *   ctx_k, ctx_v, ctx_rows    the context arrays (device, 16-byte aligned), ctx_rows rows each
 *   workspace                 as pkv_attn_extend; slot-range errors of the store are recorded
 *                             in its error word (a bad slot's pool and context rows are not
 *                             written), and so is a context row outside [0, ctx_rows)
 *                             (PKV_DERR_POSITION; that copy is skipped)
 * pkv_attn_extend rejects a context-buffer plan and this call any other (PKV_E_PLAN). */
int pkv_attn_extend_ctx(const pkv_pool *pool, const void *q, void *o, float sm_scale, const void *k_new,
                        const void *v_new, const int32_t *out_cache_loc, void *ctx_k, void *ctx_v,
                        int64_t ctx_rows, const pkv_plan_info *info, const void *plan_dev, void *workspace,
                        size_t ws_bytes, void *stream);

/* Synchronises `stream`, reads the error word of `workspace` (PKV_OK when zero, else
 * PKV_E_DEVICE with the raw word in *raw when raw != NULL). */
int pkv_get_device_error(void *workspace, void *stream, int32_t *raw);

/* Measurement hook (no counterpart in the pages: it exists so a benchmark can time the
 * tensor-core kernel alone).  The next pkv_attn_extend call records the CUDA event `start`
 * on its stream right before its attention kernel and `stop` right after it -- after the
 * key gather, before the merge -- and then clears the hook.  start, stop: cudaEvent_t
 * handles owned by the caller; NULL, NULL clears it.  Process-wide, not thread-safe. */
int pkv_set_kernel_events(void *start, void *stop);

/* Failure-detection hook (no counterpart in the pages).  Every wait inside the attention
 * kernels (one role waiting for another's copy, MMA or release) is bounded; when one gives up,
 * the kernel records PKV_DERR_TIMEOUT | which-wait in the error word, every role of that CTA
 * stops, copies and MMAs already in flight are allowed to land, tensor memory is freed and
 * the kernel returns: the context stays usable and the host sees the flag through
 * pkv_get_device_error.  This sets the limit used by attention calls launched (or captured)
 * after it, in nanoseconds; 0 restores the default of 2 s, orders of magnitude above any
 * legitimate wait.  A limit of a few nanoseconds makes the first wait that does not succeed
 * at once give up -- the way to exercise the timeout path.  Process-wide, not thread-safe
 * against concurrent launches.  pkv_get_wait_limit_ns returns the current limit. */
int pkv_set_wait_limit_ns(uint64_t ns);
uint64_t pkv_get_wait_limit_ns(void);

/* pkv_attn_decode for callers that cannot allocate device memory (no counterpart in the
 * pages: it exists for embedding).  Some callers have no workspace to pass at call time --
 * a serving loop that froze its device-memory budget after start-up, or a host program
 * without a device allocator of its own.  This call runs the same kernels as
 * pkv_attn_decode with its scratch (error word + partial-state records) in one fixed
 * device array of PKV_NOALLOC_WORKSPACE_BYTES that every GPU loading the library holds until
 * exit; the caller still passes every input and output.
 *   - plans needing more than PKV_NOALLOC_WORKSPACE_BYTES of workspace: PKV_E_WORKSPACE,
 *     nothing launched;
 *   - the first call on a device looks up the array's address on that device (with it
 *     current) and caches it: make that first call before any stream capture;
 *   - every call clears the error word on `stream` first; all calls share the array, so
 *     calls that overlap on the GPU race on it;
 *   - allocates nothing (no cudaMalloc / cudaFree / allocating library routine).       */
#define PKV_NOALLOC_WORKSPACE_BYTES (32u << 20)
int pkv_attn_decode_noalloc(const pkv_pool *pool, const pkv_batch *batch, const void *q, void *o,
                            float sm_scale, const pkv_plan_info *info, const void *plan_dev,
                            void *stream);

/* The error word of pkv_attn_decode_noalloc's fixed array on the current device (the array's
 * address is private to the library, so pkv_get_device_error cannot reach it).  Synchronises
 * `stream`; PKV_OK when the word is zero, else PKV_E_DEVICE with the raw word in *raw (may be
 * NULL).  Each pkv_attn_decode_noalloc call clears the word before it launches, so after a
 * call on `stream` this reports that call's slot-range, position and timeout flags.  Like the
 * call itself it allocates nothing; on a device with no earlier call it looks up the array's
 * address first. */
int pkv_get_noalloc_device_error(void *stream, int32_t *raw);

/* ------------------------------------------------------------------------------------ */
/* host radix tree ([RC]): token ids -> pool slots, with LRU eviction and lock_ref       */
/*                                                                                      */
/* Page size 1: children are keyed by the first token of their key.  Time is a logical   */
/* clock that advances once per match_prefix / insert; LRU ties break by node id.        */
/* Node ids are assigned in creation order (root = 0) and stay valid until the node is    */
/* evicted.                                                                              */

typedef struct pkv_tree pkv_tree;

/* A new tree evicts least recently used first (PKV_EVICT_LRU). */
pkv_tree *pkv_tree_new(void);
void pkv_tree_free(pkv_tree *t);

/* Eviction policies ([RC] "Eviction 전략" names lru, lfu, slru, fifo, mru, filo and
 * priority, and gives nodes a hit_count and a priority; [RC] "핵심 자료구조: TreeNode").
 * The page prints only the LRU order; each other order is the plainest reading of its
 * name.  Smallest key first, ties by node id:
 *   LRU (last access) | LFU (hits, last access) | SLRU (hits >= 2, last access: nodes with
 *   fewer than 2 hits go first) | FIFO (node id: created first) | MRU (-last access) |
 *   FILO (-node id) | PRIORITY (priority, last access: lowest priority first).
 * Hits: every node of the path a match_prefix returns gains one (after any split). */
enum {
    PKV_EVICT_LRU = 0,
    PKV_EVICT_LFU = 1,
    PKV_EVICT_SLRU = 2,
    PKV_EVICT_FIFO = 3,
    PKV_EVICT_MRU = 4,
    PKV_EVICT_FILO = 5,
    PKV_EVICT_PRIORITY = 6
};

/* Select the order later pkv_tree_evict calls use (any time; PKV_E_UNSUPPORTED for an
 * unknown policy). */
int pkv_tree_set_policy(pkv_tree *t, int policy);

/* Paged tree: cache whole blocks of page_size tokens only ([SG] §技術的詳細 / Technical
 * Details: its cache's insert refers to the KV by 16-token block, position / 16).
 * match_prefix, insert, match_len and schedule then use the key's first page_size * floor(n / page_size) tokens
 * and compare a block at a time, so every node key, match length and cached length is a
 * multiple of page_size; a request's trailing partial block stays out of the tree.  The
 * slots a caller inserts for a block are expected to be one pool page (pkv_batch.page_size).
 * Allowed only while the tree is empty (PKV_E_INVALID otherwise, or for page_size outside
 * [1, 4096]); page_size 1 is the token tree. */
int pkv_tree_set_page_size(pkv_tree *t, int32_t page_size);

/* Longest cached prefix of key[0..n) ([RC] "프리픽스 매칭"): writes its slots to values
 * (up to values_cap of them), the matched length to *matched and the last node on the
 * matched path to *last_node (0 = root when nothing matched).  A match that ends inside a
 * node splits that node first ([RC] "노드 분할"), so *last_node ends exactly at the match. */
int pkv_tree_match_prefix(pkv_tree *t, const int32_t *key, int64_t n, int32_t *values,
                          int64_t values_cap, int64_t *matched, int64_t *last_node);

/* Insert key -> value (n tokens each) ([RC] "삽입").  *prefix_len receives how many
 * leading tokens were already cached; value[0 .. *prefix_len) duplicate cached slots and
 * are the caller's to free. */
int pkv_tree_insert(pkv_tree *t, const int32_t *key, const int32_t *value, int64_t n,
                    int64_t *prefix_len);

/* pkv_tree_insert with a priority ([RC] "삽입": the start node's priority is raised to at
 * least `priority` and a created leaf gets it; "노드 분할": a split's upper part keeps the
 * child's priority).  pkv_tree_insert is this call with priority 0. */
int pkv_tree_insert_priority(pkv_tree *t, const int32_t *key, const int32_t *value, int64_t n,
                             int64_t priority, int64_t *prefix_len);

/* Evict unlocked leaves in the tree's policy order (least recently used first by default) until at least num_tokens slots are
 * freed or nothing is evictable ([RC] "Eviction 전략").  A parent that becomes an unlocked
 * leaf joins the candidates.  Freed slots go to freed[0 .. *num_freed) in eviction order
 * (PKV_E_WORKSPACE if freed_cap is too small; nothing is evicted then). */
int pkv_tree_evict(pkv_tree *t, int64_t num_tokens, int32_t *freed, int64_t freed_cap,
                   int64_t *num_freed);

/* Cached prefix length of key[0..n) (*len), without changing the tree: no split, no access
 * time, no hit.  For a scheduler that compares waiting requests before admitting any. */
int pkv_tree_match_len(pkv_tree *t, const int32_t *key, int64_t n, int64_t *len);

/* Cache-aware scheduling ([SG] summary §Cache-Aware Scheduling: requests whose prefix is
 * longest in the radix tree go first, so cached prefixes are used before they are evicted;
 * reported ~30 % above first-come-first-served on few-shot workloads).  The n waiting
 * requests are token lists tokens[offsets[i] .. offsets[i+1]) (host, CSR).  order[0..n)
 * receives the admission order: PKV_SCHED_LPM = longest cached prefix first, ties in queue
 * order; PKV_SCHED_FCFS = queue order.  match_len[0..n) (may be NULL) receives each
 * request's cached prefix length.  The tree is not changed. */
enum { PKV_SCHED_LPM = 0, PKV_SCHED_FCFS = 1 };
int pkv_schedule(pkv_tree *t, const int32_t *tokens, const int64_t *offsets, int32_t n, int policy,
                 int32_t *order, int64_t *match_len);

/* lock_ref on the path node..root ([RC] "참조 카운트: lock_ref"); locked nodes are never
 * evicted.  *delta (may be NULL) gets the change of the evictable size. */
int pkv_tree_inc_lock_ref(pkv_tree *t, int64_t node, int64_t *delta);
int pkv_tree_dec_lock_ref(pkv_tree *t, int64_t node, int64_t *delta);

/* A batch's match-and-lock in one call: for i = 0 .. n-1 in order, key i = keys[offsets[i] ..
 * offsets[i+1]) (host, CSR) is matched as pkv_tree_match_prefix matches it (splitting a node
 * it ends inside, updating access times) and the path to its last matched node is locked as
 * pkv_tree_inc_lock_ref locks it -- the same tree, values and nodes as the 2n single calls.
 * values (room for offsets[n] entries) receives the matched values of every key back to
 * back, key i's at values[sum of matched[0 .. i)]; matched[i] and last_nodes[i] get key i's
 * matched length and last node.  What a server does for every newly admitted batch before
 * planning it ([RC] "매칭", "참조 카운트: lock_ref"). */
int pkv_tree_match_lock_batch(pkv_tree *t, const int32_t *keys, const int64_t *offsets, int32_t n,
                              int32_t *values, int64_t *matched, int64_t *last_nodes);

/* A token pool's batch table in one call (host memory): row i of table ([n][stride] int32)
 * gets request i's cached slots cached[ca_i .. ca_i + cached_len[i]) and then its new slots
 * fresh[fa_i .. fa_i + fresh_len[i]), where ca_i and fa_i are the sums of cached_len and of
 * fresh_len over the rows before i -- the req_to_token rows of the batch ([RC] "매칭": the
 * matched values are the prefix's slots).  The rest of each row is left as it is.
 * PKV_E_INVALID if a length is negative or a row would pass stride (nothing is written). */
int pkv_fill_batch_table(const int32_t *cached, const int64_t *cached_len, const int32_t *fresh,
                         const int64_t *fresh_len, int32_t n, int32_t *table, int64_t stride);

int pkv_tree_sizes(pkv_tree *t, int64_t *evictable, int64_t *protected_size,
                   int64_t *total, int64_t *num_nodes);

/* Canonical dump for tests: per live node in id order, 8 + 2*len int64 entries
 * (id, parent id, lock_ref, last_access_time, len, num_children, hit_count, priority,
 * key[len], value[len]).
 * *used gets the entries needed; PKV_E_WORKSPACE when cap is smaller (nothing written). */
int pkv_tree_dump(pkv_tree *t, int64_t *out, int64_t cap, int64_t *used);

/* Shared-prefix cascade of a batch.  last_nodes[r] is request r's last matched node
 * (from match_prefix; its path from the root is the request's cached prefix).  Every node
 * on the paths of >= min_group requests becomes part of a span; consecutive nodes with the
 * same member set are fused into one span.  Output arrays are host buffers sized
 * cap_spans (span_*; grp_indptr needs cap_spans + 1) and cap_members (grp_req).       */
int pkv_tree_cascade(pkv_tree *t, const int64_t *last_nodes, int32_t batch, int32_t min_group,
                     int32_t *span_req, int32_t *span_start, int32_t *span_len,
                     int32_t *grp_indptr, int32_t *grp_req, int32_t cap_spans,
                     int32_t cap_members, int32_t *num_spans, int32_t *num_members);

/* ------------------------------------------------------------------------------------ */
/* token-slot allocator: owns the free slot indices ([RC] "Eviction 전략":                */
/* token_to_kv_pool_allocator.free(x.value)).  FIFO: alloc pops from the front, free     */
/* appends at the back.                                                                  */

typedef struct pkv_allocator pkv_allocator;

pkv_allocator *pkv_allocator_new(const int32_t *free_slots, int64_t n);  /* host, copied */
void pkv_allocator_free_all(pkv_allocator *a);
int pkv_allocator_alloc(pkv_allocator *a, int64_t n, int32_t *out);      /* PKV_E_NOSPACE */
int pkv_allocator_release(pkv_allocator *a, const int32_t *slots, int64_t n);
int64_t pkv_allocator_available(const pkv_allocator *a);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
