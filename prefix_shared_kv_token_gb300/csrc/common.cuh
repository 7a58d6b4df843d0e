// Device helpers shared by the kernels: thin inline-PTX wrappers (mbarrier, cp.async, TMA,
// tcgen05, mma.sync), bounded waits, conversions and the plan / workspace layouts.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define PKV_DEV __device__ __forceinline__

namespace pkv {

// ---------------------------------------------------------------------------------------
// error word (first 4 bytes of the workspace).  Kernels only ever set it (first error wins).
enum DeviceError : int32_t {
    DERR_NONE = 0,
    DERR_SLOT_RANGE = 0x100,      // a slot read from req_to_token / out_cache_loc is out of range
    DERR_TIMEOUT = 0x200,         // a bounded wait gave up (low byte: which wait)
    DERR_POSITION = 0x400,        // a work item asked for positions outside the row
};

PKV_DEV void set_error(int32_t *err, int32_t code) {
    if (err) atomicCAS(err, 0, code);
}
// The same, and when this is the first error, where it happened: words 1-3 of the header get
// three values of the caller's choosing (the fused store's bad context row: the token, the row
// and 0).
PKV_DEV void set_error_where(int32_t *err, int32_t code, int32_t w1, int32_t w2, int32_t w3) {
    if (err && atomicCAS(err, 0, code) == 0) {
        err[1] = w1;
        err[2] = w2;
        err[3] = w3;
    }
}

// ---------------------------------------------------------------------------------------
// shared-memory addresses and fences
PKV_DEV uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

PKV_DEV uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

PKV_DEV void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Programmatic dependent launch (every kernel here is launched with the programmatic stream
// serialization attribute, launch_pdl): the next kernel in the stream may be scheduled once
// every CTA of this one has issued pdl_trigger (or exited), and its CTAs then take SMs as they
// free up.  pdl_wait blocks until the preceding grid has completed and its writes are
// visible; each kernel calls it before it reads what the preceding kernels wrote -- or, when
// it reads nothing of theirs, before it exits, so that its own completion still implies
// theirs.
PKV_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
PKV_DEV void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Slot of context position t from a row of the batch table: the token table's entry, or
// with pages of 2^shift slots, the position's page times the page size plus its offset.
// A page outside the pool gives -1 (the callers flag it and read zeros).
PKV_DEV int32_t table_slot(const int32_t *row, int t, int shift, int64_t num_slots) {
    if (shift == 0) return __ldg(row + t);
    const int32_t pg = __ldg(row + (t >> shift));
    const int64_t slot = ((int64_t)pg << shift) + (t & ((1 << shift) - 1));
    return (pg < 0 || slot >= num_slots) ? -1 : (int32_t)slot;
}

// Named barrier `id` (1..15) among `count` threads (a multiple of 32).
PKV_DEV void named_bar_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
// Named barrier that also ANDs a predicate over its `count` threads: every thread gets the
// same answer, so a group can leave together.  Warp-uniform (aligned) use only.
PKV_DEV bool named_bar_and(int id, int count, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.and.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

// ---------------------------------------------------------------------------------------
// mbarrier
PKV_DEV void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
PKV_DEV void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
PKV_DEV void mbar_arrive(uint64_t *bar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
                 : "memory");
}
PKV_DEV void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
                     smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
PKV_DEV bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking probe of the same phase (try_wait may suspend the thread for a while before
// it returns false; test_wait never does).
PKV_DEV bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded waits.  A pipeline wait (a role waiting for another role's data or release) gives
// up after the launch's wait limit, a kernel argument set by pkv_set_wait_limit_ns (2 s by
// default: orders of magnitude above any legitimate wait); the caller then records the
// error and unwinds.  A drain wait -- letting copies or MMAs that are already in flight land
// before the CTA frees or abandons what they write to -- always allows kDrainTimeoutNs, so a
// short pipeline limit never cuts a drain short.
constexpr uint64_t kDefaultWaitNs = 2000000000ull;
constexpr uint64_t kDrainTimeoutNs = 2000000000ull;
// How a pipeline wait polls, fixed per launch from its limit (wait_policy on the host).  A
// wait first tries once (try_wait, which may suspend the thread briefly); after a failed
// retry, and then every (check_mask + 1) retries, it reads the timer.  The long default limit
// checks every 256 retries; a short limit (under 1 ms: the way to exercise the timeout path)
// checks on every retry, and its `quick` launches poll with the non-blocking test_wait so a
// short wait cannot pass unnoticed inside one suspended try.
struct WaitPolicy {
    uint64_t limit_ns;
    uint32_t check_mask;
    uint32_t quick;
};
__host__ __device__ inline WaitPolicy wait_policy(uint64_t limit_ns) {
    const bool quick = limit_ns < (1ull << 20);
    return WaitPolicy{limit_ns, quick ? 0u : 255u, quick ? 1u : 0u};
}

// Wait for the phase with the given parity to complete, for at most ~kDrainTimeoutNs.
// Returns false on timeout.
PKV_DEV bool mbar_wait(uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 0 && global_timer_ns() - t0 > kDrainTimeoutNs) return false;
    }
}

// ---------------------------------------------------------------------------------------
// cp.async (Ampere-style, 16 bytes, L2 only).  src_bytes < 16 zero-fills the rest.  No
// memory clobber: completion is ordered by cp.async.wait_group (which has one), and without
// it the compiler may hoist the shared-memory slot loads that feed the next copies.
PKV_DEV void cp_async_16(uint32_t dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes));
}
// One contiguous global -> shared copy (16-byte aligned addresses, size a multiple of 16),
// completing as transaction bytes on `bar` (async proxy, no thread waits for it).
PKV_DEV void bulk_copy_g2s(uint32_t dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}
PKV_DEV void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
PKV_DEV void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ---------------------------------------------------------------------------------------
// TMA (bulk tensor copies, async proxy, completion through mbarrier transaction bytes)
PKV_DEV void tma_load_3d(uint32_t dst, const CUtensorMap *map, int32_t c0, int32_t c1, int32_t c2,
                         uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
        : "memory");
}
// Four rows r0..r3 of a 2-D tensor map, starting at column `col`; box = {cols, 1}.
PKV_DEV void tma_gather4(uint32_t dst, const CUtensorMap *map, int32_t col, int32_t r0, int32_t r1, int32_t r2,
                         int32_t r3, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
        "%3, %4, %5, %6}], [%7];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(col), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(smem_u32(bar))
        : "memory");
}
PKV_DEV void prefetch_tmap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------------------------------
// tcgen05: tensor memory and the 5th-generation tensor-core MMA
PKV_DEV void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {  // whole warp
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
PKV_DEV void tmem_relinquish() { asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory"); }
PKV_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {  // whole warp
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
PKV_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
PKV_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
PKV_DEV void tc_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}
// D(tmem) (+)= A(smem desc) * B(smem desc)
PKV_DEV void mma_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// D(tmem) (+)= A(tmem) * B(smem desc)
PKV_DEV void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(
            d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
PKV_DEV void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
PKV_DEV void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 32 lanes x 32 consecutive 32-bit columns: thread i of the warp gets lane (base + i).
PKV_DEV void tmem_ld32(uint32_t taddr, uint32_t *r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
          "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}
PKV_DEV void tmem_st32(uint32_t taddr, const uint32_t *r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
        "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
        "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

PKV_DEV void tmem_st16(uint32_t taddr, const uint32_t *r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

// Shared-memory matrix descriptor for tcgen05.mma (128-byte swizzle, version 1).
//   start: byte address in shared memory; lbo / sbo: leading / stride byte offsets.
PKV_DEV uint64_t sdesc_sw128(uint32_t start, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((start >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;  // descriptor version for tcgen05
    d |= (uint64_t)2 << 61;  // SWIZZLE_128B
    return d;
}
// Instruction descriptor, kind::f16: bf16 x bf16 -> f32, dense.
//   a_mn / b_mn: 1 = operand is MN-major (else K-major).
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, int a_mn, int b_mn) {
    return (1u << 4)                       // D format: f32
           | (1u << 7)                     // A format: bf16
           | (1u << 10)                    // B format: bf16
           | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

// ---------------------------------------------------------------------------------------
// warp-level MMA (mma.sync, m16n8k16, bf16 in, f32 accumulate)
PKV_DEV void mma_bf16_16816(float *c, const uint32_t *a, const uint32_t *b) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, "
        "%2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}
PKV_DEV void ldmatrix_x4_trans(uint32_t *r, uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

// ---------------------------------------------------------------------------------------
// conversions
PKV_DEV float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// Packed fp32 pairs (sm_100+ f32x2 arithmetic: one instruction for two lanes of work).
PKV_DEV uint64_t f2_pack(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
PKV_DEV void f2_unpack(uint64_t v, float &a, float &b) { asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v)); }
PKV_DEV uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
PKV_DEV uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
// acc + the two bf16 halves of v, accumulated in fp32 (mixed-precision add.f32.bf16)
PKV_DEV void add_bf16x2_f32(uint32_t v, float &acc_lo, float &acc_hi) {
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tadd.rn.f32.bf16 %0, l, %0;\n\tadd.rn.f32.bf16 %1, h, %1;\n\t}"
        : "+f"(acc_lo), "+f"(acc_hi)
        : "r"(v));
}
PKV_DEV float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// 2^x for two bf16 values at once (ex2.approx.ftz.bf16x2): the exponent is rounded to bf16
// first, a relative weight error of about |x| * 2^-9 * ln 2.  Callers keep x <= 0, where the
// absolute error 2^x * |x| * 2^-9 * ln 2 stays below 2^-9 of the largest weight -- the order
// of rounding the weight itself to bf16, which the P.V product does anyway.  -inf gives +0.
PKV_DEV uint32_t ex2_bf16x2(uint32_t x) {
    uint32_t y;
    asm("ex2.approx.ftz.bf16x2 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}
PKV_DEV uint32_t mul_bf16x2(uint32_t a, uint32_t b) {
    uint32_t y;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(y) : "r"(a), "r"(b));
    return y;
}
PKV_DEV uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %2, %1;" : "=r"(r) : "f"(lo), "f"(hi));
    return r;
}
PKV_DEV float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
PKV_DEV float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// Two e4m3 codes (low byte first) -> bf16x2, exactly: every e4m3 value is a bf16 value.
PKV_DEV uint32_t e4m3x2_to_bf16x2(uint16_t v) {
    uint32_t h;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(v));
    float lo = __half2float(__ushort_as_half((unsigned short)(h & 0xFFFFu)));
    float hi = __half2float(__ushort_as_half((unsigned short)(h >> 16)));
    return pack_bf16x2(lo, hi);
}
// Two floats -> two e4m3 codes (round to nearest even, saturating finite values).
PKV_DEV uint16_t f32x2_to_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %2, %1;" : "=h"(r) : "f"(lo), "f"(hi));
    return r;
}

// ---------------------------------------------------------------------------------------
// plan blob layouts (host planner <-> kernels)
struct DecodeItem {      // 32 bytes
    int32_t g0;          // first KV head of the item's head group (heads g0 .. g0 + hg - 1)
    int32_t mode;        // 0: shared span (several member requests), 1: one request's tail
    int32_t nreq;        // requests in this item (<= 16 / G: one 16-row MMA tile per head)
    int32_t row_off;     // into item_req[] / item_rec[]
    int32_t src;         // batch index whose req_to_token row holds the keys
    int32_t k0;          // first key position
    int32_t k1;          // one past the last key position; < 0: seq_lens[src]
    int32_t rot;         // tile the item starts at (tiles are visited cyclically from there; the planner uses 0)
};

constexpr int kMaxSegs = 4;
// Rows that see fewer than kPreciseKeys keys give each weight a large share of the output,
// where rounding the weights to bf16 for the P.V product costs more than the output's own
// bf16 rounding leaves room for.  Items holding such rows (flagged by the planner) feed P.V
// with the weights split into bf16 high and low parts (two products into one accumulator)
// and sum the fp32 weights.
constexpr int kPreciseKeys = 32;
constexpr int32_t kItemPrecise = 1;
struct ExtendItem {      // 64 bytes
    int32_t g;           // KV head
    int32_t tok0;        // first query token (row of q / o)
    int32_t ntok;        // query tokens (<= 2 * 128 / G)
    int32_t qpos0;       // position of tok0; token t sees positions <= qpos0 + t
    int32_t pos0;        // context position of the first key of segment 0
    int32_t nseg;        // key segments, consecutive in context positions
    int32_t rec;         // -1: write o directly; else first partial record (one per token);
                         // kItemPacked: its PackInfo
    int32_t flags;       // kItemPrecise: some row sees fewer than kPreciseKeys keys; kItemPacked
    int32_t key0[kMaxSegs];   // first gathered key of each segment (row of the workspace)
    int32_t nkeys[kMaxSegs];  // keys of each segment
};

// A packed extend item: the last few tokens of up to four requests (at most 32 / G each) in
// one query tile, a 32-row group (one TMEM lane quarter, one softmax warp) each.  Its key
// segments are the shared spans the requests have in common (every group sees them) and
// each request's own remaining keys (only that request's group sees them); segment
// positions are explicit, since every member's own keys start at the same position.
constexpr int32_t kItemPacked = 4;
constexpr int kPackSegs = 5;
struct PackInfo {        // 128 bytes
    int32_t key0[kPackSegs];   // first gathered key of each segment
    int32_t nkeys[kPackSegs];  // keys of each segment
    int32_t spos[kPackSegs];   // context position of each segment's first key
    int32_t sgrp[kPackSegs];   // row group that sees the segment; -1: every group
    int32_t tok0[4];           // first query token of each group
    int32_t ntok[4];           // its tokens (0: group unused)
    int32_t qpos0[4];          // position of its first token
};

struct GatherUnit {      // 16 bytes: copy `len` slot rows of one request row into the workspace
    int32_t src;         // batch index whose req_to_token row holds the slots
    int32_t pos0;        // first position
    int32_t len;         // positions (<= 32)
    int32_t key0;        // destination key index
};

struct MergeItem {       // 16 bytes
    int32_t out_row;     // row of o (request for decode, query token for extend)
    int32_t rec0;        // first record
    int32_t nrec;        // records to merge
    int32_t rec_stride;  // distance between consecutive records of this row
};

// plan_info.offsets[] slots
enum PlanSection { SEC_ITEMS = 0, SEC_ROW_REQ = 1, SEC_ROW_REC = 2, SEC_MERGE = 3 };
// decode: offsets[4] = per-CTA item ranges (int32 [n + 1]), offsets[5] = n CTAs,
// offsets[6] = KV heads per item (hg)
enum DecodePlanSlot { SEC_CTA_OFF = 4, SEC_NUM_CTAS = 5, SEC_HEAD_GROUP = 6 };

constexpr size_t kWorkspaceHeader = 256;  // error word + padding

}  // namespace pkv
