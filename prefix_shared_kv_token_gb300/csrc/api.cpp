// Status strings, version, the device error word, device properties and the tensor-map
// encoder shared by the launchers.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <atomic>
#include <mutex>
#include <utility>
#include <vector>

#include "../../include/pkv.h"
#include "launch.h"

namespace pkv {

constexpr uint64_t kDefaultWaitLimitNs = 2000000000ull;  // 2 s

int num_sms() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
    if (cached[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 152;
        cached[dev] = n;
    }
    return cached[dev];
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        // the driver function as introduced in CUDA 12.0 (its signature has not changed since)
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

CUresult encode_tiled(CUtensorMap *map, CUtensorMapDataType dtype, cuuint32_t rank, void *base,
                      const cuuint64_t *dims, const cuuint64_t *strides_bytes, const cuuint32_t *box,
                      CUtensorMapSwizzle swizzle) {
    EncodeTiledFn fn = get_encode_fn();
    if (!fn) return CUDA_ERROR_NOT_FOUND;
    cuuint32_t elem_strides[5] = {1, 1, 1, 1, 1};
    return fn(map, dtype, rank, base, dims, strides_bytes, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

void *g_kernel_events[2] = {nullptr, nullptr};

static std::atomic<uint64_t> g_wait_limit_ns{kDefaultWaitLimitNs};
uint64_t wait_limit_ns() { return g_wait_limit_ns.load(std::memory_order_relaxed); }

}  // namespace pkv

extern "C" {

const char *pkv_strerror(int code) {
    switch (code) {
        case PKV_OK: return "ok";
        case PKV_E_INVALID: return "invalid argument";
        case PKV_E_UNSUPPORTED: return "unsupported shape or dtype";
        case PKV_E_WORKSPACE: return "workspace or buffer too small";
        case PKV_E_CUDA: return "CUDA error";
        case PKV_E_NOSPACE: return "no free KV slots";
        case PKV_E_NOTFOUND: return "unknown tree node";
        case PKV_E_DEVICE: return "device-side check failed";
        case PKV_E_PLAN: return "plan does not match the call";
        default: return "unknown error";
    }
}

int pkv_version(void) { return 100; }

int pkv_set_kernel_events(void *start, void *stop) {
    if ((start == nullptr) != (stop == nullptr)) return PKV_E_INVALID;
    pkv::g_kernel_events[0] = start;
    pkv::g_kernel_events[1] = stop;
    return PKV_OK;
}

int pkv_set_wait_limit_ns(uint64_t ns) {
    pkv::g_wait_limit_ns.store(ns == 0 ? pkv::kDefaultWaitLimitNs : ns, std::memory_order_relaxed);
    return PKV_OK;
}

uint64_t pkv_get_wait_limit_ns(void) { return pkv::wait_limit_ns(); }

int pkv_check_out_cache_loc(const int32_t *out_cache_loc, int64_t n, int64_t num_slots, int64_t *bad) {
    if (bad) *bad = -1;
    if (n < 0 || num_slots <= 0 || (n > 0 && !out_cache_loc)) return PKV_E_INVALID;
    if (n == 0) return PKV_OK;
    // The first index, in call order, whose slot is out of range or was seen before: that is
    // the smallest offending index.  A bitmap of the slots when it costs at most 16 bytes an
    // entry (plus 64 KB), one pass; else (a huge pool, a short list) sorting the entries.
    if (num_slots / 8 <= 16 * n + 65536) {
        std::vector<uint64_t> seen((size_t)((num_slots + 63) / 64), 0ull);
        for (int64_t i = 0; i < n; ++i) {
            const int32_t s = out_cache_loc[i];
            const uint64_t bit = 1ull << (s & 63);
            if (s < 0 || (int64_t)s >= num_slots || (seen[(size_t)s >> 6] & bit)) {
                if (bad) *bad = i;
                return PKV_E_INVALID;
            }
            seen[(size_t)s >> 6] |= bit;
        }
        return PKV_OK;
    }
    // (slot, index) pairs sorted by slot: a repeated slot sits next to its twin; the later
    // of the two occurrences (in call order) is the one reported
    std::vector<std::pair<int32_t, int64_t>> v;
    v.reserve((size_t)n);
    int64_t first_bad = -1;
    for (int64_t i = 0; i < n; ++i) {
        const int32_t s = out_cache_loc[i];
        if (s < 0 || (int64_t)s >= num_slots) {
            if (first_bad < 0 || i < first_bad) first_bad = i;
            continue;
        }
        v.push_back({s, i});
    }
    std::sort(v.begin(), v.end());
    for (size_t j = 1; j < v.size(); ++j)
        if (v[j].first == v[j - 1].first) {
            const int64_t i = std::max(v[j].second, v[j - 1].second);
            if (first_bad < 0 || i < first_bad) first_bad = i;
        }
    if (first_bad < 0) return PKV_OK;
    if (bad) *bad = first_bad;
    return PKV_E_INVALID;
}

int pkv_fill_batch_table(const int32_t *cached, const int64_t *cached_len, const int32_t *fresh,
                         const int64_t *fresh_len, int32_t n, int32_t *table, int64_t stride) {
    if (n < 0 || stride < 0 || (n > 0 && (!cached_len || !fresh_len || !table))) return PKV_E_INVALID;
    int64_t ca = 0, fa = 0;
    for (int32_t i = 0; i < n; ++i) {
        if (cached_len[i] < 0 || fresh_len[i] < 0 || cached_len[i] + fresh_len[i] > stride) return PKV_E_INVALID;
        ca += cached_len[i];
        fa += fresh_len[i];
    }
    if ((ca > 0 && !cached) || (fa > 0 && !fresh)) return PKV_E_INVALID;
    ca = fa = 0;
    for (int32_t i = 0; i < n; ++i) {
        int32_t *row = table + (int64_t)i * stride;
        if (cached_len[i] > 0) std::memcpy(row, cached + ca, sizeof(int32_t) * (size_t)cached_len[i]);
        if (fresh_len[i] > 0)
            std::memcpy(row + cached_len[i], fresh + fa, sizeof(int32_t) * (size_t)fresh_len[i]);
        ca += cached_len[i];
        fa += fresh_len[i];
    }
    return PKV_OK;
}

int pkv_get_device_error(void *workspace, void *stream, int32_t *raw) {
    if (!workspace) return PKV_E_INVALID;
    int32_t w = 0;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(&w, workspace, sizeof(w), cudaMemcpyDeviceToHost, s) != cudaSuccess) return PKV_E_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return PKV_E_CUDA;
    if (raw) *raw = w;
    return w == 0 ? PKV_OK : PKV_E_DEVICE;
}

}  // extern "C"
