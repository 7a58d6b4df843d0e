"""The device path driven from plain C: a C program compiled against include/pkv.h, linked
with libpkv.so and the CUDA runtime (no torch, no Python binding), stores the new tokens'
K/V with pkv_kv_store, plans and runs pkv_attn_decode or pkv_attn_extend on cudaMalloc'd
buffers, and writes the pool and the outputs back to files.  The pool must equal the
oracle's store bit for bit, and the outputs the oracle's attention read through the same
slot table (max-abs error <= 1e-2 for a bf16 pool).
"""

import os
import shutil
import subprocess

import numpy as np
import pytest

from oracle.attention import attend_pool
from oracle.kv_store import kv_store_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "prefix_shared_kv_token_gb300")

S, HKV, HQ, D = 96, 2, 8, 64
SEQ = (5, 17, 40, 1)

PROGRAM = r"""
#include <stdio.h>
#include <stdlib.h>
#include <stdint.h>
#include <math.h>
#include <cuda_runtime.h>
#include "pkv.h"

#define CK(c) do { if (!(c)) { fprintf(stderr, "FAIL line %d: %s\n", __LINE__, #c); return 1; } } while (0)

static void *load(const char *dir, const char *name, size_t bytes) {
    char path[4096];
    snprintf(path, sizeof path, "%s/%s", dir, name);
    FILE *f = fopen(path, "rb");
    if (!f) return NULL;
    void *p = malloc(bytes);
    size_t got = fread(p, 1, bytes, f);
    fclose(f);
    if (got != bytes) { free(p); return NULL; }
    return p;
}
static int save(const char *dir, const char *name, const void *p, size_t bytes) {
    char path[4096];
    snprintf(path, sizeof path, "%s/%s", dir, name);
    FILE *f = fopen(path, "wb");
    if (!f) return 0;
    size_t put = fwrite(p, 1, bytes, f);
    fclose(f);
    return put == bytes;
}
static void *dev(const void *host, size_t bytes) {
    void *d = NULL;
    if (cudaMalloc(&d, bytes) != cudaSuccess) return NULL;
    if (host && cudaMemcpy(d, host, bytes, cudaMemcpyHostToDevice) != cudaSuccess) return NULL;
    return d;
}

int main(int argc, char **argv) {
    CK(argc == 9);
    const char *dir = argv[1];
    const int S = atoi(argv[2]), hkv = atoi(argv[3]), hq = atoi(argv[4]), d = atoi(argv[5]);
    const int B = atoi(argv[6]), stride = atoi(argv[7]);
    const int extend = argv[8][0] == 'e';
    int32_t *hseq = load(dir, "seq.bin", B * 4), *hext = extend ? load(dir, "ext.bin", B * 4) : NULL;
    CK(hseq && (!extend || hext));
    int32_t *hqo = malloc((B + 1) * 4);
    hqo[0] = 0;
    for (int r = 0; r < B; ++r) hqo[r + 1] = hqo[r] + (extend ? hext[r] : 1);
    const int n = hqo[B];  /* query tokens = new tokens */
    const size_t pool_b = (size_t)S * hkv * d * 2, row_b = (size_t)hkv * d * 2, q_b = (size_t)n * hq * d * 2;
    void *hk = load(dir, "k_pool.bin", pool_b), *hv = load(dir, "v_pool.bin", pool_b);
    void *hkn = load(dir, "k_new.bin", n * row_b), *hvn = load(dir, "v_new.bin", n * row_b);
    int32_t *hloc = load(dir, "loc.bin", n * 4), *hrt = load(dir, "rt.bin", (size_t)B * stride * 4);
    void *hq_ = load(dir, "q.bin", q_b);
    CK(hk && hv && hkn && hvn && hloc && hrt && hq_);
    int32_t *hidx = malloc(B * 4);
    for (int r = 0; r < B; ++r) hidx[r] = r;

    void *dk = dev(hk, pool_b), *dv = dev(hv, pool_b), *dkn = dev(hkn, n * row_b), *dvn = dev(hvn, n * row_b);
    void *dloc = dev(hloc, n * 4), *drt = dev(hrt, (size_t)B * stride * 4), *dseq = dev(hseq, B * 4);
    void *didx = dev(hidx, B * 4), *dq = dev(hq_, q_b), *dout = dev(NULL, q_b);
    CK(dk && dv && dkn && dvn && dloc && drt && dseq && didx && dq && dout);
    cudaStream_t st;
    CK(cudaStreamCreate(&st) == cudaSuccess);

    pkv_pool pool = {dk, dv, S, hkv, d, PKV_BF16, 1.f, 1.f};
    pkv_batch batch = {(const int32_t *)drt, stride, B, (const int32_t *)didx, (const int32_t *)dseq, B, 1};
    pkv_plan_info info;
    if (extend) {
        CK(pkv_plan_extend(B, hseq, hext, hqo, hq, hkv, d, NULL, NULL, NULL, 0, &info) == PKV_OK);
    } else {
        CK(pkv_plan_decode(B, hseq, hq, hkv, d, NULL, NULL, NULL, 0, &info) == PKV_OK);
    }
    void *hplan = malloc(info.plan_bytes);
    if (extend) {
        CK(pkv_plan_extend(B, hseq, hext, hqo, hq, hkv, d, NULL, NULL, hplan, info.plan_bytes, &info) == PKV_OK);
    } else {
        CK(pkv_plan_decode(B, hseq, hq, hkv, d, NULL, NULL, hplan, info.plan_bytes, &info) == PKV_OK);
    }
    void *dplan = dev(hplan, info.plan_bytes), *dws = dev(NULL, info.workspace_bytes);
    CK(dplan && dws && cudaMemset(dws, 0, info.workspace_bytes) == cudaSuccess);

    CK(pkv_kv_store(&pool, dkn, dvn, (const int32_t *)dloc, n, dws, st) == PKV_OK);
    if (extend) {
        CK(pkv_attn_extend(&pool, &batch, dq, dout, 1.f / sqrtf((float)d), &info, dplan, dws, info.workspace_bytes,
                           st) == PKV_OK);
    } else {
        CK(pkv_attn_decode(&pool, &batch, dq, dout, 1.f / sqrtf((float)d), &info, dplan, dws, info.workspace_bytes,
                           st) == PKV_OK);
    }
    int32_t raw = -1;
    CK(pkv_get_device_error(dws, st, &raw) == PKV_OK && raw == 0);

    void *ho = malloc(q_b);
    CK(cudaMemcpy(ho, dout, q_b, cudaMemcpyDeviceToHost) == cudaSuccess);
    CK(cudaMemcpy(hk, dk, pool_b, cudaMemcpyDeviceToHost) == cudaSuccess);
    CK(cudaMemcpy(hv, dv, pool_b, cudaMemcpyDeviceToHost) == cudaSuccess);
    CK(save(dir, "o.bin", ho, q_b) && save(dir, "k_after.bin", hk, pool_b) && save(dir, "v_after.bin", hv, pool_b));
    printf("ok\n");
    return 0;
}
"""


def _bf16_bits(rng, shape):
    x = rng.standard_normal(shape).astype(np.float32)
    u = x.view(np.uint32)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)   # round to nearest even


def _run(tmp_path, files, B, stride, op):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("no nvcc")
    for name, arr in files.items():
        (tmp_path / name).write_bytes(np.ascontiguousarray(arr).tobytes())
    src = tmp_path / "abi_gpu.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "abi_gpu"
    subprocess.run([nvcc, "-x", "c", str(src), "-o", str(exe), "-I", os.path.join(ROOT, "include"), "-L", PKG,
                    "-lpkv", "-Xlinker", "-rpath," + PKG], check=True)
    r = subprocess.run([str(exe), str(tmp_path), str(S), str(HKV), str(HQ), str(D), str(B), str(stride), op],
                       capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr


def _f64(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_c_program_stores_and_extends(tmp_path):
    rng = np.random.default_rng(12)
    # (cached prefix, new tokens) per request: a short suffix over a short prefix, a long
    # suffix over one cached token, no prefix at all, one new token over a longer prefix
    spec = [(10, 7), (1, 30), (0, 5), (33, 1)]
    B, stride = len(spec), 48
    k_pool = _bf16_bits(rng, (S, HKV, D))
    v_pool = _bf16_bits(rng, (S, HKV, D))
    perm = rng.permutation(S).astype(np.int32)
    rt = np.zeros((B, stride), np.int32)
    nxt, loc = 0, []
    for r, (p, e) in enumerate(spec):
        rt[r, :p + e] = perm[nxt:nxt + p + e]
        loc.extend(rt[r, p:p + e].tolist())
        nxt += p + e
    loc = np.array(loc, np.int32)
    n = len(loc)
    k_new = _bf16_bits(rng, (n, HKV, D))
    v_new = _bf16_bits(rng, (n, HKV, D))
    q = _bf16_bits(rng, (n, HQ, D))
    seq = np.array([p + e for p, e in spec], np.int32)
    ext = np.array([e for _, e in spec], np.int32)
    _run(tmp_path, {"k_pool.bin": k_pool, "v_pool.bin": v_pool, "k_new.bin": k_new, "v_new.bin": v_new,
                    "loc.bin": loc, "rt.bin": rt, "seq.bin": seq, "ext.bin": ext, "q.bin": q}, B, stride, "e")
    want_k = kv_store_bf16(k_pool.copy(), k_new, loc)
    want_v = kv_store_bf16(v_pool.copy(), v_new, loc)
    assert np.array_equal(np.fromfile(tmp_path / "k_after.bin", np.uint16).reshape(S, HKV, D), want_k)
    assert np.array_equal(np.fromfile(tmp_path / "v_after.bin", np.uint16).reshape(S, HKV, D), want_v)
    o = _f64(np.fromfile(tmp_path / "o.bin", np.uint16).reshape(n, HQ, D))
    q64 = _f64(q)
    t0 = 0
    for r, (p, e) in enumerate(spec):
        want, _ = attend_pool(q64[t0:t0 + e], want_k, want_v, "bf16", 1.0, 1.0, rt[r], np.arange(p, p + e), D ** -0.5)
        assert np.max(np.abs(o[t0:t0 + e] - want)) <= 1e-2, r
        t0 += e


def test_c_program_stores_and_decodes(tmp_path):
    rng = np.random.default_rng(11)
    B, stride = len(SEQ), 48
    k_pool = _bf16_bits(rng, (S, HKV, D))
    v_pool = _bf16_bits(rng, (S, HKV, D))
    perm = rng.permutation(S).astype(np.int32)
    rt = np.zeros((B, stride), np.int32)
    # requests 1 and 2 share their first 12 slots (a cached prefix); the others are disjoint
    rt[0, :SEQ[0]] = perm[:SEQ[0]]
    rt[1, :SEQ[1]] = perm[5:5 + SEQ[1]]
    rt[2, :12] = rt[1, :12]
    rt[2, 12:SEQ[2]] = perm[22:22 + SEQ[2] - 12]
    rt[3, :SEQ[3]] = perm[50:50 + SEQ[3]]
    loc = np.array([rt[r, SEQ[r] - 1] for r in range(B)], np.int32)   # each decode token's own slot
    k_new = _bf16_bits(rng, (B, HKV, D))
    v_new = _bf16_bits(rng, (B, HKV, D))
    q = _bf16_bits(rng, (B, HQ, D))
    _run(tmp_path, {"k_pool.bin": k_pool, "v_pool.bin": v_pool, "k_new.bin": k_new, "v_new.bin": v_new,
                    "loc.bin": loc, "rt.bin": rt, "seq.bin": np.array(SEQ, np.int32), "q.bin": q}, B, stride, "d")

    # the store: bit-exact against the oracle's scatter
    want_k = kv_store_bf16(k_pool.copy(), k_new, loc)
    want_v = kv_store_bf16(v_pool.copy(), v_new, loc)
    got_k = np.fromfile(tmp_path / "k_after.bin", np.uint16).reshape(S, HKV, D)
    got_v = np.fromfile(tmp_path / "v_after.bin", np.uint16).reshape(S, HKV, D)
    assert np.array_equal(got_k, want_k) and np.array_equal(got_v, want_v)

    # the decode: each request's query at position L - 1 over its whole row of the stored pool
    o = np.fromfile(tmp_path / "o.bin", np.uint16).reshape(B, HQ, D)
    o64 = (o.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    q64 = (q.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    for r in range(B):
        want, _ = attend_pool(q64[r:r + 1], want_k, want_v, "bf16", 1.0, 1.0, rt[r], [SEQ[r] - 1], D ** -0.5)
        assert np.max(np.abs(o64[r] - want[0])) <= 1e-2, r
