"""The boundary used from plain C: a C program compiled against include/pkv.h and linked
with the in-tree libpkv.so drives the host entry points (tree, allocator, planner) with no
Python in between, and checks the worked example of "[SGLang] RadixAttention: Radix Tree
기반 프리픽스 캐싱의 핵심" ("Radix Tree 구조도": after inserting [1 2 3 4 5] and [1 2 3 6 7],
a query [1 2 3 4 5 8] hits 5 tokens and [1 2 3] is a shared node).  No device call is made.
"""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "prefix_shared_kv_token_gb300")

PROGRAM = r"""
#include <stdio.h>
#include <stdint.h>
#include "pkv.h"

#define CHECK(c) do { if (!(c)) { printf("FAIL line %d: %s\n", __LINE__, #c); return 1; } } while (0)

int main(void) {
    CHECK(pkv_version() > 0);
    CHECK(pkv_strerror(PKV_OK) != NULL);

    /* allocator: slots handed out in list order, released ones come back */
    const int32_t free_slots[8] = {7, 3, 5, 0, 1, 2, 4, 6};
    pkv_allocator *al = pkv_allocator_new(free_slots, 8);
    CHECK(al != NULL && pkv_allocator_available(al) == 8);
    int32_t got[5];
    CHECK(pkv_allocator_alloc(al, 5, got) == PKV_OK);
    CHECK(got[0] == 7 && got[1] == 3 && got[4] == 1 && pkv_allocator_available(al) == 3);
    CHECK(pkv_allocator_alloc(al, 4, got) != PKV_OK);          /* only 3 left */
    CHECK(pkv_allocator_release(al, got, 2) == PKV_OK && pkv_allocator_available(al) == 5);

    /* the worked example: insert [1 2 3 4 5] -> slots 0..4, then [1 2 3 6 7] -> 0 1 2 5 6 */
    pkv_tree *t = pkv_tree_new();
    CHECK(t != NULL);
    const int32_t k1[5] = {1, 2, 3, 4, 5}, v1[5] = {0, 1, 2, 3, 4};
    const int32_t k2[5] = {1, 2, 3, 6, 7}, v2[5] = {0, 1, 2, 5, 6};
    int64_t pre = -1;
    CHECK(pkv_tree_insert(t, k1, v1, 5, &pre) == PKV_OK && pre == 0);
    CHECK(pkv_tree_insert(t, k2, v2, 5, &pre) == PKV_OK && pre == 3);
    const int32_t q[6] = {1, 2, 3, 4, 5, 8};
    int32_t vals[8];
    int64_t matched = -1, node = -1;
    CHECK(pkv_tree_match_prefix(t, q, 6, vals, 8, &matched, &node) == PKV_OK);
    CHECK(matched == 5 && vals[0] == 0 && vals[3] == 3 && vals[4] == 4 && node >= 0);
    int64_t ev = -1, prot = -1, total = -1, nodes = -1;
    CHECK(pkv_tree_sizes(t, &ev, &prot, &total, &nodes) == PKV_OK);
    CHECK(total == 7 && nodes == 4);            /* root + [1 2 3] + [4 5] + [6 7] */
    pkv_tree_free(t);

    /* a decode plan for three requests, sized first, then written */
    const int32_t seq[3] = {80, 200, 1};
    pkv_plan_info info;
    CHECK(pkv_plan_decode(3, seq, 32, 8, 128, NULL, NULL, NULL, 0, &info) == PKV_OK);
    CHECK(info.op == 1 && info.batch == 3 && info.plan_bytes > 0 && info.workspace_bytes >= 256);
    static unsigned char blob[1 << 20];
    CHECK(info.plan_bytes <= sizeof(blob));
    CHECK(pkv_plan_decode(3, seq, 32, 8, 128, NULL, NULL, blob, info.plan_bytes, &info) == PKV_OK);
    CHECK(pkv_plan_decode(3, seq, 32, 8, 128, NULL, NULL, blob, 1, &info) != PKV_OK);  /* too small */
    const int32_t bad[1] = {0};
    CHECK(pkv_plan_decode(1, bad, 32, 8, 128, NULL, NULL, NULL, 0, &info) != PKV_OK);  /* seq_len < 1 */

    pkv_allocator_free_all(al);
    printf("ok\n");
    return 0;
}
"""


def test_c_program_drives_the_host_api(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if not cc:
        pytest.skip("no C compiler")
    lib = os.path.join(PKG, "libpkv.so")
    assert os.path.exists(lib), "libpkv.so is built at session start"
    src = tmp_path / "abi.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "abi"
    subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe),
                    "-L", PKG, "-lpkv", "-Wl,-rpath," + PKG], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
