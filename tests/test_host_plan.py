"""Planner checks on the host: every (request, query head, key position) is covered by
exactly one work item, records and merges are consistent, and malformed inputs are
rejected.  Also checks that libpkv exports every entry point include/pkv.h declares."""

import os
import re

import numpy as np
import pytest

import prefix_shared_kv_token_gb300 as pkv
from prefix_shared_kv_token_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

DEC = np.dtype([("g0", "<i4"), ("mode", "<i4"), ("nreq", "<i4"), ("row_off", "<i4"), ("src", "<i4"),
                ("k0", "<i4"), ("k1", "<i4"), ("rot", "<i4")])
EXT = np.dtype([("g", "<i4"), ("tok0", "<i4"), ("ntok", "<i4"), ("qpos0", "<i4"), ("pos0", "<i4"),
                ("nseg", "<i4"), ("rec", "<i4"), ("flags", "<i4"), ("key0", "<i4", (4,)), ("nkeys", "<i4", (4,))])
GU = np.dtype([("src", "<i4"), ("pos0", "<i4"), ("len", "<i4"), ("key0", "<i4")])
MRG = np.dtype([("out_row", "<i4"), ("rec0", "<i4"), ("nrec", "<i4"), ("stride", "<i4")])
PACK = np.dtype([("key0", "<i4", (5,)), ("nkeys", "<i4", (5,)), ("spos", "<i4", (5,)), ("sgrp", "<i4", (5,)),
                 ("tok0", "<i4", (4,)), ("ntok", "<i4", (4,)), ("qpos0", "<i4", (4,))])


def test_header_symbols_exported():
    hdr = open(os.path.join(ROOT, "include", "pkv.h")).read()
    declared = set(re.findall(r"\b(pkv_[a-z_0-9]+)\s*\(", hdr))
    assert len(declared) >= 20
    for name in sorted(declared):
        assert hasattr(_lib.lib, name), name
    assert set(_lib.SIGNATURES) == declared


def _sections(plan, dtype, n, off):
    b = plan.blob
    return np.frombuffer(b[off:off + n * dtype.itemsize].tobytes(), dtype=dtype)


def _check_cta_ranges(plan, off, nctas, nitems):
    # persistent CTAs: contiguous per-CTA item ranges that partition the item list
    nctas = int(nctas)
    assert 1 <= nctas <= max(1, nitems)
    cta = np.frombuffer(plan.blob[off:off + 4 * (nctas + 1)].tobytes(), np.int32)
    assert cta[0] == 0 and cta[-1] == nitems and np.all(np.diff(cta) >= (1 if nitems else 0))


def _decode_cover(plan, seq, hkv, cascade_spans=None):
    info = plan.info
    items = _sections(plan, DEC, info.num_items, info.offsets[0])
    nrows = (info.offsets[2] - info.offsets[1]) // 4
    row_req = np.frombuffer(plan.blob[info.offsets[1]:info.offsets[1] + 4 * nrows].tobytes(), np.int32)
    row_rec = np.frombuffer(plan.blob[info.offsets[2]:info.offsets[2] + 4 * nrows].tobytes(), np.int32)
    merges = _sections(plan, MRG, info.num_merge, info.offsets[3])
    B = len(seq)
    # persistent CTAs: contiguous per-CTA item ranges that partition the item list
    nctas, hg = int(info.offsets[5]), int(info.offsets[6])
    assert hg in (1, 2, 4, 8) and hkv % hg == 0 and 1 <= nctas <= max(1, info.num_items)
    cta_off = np.frombuffer(plan.blob[info.offsets[4]:info.offsets[4] + 4 * (nctas + 1)].tobytes(), np.int32)
    assert cta_off[0] == 0 and cta_off[-1] == info.num_items and np.all(np.diff(cta_off) >= (1 if info.num_items else 0))
    G = info.num_q_heads // hkv
    cover = [np.zeros((hkv, seq[r]), np.int32) for r in range(B)]
    recs_seen = {}
    for it in items:
        assert it["g0"] % hg == 0 and 1 <= it["nreq"] <= 16 // G
        # every item reads its keys in order from its first tile: member groups of one span
        # chunk then read each tile at about the same time, so all but the first hit L2
        assert it["rot"] == 0
        for i in range(it["nreq"]):
            r = row_req[it["row_off"] + i]
            k1 = it["k1"] if it["k1"] >= 0 else seq[r]
            cover[r][it["g0"]:it["g0"] + hg, it["k0"]:k1] += 1
            recs_seen.setdefault(r, set()).add(row_rec[it["row_off"] + i])
    # tensor-core span items: query rows gathered from members, keys gathered from the span
    nx, nu, nk, nq = (int(info.offsets[i]) for i in (8, 10, 11, 13))
    if nx:
        xitems = _sections(plan, EXT, nx, info.offsets[7])
        nprec = int(info.offsets[18])   # short requests' items (precise weights), after the spans'
        if nx > nprec:
            _check_cta_ranges(plan, info.offsets[16], info.offsets[17], nx - nprec)
        if nprec:
            _check_cta_ranges(plan, info.offsets[19], info.offsets[20], nprec)
        assert all(bool(it["flags"] & 1) == (k >= nx - nprec) for k, it in enumerate(xitems))
        units = _sections(plan, GU, nu, info.offsets[9])
        qsrc = np.frombuffer(plan.blob[info.offsets[12]:info.offsets[12] + 4 * nq].tobytes(), np.int32)
        nrl = max(int(it["rec"]) + int(it["ntok"]) for it in xitems)
        rec_list = np.frombuffer(plan.blob[info.offsets[14]:info.offsets[14] + 4 * nrl].tobytes(), np.int32)
        g_src, g_pos = np.full(nk, -1), np.full(nk, -1)
        for u in units:
            for i in range(u["len"]):
                assert g_src[u["key0"] + i] == -1
                g_src[u["key0"] + i], g_pos[u["key0"] + i] = u["src"], u["pos0"] + i
        assert np.all(g_src >= 0)
        assert 0 < int(info.workspace_bytes) and int(info.offsets[15]) % 256 == 0
        for it in xitems:
            assert it["nseg"] == 1 and 1 <= it["ntok"] <= 2 * (128 // G) and it["rec"] >= 0
            keys = np.arange(it["key0"][0], it["key0"][0] + it["nkeys"][0])
            for t in range(it["ntok"]):
                r = int(qsrc[it["tok0"] + t])
                assert np.all(g_pos[keys] <= it["qpos0"] + t)  # unmasked: the span precedes the query
                cover[r][it["g"], g_pos[keys]] += 1
                recs_seen.setdefault(r, set()).add(int(rec_list[it["rec"] + t]))
    for r in range(B):
        assert np.all(cover[r] == 1), r
    merged = {int(m["out_row"]): m for m in merges}
    for r in range(B):
        rec = recs_seen[r]
        if r in merged:
            m = merged[r]
            assert rec == set(range(m["rec0"], m["rec0"] + m["nrec"]))
        else:
            assert rec == {-1}
    return items


@pytest.mark.parametrize("chunk", [0, 64, 1000])
def test_decode_plan_covers_every_key_once(chunk):
    rng = np.random.default_rng(0)
    seq = rng.integers(1, 900, size=37).astype(np.int32)
    plan = pkv.plan_decode(seq, 32, 8, 128, None, {"chunk_keys": chunk} if chunk else None)
    _decode_cover(plan, seq, 8)


def test_decode_plan_with_cascade():
    # requests 0..5 share positions [0, 100); requests 0..2 also share [100, 130)
    seq = np.array([300, 150, 131, 120, 101, 400], np.int32)
    casc = pkv.Cascade(span_req=np.array([0, 1], np.int32), span_start=np.array([0, 100], np.int32),
                       span_len=np.array([100, 30], np.int32), grp_indptr=np.array([0, 6, 9], np.int32),
                       grp_req=np.array([0, 1, 2, 3, 4, 5, 0, 1, 2], np.int32))
    plan = pkv.plan_decode(seq, 8, 2, 64, casc, {"span_chunk": 4096, "chunk_keys": 256})
    items = _decode_cover(plan, seq, 2)
    # G = 4: 4 member requests per span item, both KV heads in one item -> 2 + 1 span items
    assert plan.info.num_span_items == 3
    assert sum(1 for it in items if it["mode"] == 0) == 3


@pytest.mark.parametrize("G", [1, 4, 8])
def test_decode_plan_tensor_spans(G):
    # a 700-key span shared by 40 requests (tensor-core path), a nested 300-key span shared by
    # 14 of them (tensor-core path) and a 100-key span shared by 3 (decode kernel)
    rng = np.random.default_rng(3)
    B = 45
    seq = (1000 + rng.integers(1, 400, size=B)).astype(np.int32)
    span_req = np.array([0, 0, 40], np.int32)
    span_start = np.array([0, 700, 0], np.int32)
    span_len = np.array([700, 300, 100], np.int32)
    grp = [list(range(40)), list(range(14)), [40, 41, 42]]
    casc = pkv.Cascade(span_req=span_req, span_start=span_start, span_len=span_len,
                       grp_indptr=np.cumsum([0] + [len(g) for g in grp]).astype(np.int32),
                       grp_req=np.concatenate(grp).astype(np.int32))
    plan = pkv.plan_decode(seq, 8 * G, 8, 128, casc)
    _decode_cover(plan, seq, 8)
    info = plan.info
    assert int(info.offsets[8]) > 0 and int(info.offsets[11]) == 1000  # both big spans gathered once
    assert int(info.offsets[13]) == 40 + 14


@pytest.mark.parametrize("hq,hkv", [(32, 8), (48, 12), (16, 16), (8, 1), (64, 8)])
def test_decode_plan_head_groups(hq, hkv):
    rng = np.random.default_rng(1)
    seq = rng.integers(1, 700, size=23).astype(np.int32)
    plan = pkv.plan_decode(seq, hq, hkv, 128, None)
    _decode_cover(plan, seq, hkv)
    hg = int(plan.info.offsets[6])
    assert hg == max(h for h in (1, 2, 4, 8) if hkv % h == 0)


def test_decode_plan_short_contexts_go_precise():
    # contexts shorter than 32 keys: one precise tensor-core item per KV head, whole context,
    # no decode-kernel items; a longer request in the same batch stays in the decode kernel
    seq = np.array([2, 31, 17, 32, 500], np.int32)
    casc = pkv.Cascade(span_req=np.array([3], np.int32), span_start=np.array([0], np.int32),
                       span_len=np.array([2], np.int32), grp_indptr=np.array([0, 5], np.int32),
                       grp_req=np.array([0, 1, 2, 3, 4], np.int32))
    plan = pkv.plan_decode(seq, 32, 8, 128, casc)
    items = _decode_cover(plan, seq, 8)
    info = plan.info
    assert int(info.offsets[18]) == 3 * 8
    row_req = np.frombuffer(plan.blob[info.offsets[1]:info.offsets[2]].tobytes(), np.int32)
    reqs = {int(row_req[it["row_off"] + i]) for it in items for i in range(it["nreq"])}
    assert reqs == {3, 4}
    only_short = pkv.plan_decode(np.array([5, 9], np.int32), 32, 8, 128, None)
    assert only_short.info.num_items == 0
    _decode_cover(only_short, np.array([5, 9], np.int32), 8)


def test_decode_plan_cuts_small_batches_finer():
    # 64 requests x 300 unshared keys: 256-key chunks would leave most CTAs idle
    seq = np.full(64, 300, np.int32)
    plan = pkv.plan_decode(seq, 32, 8, 128, None)
    items = _decode_cover(plan, seq, 8)
    assert len(items) >= 2 * 152 * 0.9 and (items["k1"] - items["k0"]).max() < 256
    big = pkv.plan_decode(seq, 32, 8, 128, None, {"chunk_keys": 256})   # explicit size is kept
    assert (_decode_cover(big, seq, 8)["k1"] - _decode_cover(big, seq, 8)["k0"]).max() == 256


def test_decode_plan_balances_ctas():
    # LPT: no CTA carries more than the mean load plus one item
    rng = np.random.default_rng(2)
    seq = rng.integers(100, 3000, size=300).astype(np.int32)
    plan = pkv.plan_decode(seq, 32, 8, 128, None, {"chunk_keys": 256, "num_sms": 20})
    items = _decode_cover(plan, seq, 8)
    info = plan.info
    nctas = int(info.offsets[5])
    assert nctas == 20
    cta_off = np.frombuffer(plan.blob[info.offsets[4]:info.offsets[4] + 4 * (nctas + 1)].tobytes(), np.int32)
    keys = (items["k1"] - items["k0"]).astype(np.int64)
    load = np.array([keys[cta_off[b]:cta_off[b + 1]].sum() for b in range(nctas)])
    assert load.max() <= keys.sum() / nctas + keys.max()


def test_decode_plan_rejects_bad_cascade():
    seq = np.array([50, 50], np.int32)
    bad = pkv.Cascade(span_req=np.array([0], np.int32), span_start=np.array([5], np.int32),
                      span_len=np.array([10], np.int32), grp_indptr=np.array([0, 2], np.int32),
                      grp_req=np.array([0, 1], np.int32))
    with pytest.raises(pkv.PkvError):
        pkv.plan_decode(seq, 8, 2, 64, bad)   # a span must start where the previous ended (0)
    with pytest.raises(pkv.PkvError):
        pkv.plan_decode(np.array([0], np.int32), 8, 2, 64)  # empty context
    with pytest.raises(pkv.PkvError):
        pkv.plan_decode(seq, 12, 8, 64)      # G not in {1, 2, 4, 8}
    with pytest.raises(pkv.PkvError):
        pkv.plan_decode(seq, 8, 2, 96)       # head_dim


@pytest.mark.parametrize("cascade", [False, True])
def test_extend_plan_covers_causal_triangle(cascade):
    ext = np.array([70, 33, 1, 129], np.int32)
    pre = np.array([300, 300, 300, 0], np.int32) if not cascade else np.array([300, 300, 300, 0], np.int32)
    seq = pre + ext
    qo = np.concatenate([[0], np.cumsum(ext)]).astype(np.int32)
    casc = None
    if cascade:
        casc = pkv.Cascade(span_req=np.array([1], np.int32), span_start=np.array([0], np.int32),
                           span_len=np.array([250], np.int32), grp_indptr=np.array([0, 3], np.int32),
                           grp_req=np.array([0, 1, 2], np.int32))
    plan = pkv.plan_extend(seq, ext, qo, 32, 8, 128, casc)
    info = plan.info
    items = _sections(plan, EXT, info.num_items, info.offsets[0])
    nx = int(info.offsets[10])   # rows that see few keys: their own list, after the common one
    _check_cta_ranges(plan, info.offsets[7], info.offsets[8], info.num_items - nx)
    if nx:
        _check_cta_ranges(plan, info.offsets[11], info.offsets[12], nx)
        assert int(info.offsets[9]) == int(info.offsets[0]) + 64 * (info.num_items - nx)
    for k, it in enumerate(items):   # flagged exactly when its first row sees fewer than 32 keys
        assert bool(it["flags"] & 1) == (it["qpos0"] + 1 < 32) and (k >= info.num_items - nx) == bool(it["flags"] & 1)
    units = _sections(plan, GU, info.offsets[5], info.offsets[4])
    # gathered key -> (source request, position); every gathered key is written once
    nk = int(info.offsets[6])
    g_src, g_pos = np.full(nk, -1), np.full(nk, -1)
    for u in units:
        for i in range(u["len"]):
            assert g_src[u["key0"] + i] == -1
            g_src[u["key0"] + i], g_pos[u["key0"] + i] = u["src"], u["pos0"] + i
    assert np.all(g_src >= 0)
    T = int(qo[-1])
    req_of_tok = np.repeat(np.arange(4), ext)
    pos_of_tok = np.concatenate([np.arange(pre[r], seq[r]) for r in range(4)])
    members = {0: {0, 1, 2}, 1: {0, 1, 2}, 2: {0, 1, 2}, 3: {3}}
    cover = np.zeros((T, 8, int(seq.max())), np.int32)
    packs = _sections(plan, PACK, int(info.offsets[14]), info.offsets[13])
    for it in items:
        if it["flags"] & 4:   # packed: row groups of several requests' last tokens
            pk = packs[it["rec"]]
            assert 2 <= it["nseg"] <= 5 and it["ntok"] == 128 // 4
            ngrp = 0
            for m in range(4):
                for t in range(pk["ntok"][m]):
                    tok = pk["tok0"][m] + t
                    assert 1 <= pk["ntok"][m] <= 32 // 4
                    for sgi in range(it["nseg"]):
                        if pk["sgrp"][sgi] not in (-1, m):
                            continue
                        for k in range(pk["nkeys"][sgi]):
                            pos = pk["spos"][sgi] + k
                            if pos <= pk["qpos0"][m] + t:
                                gk = pk["key0"][sgi] + k
                                assert g_pos[gk] == pos
                                assert g_src[gk] == req_of_tok[tok] or (casc is not None and g_src[gk] in members[req_of_tok[tok]])
                                cover[tok, it["g"], pos] += 1
                ngrp += pk["ntok"][m] > 0
            assert ngrp >= 2
            continue
        assert it["rec"] == -1 and 1 <= it["nseg"] <= 4
        for t in range(it["ntok"]):
            tok = it["tok0"] + t
            pos = it["pos0"]
            for sgi in range(it["nseg"]):
                for k in range(it["nkeys"][sgi]):
                    if pos + k <= it["qpos0"] + t:
                        gk = it["key0"][sgi] + k
                        assert g_pos[gk] == pos + k
                        assert g_src[gk] == req_of_tok[tok] or (casc is not None and g_src[gk] in members[req_of_tok[tok]])
                        cover[tok, it["g"], pos + k] += 1
                pos += it["nkeys"][sgi]
    for tok in range(T):
        want = np.zeros(cover.shape[2], np.int32)
        want[:pos_of_tok[tok] + 1] = 1
        assert np.array_equal(cover[tok, 0], want), tok
        assert np.all(cover[tok] == cover[tok, 0])
    if cascade:
        assert info.num_span_items > 0 and int(info.offsets[6]) < int(seq.sum())  # the span is gathered once
        # requests 0 and 2 end with 6 and 1 tokens after the shared span: one packed tile per head
        assert int(info.offsets[14]) == 1 and sum(1 for it in items if it["flags"] & 4) == 8


def test_struct_layouts_match_header(tmp_path):
    """The ctypes mirrors of the public structs have the header's sizes and field offsets."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if not cc:
        pytest.skip("no C compiler")
    structs = {"pkv_pool": _lib.PkvPool, "pkv_batch": _lib.PkvBatch, "pkv_cascade": _lib.PkvCascade,
               "pkv_plan_opts": _lib.PkvPlanOpts, "pkv_plan_info": _lib.PkvPlanInfo}
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "pkv.h"', "int main(void) {"]
    for name, cls in structs.items():
        lines.append(f'printf("{name} size %zu\\n", sizeof({name}));')
        for fname, _ in cls._fields_:
            lines.append(f'printf("{name} {fname} %zu\\n", offsetof({name}, {fname}));')
    lines += ["return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run([cc, "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    got = {tuple(l.split()[:2]): int(l.split()[2]) for l in out if l.strip()}
    import ctypes as C
    for name, cls in structs.items():
        assert got[(name, "size")] == C.sizeof(cls), name
        for fname, _ in cls._fields_:
            assert got[(name, fname)] == getattr(cls, fname).offset, (name, fname)


def test_decode_plan_tiny_batch_is_flat():
    # 4 requests of 80 keys sharing 64 (the tiny decode workload's shape): one item per request
    # over its whole context, direct outputs, no span items, no records, no merge
    seq = np.full(4, 80, np.int32)
    casc = pkv.Cascade(span_req=np.array([0], np.int32), span_start=np.array([0], np.int32),
                       span_len=np.array([64], np.int32), grp_indptr=np.array([0, 4], np.int32),
                       grp_req=np.arange(4, dtype=np.int32))
    plan = pkv.plan_decode(seq, 8, 2, 64, casc)
    items = _decode_cover(plan, seq, 2)
    assert len(items) == 4 and plan.info.num_span_items == 0
    assert plan.info.num_records == 0 and plan.info.num_merge == 0
    assert np.all(items["k0"] == 0) and np.all(items["k1"] == 80)
    # explicit chunk options keep the general plan (span items, records, merges)
    gen = pkv.plan_decode(seq, 8, 2, 64, casc, {"span_chunk": 64})
    _decode_cover(gen, seq, 2)
    assert gen.info.num_span_items > 0 and gen.info.num_merge == 4


def test_decode_plan_span_pass_beside_the_decode_kernel():
    # a 1,024-key prefix shared by 64 requests (tensor-core span) and long unshared tails: the
    # span pass is small next to the decode kernel, so it gets a few SMs of its own and runs
    # beside it, in about two long items per SM (fewer records than one item per SM)
    rng = np.random.default_rng(5)
    seq = (1024 + rng.integers(1500, 3000, size=64)).astype(np.int32)
    casc = pkv.Cascade(span_req=np.array([0], np.int32), span_start=np.array([0], np.int32),
                       span_len=np.array([1024], np.int32), grp_indptr=np.array([0, 64], np.int32),
                       grp_req=np.arange(64, dtype=np.int32))
    auto = pkv.plan_decode(seq, 32, 8, 128, casc)
    _decode_cover(auto, seq, 8)
    x_auto = int(auto.info.offsets[17])
    assert 12 <= x_auto < 152 and int(auto.info.offsets[5]) == 152 - x_auto
    serial = pkv.plan_decode(seq, 32, 8, 128, casc, {"span_sms": -1})
    _decode_cover(serial, seq, 8)
    assert int(serial.info.offsets[5]) == 152 and int(serial.info.offsets[17]) > x_auto
    assert auto.info.num_records <= serial.info.num_records
    fixed = pkv.plan_decode(seq, 32, 8, 128, casc, {"span_sms": 20})
    _decode_cover(fixed, seq, 8)
    assert int(fixed.info.offsets[17]) <= 20 and int(fixed.info.offsets[5]) == 132
    # a span pass large next to the decode kernel stays after it
    short = np.full(64, 1100, np.int32)
    big = pkv.plan_decode(short, 32, 8, 128, casc)
    _decode_cover(big, short, 8)
    assert int(big.info.offsets[5]) == min(152, big.info.num_items)
