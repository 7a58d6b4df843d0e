"""GPU parity: the CUDA path (through the C ABI) against the oracle on the same seeded inputs.

Bars: kv_store and every index table bit-exact; attention max-abs error <= 1e-2 for a bf16
pool and <= 5e-2 for an fp8 pool, against the float64 oracle (contiguous recompute, which
never looks at slots or tables).
"""

import numpy as np
import pytest
import torch

import workloads as W
from oracle import step as ostep
from oracle.fp8 import quantize_to_pool
from oracle.kv_store import kv_store_bf16, kv_store_fp8

pytestmark = pytest.mark.gpu

TOL = {"bf16": 1e-2, "fp8_e4m3": 5e-2}


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _pkv():
    import prefix_shared_kv_token_gb300 as pkv
    from prefix_shared_kv_token_gb300.runtime import PrefixCache
    return pkv, PrefixCache


def _f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def _bits(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 else t.cpu().numpy()


def run_step(w, cascade=True, opts=None, kinds=("extend", "decode"), page_size=1):
    pkv, PrefixCache = _pkv()
    pc = PrefixCache(w, page_size=page_size)
    pc.populate()
    calls = {}
    for kind in kinds:
        if any(r.kind == kind for r in w.requests):
            calls[kind] = pc.prepare(kind, cascade=cascade, opts=opts)
    for c in calls.values():
        c.run()
    torch.cuda.synchronize()
    for c in calls.values():
        assert pkv.get_device_error(c.workspace) == 0
    assert pkv.get_device_error(pc.err) == 0
    return pc, calls


def check_outputs(w, calls, tol=None):
    tol = tol or TOL[w.dtype]
    for kind, c in calls.items():
        want = ostep.expected_outputs(w, kind)
        got = _f64(c.o)
        assert got.shape == want.shape
        assert np.all(np.isfinite(got))
        err = np.max(np.abs(got - want))
        assert err <= tol, (kind, err)


def check_pool(w, pc):
    """Every cached and new token's pool row equals the oracle's store of its K/V."""
    rows_k, rows_v, slots = [], [], []
    for r in w.requests:
        toks = W.context_tokens(w, r)
        vals, _ = pc.tree.match_prefix(toks[:len(toks) - r.n_new])
        kb, vb = W.context_kv_bits(w, r)
        slots.append(vals)
        rows_k.append(kb[:len(vals)])
        rows_v.append(vb[:len(vals)])
    slots = np.concatenate(slots)
    kb, vb = np.concatenate(rows_k), np.concatenate(rows_v)
    idx = torch.from_numpy(slots.astype(np.int64)).to(pc.pool.k.device)
    gk, gv = _bits(pc.pool.k[idx]), _bits(pc.pool.v[idx])
    if w.dtype == "bf16":
        assert np.array_equal(gk, kb) and np.array_equal(gv, vb)
    else:
        assert np.array_equal(gk, quantize_to_pool(W.bf16_bits_to_f64(kb), w.k_scale))
        assert np.array_equal(gv, quantize_to_pool(W.bf16_bits_to_f64(vb), w.v_scale))


# ------------------------------------------------------------------------------ kv_store

@pytest.mark.parametrize("n,hkv,d", [(1, 8, 128), (7, 2, 64), (333, 8, 128), (4096, 8, 128)])
@pytest.mark.parametrize("dtype,scale", [("bf16", 1.0), ("fp8_e4m3", 1.0), ("fp8_e4m3", 0.0125), ("fp8_e4m3", 3.7)])
def test_kv_store_bit_exact(n, hkv, d, dtype, scale):
    pkv, _ = _pkv()
    S = 5000
    rng = np.random.default_rng(n + hkv)
    x = rng.standard_normal((2, n, hkv, d)).astype(np.float32) * np.float32(scale * 40)
    x[:, :, 0, :4] = [500.0, -1e4, 3e-3 * scale, -2e-4 * scale]       # saturation and subnormal cases
    bits = W.generate.to_bf16_bits(x)
    loc = rng.permutation(S)[:n].astype(np.int32)
    pool = pkv.Pool.allocate(S, hkv, d, dtype, scale, scale)
    init = rng.integers(0, 255, size=pool.k.numel() * pool.k.element_size(), dtype=np.uint8)
    pool.k.view(torch.uint8).view(-1).copy_(torch.from_numpy(init))
    pool.v.view(torch.uint8).view(-1).copy_(torch.from_numpy(init[::-1].copy()))
    k0, v0 = _bits(pool.k), _bits(pool.v)
    dev = lambda b: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).cuda()
    err = torch.zeros(4, dtype=torch.int32, device="cuda")
    pkv.kv_store(pool, dev(bits[0]), dev(bits[1]), torch.from_numpy(loc).cuda(), err)
    torch.cuda.synchronize()
    assert pkv.get_device_error(err) == 0
    if dtype == "bf16":
        want_k, want_v = kv_store_bf16(k0, bits[0], loc), kv_store_bf16(v0, bits[1], loc)
    else:
        want_k, want_v = kv_store_fp8(k0, bits[0], loc, scale), kv_store_fp8(v0, bits[1], loc, scale)
    assert np.array_equal(_bits(pool.k), want_k)
    assert np.array_equal(_bits(pool.v), want_v)


def test_kv_store_out_of_range_slot_is_reported_not_written():
    pkv, _ = _pkv()
    pool = pkv.Pool.allocate(64, 2, 64)
    k = torch.ones((3, 2, 64), dtype=torch.bfloat16, device="cuda")
    loc = torch.tensor([5, 64, 7], dtype=torch.int32, device="cuda")   # 64 == num_slots
    err = torch.zeros(4, dtype=torch.int32, device="cuda")
    pkv.kv_store(pool, k, k, loc, err)
    assert pkv.get_device_error(err) == 0x100
    assert pool.k[5].float().sum().item() == 128 and pool.k[7].float().sum().item() == 128
    assert pool.k.float().sum().item() == 256


def test_kv_store_empty_is_noop():
    pkv, _ = _pkv()
    pool = pkv.Pool.allocate(8, 1, 64)
    e = torch.empty((0, 1, 64), dtype=torch.bfloat16, device="cuda")
    pkv.kv_store(pool, e, e, torch.empty(0, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()


# ------------------------------------------------------------------------------ decode

def test_tiny_decode_full():
    w = W.config(1)
    pc, calls = run_step(w)
    check_outputs(w, calls)
    check_pool(w, pc)


@pytest.mark.parametrize("cascade", [True, False])
@pytest.mark.parametrize("hq,hkv,d", [(32, 8, 128), (8, 8, 64), (16, 8, 128), (64, 8, 64)])
def test_decode_small(cascade, hq, hkv, d):
    w = W.batched_decode(seed=31, n_req=21, prefix=200, lo=1, hi=300, hq=hq, hkv=hkv, d=d, num_slots=20000)
    pc, calls = run_step(w, cascade=cascade)
    check_outputs(w, calls)
    if cascade:
        assert calls["decode"].plan.info.num_span_items > 0


@pytest.mark.parametrize("hq,hkv,d", [(32, 8, 128), (8, 8, 128), (16, 8, 64), (64, 8, 128), (8, 2, 64)])
def test_decode_tensor_core_spans(hq, hkv, d):
    # a 700-key prefix shared by 40 requests: attended on the tensor cores as a dense block
    w = W.batched_decode(seed=36, n_req=40, prefix=700, lo=1, hi=300, hq=hq, hkv=hkv, d=d, num_slots=40000)
    pc, calls = run_step(w)
    assert int(calls["decode"].plan.info.offsets[8]) > 0
    check_outputs(w, calls)


@pytest.mark.parametrize("dtype", ["bf16", "fp8_e4m3"])
def test_decode_tensor_core_nested_spans(dtype):
    # root shared by 256 leaves, 16 depth-1 nodes shared by 16 leaves each (both tensor-core
    # spans), unique 256-key leaves; plus 4 extending branches in the same batch
    w = W.tot_mixed(seed=37, root_len=512, depth=2, branch=16, seg=256, n_new_branches=4, num_slots=90000,
                    dtype=dtype)
    pc, calls = run_step(w)
    assert int(calls["decode"].plan.info.offsets[8]) > 0
    check_outputs(w, calls)


@pytest.mark.parametrize("cascade", [True, False])
def test_decode_fp8_small(cascade):
    w = W.batched_decode(seed=32, n_req=9, prefix=150, lo=20, hi=200, num_slots=8000, dtype="fp8_e4m3")
    pc, calls = run_step(w, cascade=cascade)
    check_outputs(w, calls)
    check_pool(w, pc)


@pytest.mark.parametrize("chunk", [64, 100, 4096])
def test_decode_chunking(chunk):
    w = W.batched_decode(seed=33, n_req=6, prefix=64, lo=100, hi=700, hq=8, hkv=2, d=64, num_slots=6000)
    _, calls = run_step(w, opts={"chunk_keys": chunk, "span_chunk": chunk})
    check_outputs(w, calls)


def test_multiturn_small():
    w = W.multiturn_decode(seed=34, n_conv=3, turns=3, user=(20, 90), reply=(5, 60), num_slots=20000)
    pc, calls = run_step(w)
    check_outputs(w, calls)
    check_pool(w, pc)


@pytest.mark.parametrize("hq,hkv,d", [(32, 8, 128), (8, 2, 64)])
def test_decode_short_contexts(hq, hkv, d):
    # contexts of 2 .. 31 keys: each weight carries a large share of the output, the case the
    # kernels feed with bf16 high + low weights
    b = W.generate._Builder(38, hq, hkv, d, 4096)
    for n in range(2, 32):
        b.request(b.segment(-1, n), "decode", 1)
    w = b.finish("short", 38, 4096)
    _, calls = run_step(w)
    check_outputs(w, calls)


def test_decode_context_of_one_token():
    b = W.generate._Builder(35, 8, 2, 64, 64)
    leaves = [b.segment(-1, 1) for _ in range(3)]      # contexts of a single (query) token
    for leaf in leaves:
        b.request(leaf, "decode", 1)
    w = b.finish("single", 35, 64)
    _, calls = run_step(w)
    got = _f64(calls["decode"].o)
    want = ostep.expected_outputs(w, "decode")
    assert np.max(np.abs(got - want)) <= 1e-2     # one key: the output is its value (bf16-rounded)


# ------------------------------------------------------------------------------ extend

@pytest.mark.parametrize("cascade", [True, False])
@pytest.mark.parametrize("hq,hkv,d", [(32, 8, 128), (8, 2, 64), (16, 16, 128), (64, 8, 128)])
def test_extend_small(cascade, hq, hkv, d):
    w = W.fewshot_extend(seed=41, n_req=3, prefix=300, suffix=70, hq=hq, hkv=hkv, d=d, num_slots=4000)
    pc, calls = run_step(w, cascade=cascade)
    check_outputs(w, calls)
    check_pool(w, pc)


@pytest.mark.parametrize("prefix,suffix", [(1, 1), (127, 129), (256, 33), (5, 300)])
def test_extend_ragged(prefix, suffix):
    w = W.fewshot_extend(seed=42 + prefix, n_req=2, prefix=prefix, suffix=suffix, num_slots=4000)
    _, calls = run_step(w)
    check_outputs(w, calls)


@pytest.mark.parametrize("cascade", [True, False])
@pytest.mark.parametrize("hq,hkv,prefix,suffix", [
    (16, 16, 100, 60),   # 2 key tiles; rows 0..27 see no key of the second
    (16, 16, 250, 3),
    (8, 4, 129, 64),     # a full 128-row query tile over 2 key tiles
    (32, 8, 1000, 20),   # 8 key tiles
    (32, 8, 300, 31),    # 3 key tiles: the even-tile warpgroup takes one more
    (16, 16, 10, 128),   # rows that see fewer than 32 keys (precise weights), 2 key tiles
])
def test_extend_one_query_tile_over_several_key_tiles(cascade, hq, hkv, prefix, suffix):
    """A single query tile over two or more key tiles is split between the two softmax
    warpgroups (alternate key tiles, partial states combined at the end)."""
    w = W.fewshot_extend(seed=47 + prefix, n_req=2, prefix=prefix, suffix=suffix, hq=hq, hkv=hkv, d=128,
                         num_slots=4000)
    _, calls = run_step(w, cascade=cascade)
    check_outputs(w, calls)


def test_extend_without_prefix():
    b = W.generate._Builder(43, 32, 8, 128, 2000)
    leaves = [b.segment(-1, n) for n in (1, 77, 160)]
    for leaf, n in zip(leaves, (1, 77, 160)):
        b.request(leaf, "extend", n)
    w = b.finish("noprefix", 43, 2000)
    _, calls = run_step(w)
    check_outputs(w, calls)


@pytest.mark.parametrize("cascade", [True, False])
def test_extend_fp8_small(cascade):
    w = W.fewshot_extend(seed=44, n_req=3, prefix=200, suffix=90, num_slots=4000, dtype="fp8_e4m3")
    pc, calls = run_step(w, cascade=cascade)
    check_outputs(w, calls)
    check_pool(w, pc)


def test_tot_mixed_small():
    w = W.tot_mixed(seed=45, root_len=300, depth=2, branch=3, seg=40, n_new_branches=2, num_slots=8000)
    pc, calls = run_step(w)
    assert set(calls) == {"extend", "decode"}
    check_outputs(w, calls)
    check_pool(w, pc)


def test_shared_equals_duplicated_prefix():
    """Same K/V reached through one shared span or through per-request copies (no
    sharing): the kernels give identical results either way within fp32 noise."""
    w = W.fewshot_extend(seed=46, n_req=4, prefix=180, suffix=40, hq=8, hkv=2, d=64, num_slots=4000)
    _, shared = run_step(w, cascade=True)
    _, plain = run_step(w, cascade=False)
    a, b = _f64(shared["extend"].o), _f64(plain["extend"].o)
    assert np.max(np.abs(a - b)) <= 2 * 2.0 ** -8


# ------------------------------------------------------------------------------ paged pool

@pytest.mark.parametrize("page", [4, 16])
@pytest.mark.parametrize("cascade", [True, False])
@pytest.mark.parametrize("hq,hkv,d", [(32, 8, 128), (8, 2, 64)])
def test_paged_extend(page, cascade, hq, hkv, d):
    """Page-table batches: the extend gathers read slot = page * P + position % P; the
    shared prefix is shared in whole blocks (its partial last block is per request)."""
    w = W.fewshot_extend(seed=60 + page, n_req=3, prefix=300, suffix=70, hq=hq, hkv=hkv, d=d, num_slots=4096)
    pc, calls = run_step(w, cascade=cascade, page_size=page)
    assert calls["extend"].batch.page_size == page
    check_outputs(w, calls)
    check_pool(w, pc)


@pytest.mark.parametrize("page", [2, 16])
@pytest.mark.parametrize("cascade", [True, False])
def test_paged_decode(page, cascade):
    w = W.batched_decode(seed=61, n_req=20, prefix=200, lo=5, hi=90, num_slots=8192)
    pc, calls = run_step(w, cascade=cascade, page_size=page)
    check_outputs(w, calls)
    check_pool(w, pc)


def test_paged_decode_tensor_core_spans():
    # a span shared by >= 12 requests and >= 256 keys goes through the gather + extend path
    w = W.batched_decode(seed=62, n_req=24, prefix=520, lo=3, hi=40, num_slots=16384)
    _, calls = run_step(w, page_size=16)
    assert calls["decode"].plan.info.offsets[8] > 0
    check_outputs(w, calls)


@pytest.mark.parametrize("page", [8, 16])
def test_paged_fp8_tot_mixed(page):
    w = W.tot_mixed(seed=63, root_len=300, depth=2, branch=3, seg=40, n_new_branches=2, num_slots=8192,
                    dtype="fp8_e4m3")
    pc, calls = run_step(w, page_size=page)
    assert set(calls) == {"extend", "decode"}
    check_outputs(w, calls)
    check_pool(w, pc)


def test_paged_equals_token_pool():
    """The same workload through a token table and through a page table: identical outputs
    (the kernels read the same K/V; only the slots differ)."""
    w = W.fewshot_extend(seed=64, n_req=4, prefix=180, suffix=40, hq=8, hkv=2, d=64, num_slots=4096)
    _, tok = run_step(w, cascade=False)
    _, pag = run_step(w, cascade=False, page_size=16)
    assert torch.equal(tok["extend"].o, pag["extend"].o)


def test_paged_page_out_of_range_is_flagged():
    """A page-table entry whose page lies outside the pool reads as zeros and sets
    PKV_DERR_SLOT_RANGE (the kernel's own bounds check; nothing outside the pool is read)."""
    pkv, _ = _pkv()
    w = W.batched_decode(seed=65, n_req=4, prefix=40, lo=5, hi=20, num_slots=1024)
    pc, calls = run_step(w, cascade=False, page_size=16)
    c = calls["decode"]
    c.batch.req_to_token[0, 0] = 1024 // 16        # one past the last page
    c.workspace.zero_()
    c.attend()
    torch.cuda.synchronize()
    assert pkv.get_device_error(c.workspace) & 0x100


def test_pipelined_end_to_end_gives_the_device_outputs():
    """The bench's end-to-end loop (inputs copied in and outputs copied out on their own
    streams while the neighbouring step computes, two buffer sets) returns exactly the
    outputs of a plain device run."""
    from prefix_shared_kv_token_gb300.runtime import run_e2e_pipelined
    w = W.tot_mixed(seed=45, root_len=300, depth=2, branch=3, seg=40, n_new_branches=2, num_slots=8000)
    _, calls = run_step(w)
    ref = {k: c.o.cpu().clone() for k, c in calls.items()}
    cl = list(calls.values())
    for c in cl:
        c.pin_host()
        c.host["o"].zero_()
    sets = [c.e2e_sets(2) for c in cl]
    ms = run_e2e_pipelined(sets, 5)
    assert ms > 0
    for c in cl:
        assert torch.equal(c.host["o"], ref[c.kind]), c.kind


def test_decode_graph_replay_matches_the_call():
    """A decode call captured once into a CUDA graph and replayed gives the call's outputs
    (bit for bit), and replays again on the same workspace."""
    w = W.batched_decode(seed=67, n_req=30, prefix=400, lo=10, hi=300, num_slots=1 << 15)
    _, calls = run_step(w)
    c = calls["decode"]
    first = c.o.clone()
    c.capture_attend()
    for _ in range(3):
        c.o.zero_()
        c.replay_attend()
        torch.cuda.synchronize()
        assert torch.equal(c.o, first)
    check_outputs(w, calls)


@pytest.mark.parametrize("hq,hkv,d,suffix,n_req", [
    (32, 8, 128, 70, 9),    # G 4: 6 last tokens per request, packed 4 + 4 (+ 1 alone)
    (32, 8, 128, 65, 4),    # 1 last token each
    (64, 8, 128, 66, 5),    # G 8: 2 last tokens (4-token row groups)
    (16, 8, 64, 140, 3),    # G 2: 12 last tokens (16-token row groups)
    (16, 16, 128, 20, 6),   # G 1: a whole 20-token suffix per row group
])
def test_extend_packed_last_tokens(hq, hkv, d, suffix, n_req):
    """Requests sharing a cached prefix whose last few new tokens are packed, a 32-row group
    each, into shared query tiles (each group also sees only its own remaining keys)."""
    w = W.fewshot_extend(seed=68 + suffix, n_req=n_req, prefix=300, suffix=suffix, hq=hq, hkv=hkv, d=d,
                         num_slots=8192)
    _, calls = run_step(w)
    assert int(calls["extend"].plan.info.offsets[14]) >= 1     # packed tiles were planned
    check_outputs(w, calls)


# ------------------------------------------------------------------------------ pool layouts

@pytest.mark.parametrize("dtype", ["bf16", "fp8_e4m3"])
@pytest.mark.parametrize("page", [1, 16])
def test_interleaved_and_separate_pools_give_identical_results(dtype, page):
    # the same step with a slot's K and V rows adjacent (one copy per key in decode) and in two
    # dense arrays: the kernels do the same arithmetic, so outputs and stored rows match bit
    # for bit, and both match the oracle
    pkv, PrefixCache = _pkv()
    w = W.tot_mixed(seed=39, root_len=600, depth=2, branch=4, seg=160, n_new_branches=3, num_slots=16384,
                    dtype=dtype)
    outs = {}
    for layout in ("interleaved", "separate"):
        pc = PrefixCache(w, page_size=page, kv_layout=layout)
        assert pc.pool.layout == layout
        pc.populate()
        calls = {k: pc.prepare(k) for k in ("extend", "decode")}
        for c in calls.values():
            c.run()
        torch.cuda.synchronize()
        for c in calls.values():
            assert pkv.get_device_error(c.workspace) == 0
        check_outputs(w, calls)
        check_pool(w, pc)
        outs[layout] = {k: c.o.clone() for k, c in calls.items()}
    for k in outs["separate"]:
        assert torch.equal(outs["interleaved"][k], outs["separate"][k]), k


@pytest.mark.parametrize("dtype,page,cascade", [("bf16", 1, True), ("bf16", 1, False), ("fp8_e4m3", 1, True),
                                                ("bf16", 16, True)])
def test_fused_store_extend_equals_store_then_extend(dtype, page, cascade):
    # kv_store + attn_extend as one call (the new rows stored into the pool and straight into
    # their gathered rows) against the separate store and the gather of every position:
    # outputs and pool rows bit for bit, both against the oracle
    pkv, PrefixCache = _pkv()
    w = W.fewshot_extend(seed=41, n_req=7, prefix=333, suffix=150, num_slots=8192, dtype=dtype)
    res = {}
    for fused in (True, False):
        pc = PrefixCache(w, page_size=page, fuse_store=fused)
        pc.populate()
        c = pc.prepare("extend", cascade=cascade)
        assert c.fused == fused and int(c.plan.info.offsets[16]) == (2 if fused else 0)
        c.run()
        torch.cuda.synchronize()
        assert pkv.get_device_error(c.workspace) == 0
        check_outputs(w, {"extend": c})
        check_pool(w, pc)
        idx = c.out_cache_loc.long()
        res[fused] = (c.o.clone(), pc.pool.k[idx].clone(), pc.pool.v[idx].clone())
    for a, b in zip(res[True], res[False]):
        assert torch.equal(a, b)
