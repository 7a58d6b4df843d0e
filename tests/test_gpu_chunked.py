"""Chunked prefill and multi-layer pools on the GPU, against the oracle.

A long prompt is extended chunk by chunk, each chunk over the chunks before it, which the
radix tree has cached by then ("Efficiently Programming Large Language Models using SGLang"
summary, §RadixAttention: only the uncached remainder is prefilled).  Every chunk's outputs
must equal the plain causal attention over the whole prompt (the oracle never looks at
chunks, slots or tables).  A model has one pool per layer: the same tables, slots and plan
serve every layer, each with its own K/V and queries.
"""

import numpy as np
import pytest
import torch

import workloads as W
from oracle import step as ostep

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _run(calls):
    import prefix_shared_kv_token_gb300 as pkv
    for c in calls:
        c.run()
    torch.cuda.synchronize()
    for c in calls:
        assert pkv.get_device_error(c.workspace) == 0


def _check(w, call, tol=1e-2):
    got = call.o.float().cpu().numpy().astype(np.float64)
    want = np.concatenate([ostep.request_output(w, r)[0] for r in call.requests])
    err = np.max(np.abs(got - want))
    assert err <= tol, err


def _check_pool_and_context(w, pc):
    """Every prompt's pool rows equal the oracle's store of its K/V, bit for bit; with a
    context buffer, the prompt's context rows hold exactly the values the pool holds (bf16
    bits, or the fp8 code converted to bf16)."""
    from oracle.fp8 import e4m3_decode, quantize_to_pool
    last = {}
    for r in w.requests:
        if r.path[0] not in last or w.context_len(r) > w.context_len(last[r.path[0]]):
            last[r.path[0]] = r
    for root, r in last.items():
        toks = W.context_tokens(w, r)
        vals, _ = pc.tree.match_prefix(toks)
        assert len(vals) == len(toks)
        kb, vb = W.context_kv_bits(w, r)
        idx = torch.from_numpy(vals.astype(np.int64)).cuda()
        for pool_t, bits, scale, name in ((pc.pool.k, kb, w.k_scale, "k"), (pc.pool.v, vb, w.v_scale, "v")):
            got = pool_t[idx].cpu()
            if w.dtype == "bf16":
                want_pool = bits
                assert np.array_equal(got.view(torch.int16).numpy().view(np.uint16), want_pool)
                want_ctx = want_pool
            else:
                codes = quantize_to_pool(W.bf16_bits_to_f64(bits), scale)
                assert np.array_equal(got.numpy(), codes)
                # every e4m3 value is a bf16 value: the cast is exact
                want_ctx = torch.from_numpy(e4m3_decode(codes).astype(np.float32)).to(torch.bfloat16) \
                    .view(torch.int16).numpy().view(np.uint16)
            if pc.ctx is not None:
                r0 = pc.ctx["row0"][root]
                ctx = pc.ctx[name][r0:r0 + len(toks)].cpu().view(torch.int16).numpy().view(np.uint16)
                assert np.array_equal(ctx, want_ctx), name


@pytest.mark.parametrize("fused", [True, False])
@pytest.mark.parametrize("prompt,chunk", [(1000, 256), (700, 700), (513, 128)])
def test_chunked_prefill_matches_oracle(prompt, chunk, fused):
    from prefix_shared_kv_token_gb300.runtime import PrefixCache
    w = W.chunked_prefill(seed=61, n_req=3, prompt=prompt, chunk=chunk, num_slots=8000)
    pc = PrefixCache(w)
    calls = pc.prepare_chunked(fused=fused)
    assert len(calls) == -(-prompt // chunk)
    assert all((c.ctx is not None) == fused for c in calls)
    _run(calls)
    for c in calls:
        _check(w, c)
    # the whole prompts are cached afterwards, in the pool and (fused) in the context buffer
    for r in w.requests:
        if w.meta["chunk"][r.rid] == len(calls) - 1:
            vals, _ = pc.tree.match_prefix(W.context_tokens(w, r))
            assert len(vals) == prompt
    _check_pool_and_context(w, pc)


@pytest.mark.parametrize("fused", [True, False])
def test_chunked_prefill_fp8(fused):
    from prefix_shared_kv_token_gb300.runtime import PrefixCache
    w = W.chunked_prefill(seed=63, n_req=2, prompt=600, chunk=200, num_slots=4000, dtype="fp8_e4m3")
    pc = PrefixCache(w)
    calls = pc.prepare_chunked(fused=fused)
    _run(calls)
    for c in calls:
        _check(w, c, tol=5e-2)
    _check_pool_and_context(w, pc)


def test_fused_chunk_reports_a_bad_slot_without_writing():
    import prefix_shared_kv_token_gb300 as pkv
    from prefix_shared_kv_token_gb300.runtime import PrefixCache
    w = W.chunked_prefill(seed=64, n_req=1, prompt=300, chunk=150, num_slots=2000)
    pc = PrefixCache(w)
    calls = pc.prepare_chunked(fused=True)
    c = calls[0]
    c.out_cache_loc[3] = w.num_slots + 5          # host-made bad slot: skipped and reported
    c.attend()
    torch.cuda.synchronize()
    assert pkv.get_device_error(c.workspace) & 0x100


@pytest.mark.parametrize("fused", [True, False])
def test_multi_layer_pools_share_tables_and_plan(fused):
    from prefix_shared_kv_token_gb300 import Pool
    from prefix_shared_kv_token_gb300.runtime import PrefixCache
    layers = [W.chunked_prefill(seed=70 + l, n_req=2, prompt=500, chunk=250, num_slots=3000) for l in range(3)]
    pc = PrefixCache(layers[0])
    base = pc.prepare_chunked(fused=fused)
    pools = [pc.pool] + [Pool.allocate(w.num_slots, w.num_kv_heads, w.head_dim, w.dtype, w.k_scale, w.v_scale, "cuda")
                         for w in layers[1:]]
    # each layer keeps its own context arrays (fused), shared by that layer's chunks
    ctxs = [None if not fused else (torch.zeros_like(pc.ctx["k"]), torch.zeros_like(pc.ctx["v"])) for _ in layers]
    per_layer = [[c if l == 0 else c.layer(pools[l], layers[l], ctx=ctxs[l]) for c in base] for l in range(3)]
    for step in range(len(base)):                  # a forward pass: every layer, step by step
        _run([per_layer[l][step] for l in range(3)])
    for l in range(3):
        for c in per_layer[l]:
            _check(layers[l], c)
        assert per_layer[l][0].plan is base[0].plan   # one plan for all layers


@pytest.mark.parametrize("path", ["context_buffer", "fused_store"])
def test_store_reports_an_out_of_range_row_without_writing_it(path):
    # The store of a context-buffer or fused-store call writes each new token's K/V to the
    # pool and to row tok_row[token] of the context / gathered arrays.  A host-made row past
    # those arrays must be reported (PKV_DERR_POSITION, header words = token and row) and its
    # copy skipped; the pool rows are still stored.
    import prefix_shared_kv_token_gb300 as pkv
    from prefix_shared_kv_token_gb300.runtime import PrefixCache
    if path == "context_buffer":
        w = W.chunked_prefill(seed=66, n_req=1, prompt=300, chunk=150, num_slots=2000)
        pc = PrefixCache(w)
        c = pc.prepare_chunked(fused=True)[0]
        rows = int(c.ctx[0].shape[0])
        before = c.ctx[0].clone()
    else:
        w = W.fewshot_extend(seed=67, n_req=3, prefix=200, suffix=40, num_slots=4096)
        pc = PrefixCache(w, fuse_store=True)
        pc.populate()
        c = pc.prepare("extend", cascade=True)
        assert c.fused
        rows = int(c.plan.info.offsets[6])
    tok, bad = 3, rows + 7
    at = int(c.plan.info.offsets[15]) + 4 * tok
    c.plan_dev[at:at + 4] = torch.tensor([bad], dtype=torch.int32).view(torch.uint8).to(c.plan_dev.device)
    c.workspace.zero_()
    c.attend()
    torch.cuda.synchronize()
    words = c.workspace[:4].view(torch.int32).cpu().tolist()
    assert words[0] == 0x400 and words[1] == tok and words[2] == bad, words
    assert pkv.get_device_error(c.workspace) == 0x400
    # the token's pool rows were stored (bf16: the new rows themselves)
    slot = int(c.out_cache_loc[tok])
    assert torch.equal(pc.pool.k[slot].view(torch.int16).cpu(), c.k_new[tok].view(torch.int16).cpu())
    assert torch.equal(pc.pool.v[slot].view(torch.int16).cpu(), c.v_new[tok].view(torch.int16).cpu())
    if path == "context_buffer":
        # no context row was written for it: its own row keeps what it held before
        ok = int(torch.from_numpy(c.plan.blob[int(c.plan.info.offsets[15]):][:4 * (tok + 1)].copy())
                 .view(torch.int32)[tok])
        assert torch.equal(c.ctx[0][ok], before[ok])
