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


@pytest.mark.parametrize("prompt,chunk", [(1000, 256), (700, 700), (513, 128)])
def test_chunked_prefill_matches_oracle(prompt, chunk):
    from prefix_shared_kv_token_gb300.runtime import PrefixCache
    w = W.chunked_prefill(seed=61, n_req=3, prompt=prompt, chunk=chunk, num_slots=8000)
    pc = PrefixCache(w)
    calls = pc.prepare_chunked()
    assert len(calls) == -(-prompt // chunk)
    _run(calls)
    for c in calls:
        _check(w, c)
    # the whole prompts are cached afterwards
    for r in w.requests:
        if w.meta["chunk"][r.rid] == len(calls) - 1:
            vals, _ = pc.tree.match_prefix(W.context_tokens(w, r))
            assert len(vals) == prompt


def test_chunked_prefill_fp8():
    from prefix_shared_kv_token_gb300.runtime import PrefixCache
    w = W.chunked_prefill(seed=63, n_req=2, prompt=600, chunk=200, num_slots=4000, dtype="fp8_e4m3")
    pc = PrefixCache(w)
    calls = pc.prepare_chunked()
    _run(calls)
    for c in calls:
        _check(w, c, tol=5e-2)


def test_multi_layer_pools_share_tables_and_plan():
    from prefix_shared_kv_token_gb300 import Pool
    from prefix_shared_kv_token_gb300.runtime import PrefixCache
    layers = [W.chunked_prefill(seed=70 + l, n_req=2, prompt=500, chunk=250, num_slots=3000) for l in range(3)]
    pc = PrefixCache(layers[0])
    base = pc.prepare_chunked()
    pools = [pc.pool] + [Pool.allocate(w.num_slots, w.num_kv_heads, w.head_dim, w.dtype, w.k_scale, w.v_scale, "cuda")
                         for w in layers[1:]]
    per_layer = [[c if l == 0 else c.layer(pools[l], layers[l]) for c in base] for l in range(3)]
    for step in range(len(base)):                  # a forward pass: every layer, step by step
        _run([per_layer[l][step] for l in range(3)])
    for l in range(3):
        for c in per_layer[l]:
            _check(layers[l], c)
        assert per_layer[l][0].plan is base[0].plan   # one plan for all layers
