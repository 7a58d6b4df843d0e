"""Multi-step serving on the GPU (cache-aware admission, LRU eviction under memory pressure,
prefill and decode steps, decode plans reused across steps), every attention output of every
step checked against the oracle.

The oracle recomputes each query from its context alone -- the tokens and positions, whose
K/V the seeded generator defines -- so it never sees slots, tables, the tree, the scheduler
or eviction.  A wrong slot anywhere (an evicted entry reused while still referenced, a
duplicate released too early, a stale table row) changes an output.
"""

import numpy as np
import pytest
import torch

import workloads as W
from oracle.attention import attend, bf16_to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _check_records(stream, records, tol=1e-2):
    s = stream
    worst = 0.0
    for rec in records:
        got = rec.o.float().cpu().numpy().astype(np.float64)
        row = 0
        for rid, poss, ctx in zip(rec.rids, rec.positions, rec.contexts):
            L = poss[-1] + 1
            k, v = W.token_kv(s.seed, ctx[:L], range(L), s.num_kv_heads, s.head_dim)
            q = np.stack([W.stream_query(s.seed, rid, p, s.num_q_heads, s.head_dim) for p in poss])
            want, _ = attend(bf16_to_f64(q), bf16_to_f64(k), bf16_to_f64(v), s.sm_scale, np.asarray(poss))
            err = np.max(np.abs(got[row:row + len(poss)] - want))
            worst = max(worst, err)
            row += len(poss)
        assert row == got.shape[0]
    assert worst <= tol, worst
    return worst


@pytest.mark.parametrize("policy", ["lpm", "fcfs"])
def test_serving_steps_match_oracle_under_eviction(policy):
    from prefix_shared_kv_token_gb300.serving import ServingSim
    s = W.serving_stream(seed=81, n_groups=3, per_group=6, shared=200, unique=(10, 40), out=(2, 6), per_step=4,
                         hq=8, hkv=2, d=64)
    total = sum(len(r.prompt) + r.out_len for r in s.requests)
    sim = ServingSim(s, capacity=900, policy=policy, max_running=6, prefill_budget=600, record=True)
    sim.run()
    st = sim.summary()
    assert sim.done() and st["finished"] == len(s.requests)
    assert total > 900 and st["evicted_tokens"] > 0           # the pool was too small: eviction ran
    assert st["cached_tokens"] > 0 and st["plans"] < st["steps"]  # prefix hits; plans were reused
    _check_records(s, sim.records)


def test_longest_prefix_first_hits_more_than_fcfs():
    # all 32 requests wait from step 0; 4 run at a time; the pool holds about two prompts'
    # worth of uncached tokens, so admitting by cached prefix keeps a group's prefix in use
    # while arrival order (groups interleaved) evicts and recomputes prefixes
    from prefix_shared_kv_token_gb300.serving import ServingSim
    s = W.serving_stream(seed=82, n_groups=4, per_group=8, shared=300, unique=(10, 30), out=(2, 4), per_step=32,
                         hq=8, hkv=2, d=64)
    st = {}
    for policy in ("lpm", "fcfs"):
        sim = ServingSim(s, capacity=800, policy=policy, max_running=4, prefill_budget=2000)
        sim.run()
        st[policy] = sim.summary()
        assert st[policy]["finished"] == len(s.requests)
    assert st["lpm"]["hit_rate"] > st["fcfs"]["hit_rate"], st
    assert st["lpm"]["prefill_tokens"] < st["fcfs"]["prefill_tokens"], st


@pytest.mark.parametrize("page", [4, 16])
def test_paged_serving_steps_match_oracle_under_eviction(page):
    """The same serving loop over a paged pool (whole blocks cached, page tables, partial
    blocks private and freed at finish): every output still matches the oracle."""
    from prefix_shared_kv_token_gb300.serving import ServingSim
    s = W.serving_stream(seed=83, n_groups=3, per_group=6, shared=200, unique=(10, 40), out=(2, 6), per_step=4,
                         hq=8, hkv=2, d=64)
    sim = ServingSim(s, capacity=1024, policy="lpm", max_running=6, prefill_budget=600, record=True,
                     page_size=page)
    sim.run()
    st = sim.summary()
    assert sim.done() and st["finished"] == len(s.requests)
    assert st["evicted_tokens"] > 0 and st["cached_tokens"] > 0
    assert st["cached_tokens"] % page == 0          # every hit is whole blocks
    _check_records(s, sim.records)
    # every page is back in the free list or held by the tree
    assert sim.alloc.available * page + sim.tree.sizes()["total"] == 1024
