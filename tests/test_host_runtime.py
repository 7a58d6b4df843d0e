"""Host half of the runtime (no GPU): planning a call's tables and timing it leaves the cache
holding what it held -- same nodes, tokens, slots and locks, same free slots (only access
times and hit counts move, as any match moves them) -- so the bench can report the host
planning cost of a step without disturbing the calls it times."""

import numpy as np
import pytest

import workloads as W


def _cache_without_device(w):
    """A PrefixCache whose tree and allocator hold every request's cached part (as populate()
    leaves them), with a host-memory pool: nothing is stored, only the host state is built."""
    from prefix_shared_kv_token_gb300.runtime import PrefixCache, _ctx_tokens
    pc = PrefixCache(w, device="cpu")
    for r in w.requests:
        toks = _ctx_tokens(w, r)
        c = len(toks) - r.n_new
        vals, _ = pc.tree.match_prefix(toks[:c])
        new = pc._extend_slots(vals, c - len(vals))
        assert pc.tree.insert(toks[:c], np.concatenate([vals, new]).astype(np.int32)) == len(vals)
    return pc


@pytest.mark.parametrize("kind,make", [
    ("extend", lambda: W.fewshot_extend(seed=2, n_req=6, prefix=100, suffix=20, num_slots=4096)),
    ("decode", lambda: W.batched_decode(seed=3, n_req=9, prefix=80, lo=5, hi=40, num_slots=4096)),
])
def test_host_step_timing_leaves_the_cache_unchanged(kind, make):
    w = make()
    pc = _cache_without_device(w)
    def structure():   # (id, parent, lock_ref, key, value, children, priority): no access time or hits
        return [(n[0], n[1], n[2], n[4], n[5], n[6], n[8]) for n in pc.tree.dump()]

    before_tree = structure()
    before_free = pc.alloc.available
    ms = pc.host_step_ms(kind, reps=3)
    assert ms > 0
    assert structure() == before_tree             # no lock or split left behind...
    assert pc.alloc.available == before_free      # ...and every slot given back


def test_plan_host_tables_match_the_tree():
    w = W.batched_decode(seed=5, n_req=7, prefix=64, lo=3, hi=30, num_slots=2048)
    pc = _cache_without_device(w)
    h = pc._plan_host("decode", True, None, 2, None)
    for r, row, s in zip(h["reqs"], h["rows"], h["seq"]):
        assert len(row) == s == w.context_len(r)
    # the slot check ran: the new slots are distinct and inside the pool
    import prefix_shared_kv_token_gb300 as pkv
    assert pkv.check_out_cache_loc(h["loc"], w.num_slots) == -1
    assert h["cascade"] is not None and h["cascade"].num_spans >= 1
