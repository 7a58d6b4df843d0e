"""Test helper: the oracle's per-request outputs of a full-size workload, computed by a pool of
worker processes (spawn: safe after the parent has used the GPU).  Each worker rebuilds the
workload from its seed -- the generators are deterministic -- and runs oracle.step on its share
of the requests.  Test infrastructure only."""

from __future__ import annotations

import multiprocessing as mp
import os

_CACHE = {}


def _work(task):
    cfg, rids = task
    import workloads as W
    from oracle import step as ostep
    if cfg not in _CACHE:
        _CACHE.clear()
        _CACHE[cfg] = W.config(cfg)
    w = _CACHE[cfg]
    by_id = {r.rid: r for r in w.requests}
    return [(rid, ostep.request_output(w, by_id[rid])[0]) for rid in rids]


def outputs_by_request(cfg, rids, procs=None):
    """{request id: oracle output [n_q, Hq, d]} for configuration ``cfg``'s listed requests."""
    procs = procs or max(1, min(16, (os.cpu_count() or 1)))
    rids = list(rids)
    chunks = [rids[i::procs] for i in range(procs) if rids[i::procs]]
    with mp.get_context("spawn").Pool(len(chunks)) as pool:
        parts = pool.map(_work, [(cfg, c) for c in chunks])
    return {rid: o for part in parts for rid, o in part}
