"""Parity at the five workloads' full sizes, in the launch configuration bench.py times
(same PrefixCache / plan / kernels): sampled outputs against the oracle, computed one request
at a time, plus properties that hold at any size (finite outputs, clean error word, the
stored pool rows of sampled requests bit-exact)."""

import numpy as np
import pytest
import torch

import workloads as W
from oracle import step as ostep
from oracle.fp8 import quantize_to_pool

pytestmark = pytest.mark.gpu

TOL = {"bf16": 1e-2, "fp8_e4m3": 5e-2}


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("cfg,page", [(1, 1), (2, 1), (3, 1), (4, 1), (5, 1), (3, 16), (4, 16)])
def test_config_full_size(cfg, page):
    import prefix_shared_kv_token_gb300 as pkv
    from prefix_shared_kv_token_gb300.runtime import PrefixCache

    w = W.config(cfg)
    pc = PrefixCache(w, page_size=page)
    pc.populate()
    calls = {k: pc.prepare(k) for k in ("extend", "decode") if any(r.kind == k for r in w.requests)}
    for c in calls.values():
        c.run()
    # decode calls as the bench times them: replayed from a CUDA graph captured once
    if "decode" in calls:
        calls["decode"].capture_attend()
        calls["decode"].o.zero_()
        calls["decode"].replay_attend()
    torch.cuda.synchronize()
    rng = np.random.default_rng(100 + cfg)
    tol = TOL[w.dtype]
    for kind, c in calls.items():
        assert pkv.get_device_error(c.workspace) == 0
        got = c.o.float().cpu().numpy()
        assert np.all(np.isfinite(got))
        reqs = [r for r in w.requests if r.kind == kind]
        qo = np.concatenate([[0], np.cumsum([r.n_new if kind == "extend" else 1 for r in reqs])])
        picks = []
        for ri in rng.choice(len(reqs), size=min(len(reqs), 24), replace=False):
            nq = reqs[ri].n_new if kind == "extend" else 1
            qis = sorted(set(rng.integers(0, nq, size=min(nq, 3)).tolist()) | {nq - 1})
            picks += [(int(ri), qi) for qi in qis]
        want = ostep.expected_sample(w, kind, picks)
        err = max(float(np.max(np.abs(got[qo[ri] + qi] - want[(ri, qi)]))) for ri, qi in picks)
        assert err <= tol, (kind, err)
    # stored rows of a few requests' contexts, bit-exact
    for r in [w.requests[i] for i in rng.choice(len(w.requests), size=min(4, len(w.requests)), replace=False)]:
        toks = W.context_tokens(w, r)
        vals, _ = pc.tree.match_prefix(toks[:len(toks) - r.n_new])
        kb, vb = W.context_kv_bits(w, r)
        idx = torch.from_numpy(vals.astype(np.int64)).cuda()
        gk = pc.pool.k[idx].cpu()
        gv = pc.pool.v[idx].cpu()
        if w.dtype == "bf16":
            assert np.array_equal(gk.view(torch.int16).numpy().view(np.uint16), kb[:len(vals)])
            assert np.array_equal(gv.view(torch.int16).numpy().view(np.uint16), vb[:len(vals)])
        else:
            assert np.array_equal(gk.numpy(), quantize_to_pool(W.bf16_bits_to_f64(kb[:len(vals)]), w.k_scale))
            assert np.array_equal(gv.numpy(), quantize_to_pool(W.bf16_bits_to_f64(vb[:len(vals)]), w.v_scale))
