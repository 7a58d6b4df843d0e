"""Failure detection on the GPU without a fault: every wait inside the attention kernels is
bounded, and pkv_set_wait_limit_ns makes that bound short enough that the waits give up.
The kernels must then record PKV_DERR_TIMEOUT in the error word, let their copies and MMAs
in flight land, free their tensor memory and return -- the call completes, the context stays
usable, and the next call with the default limit matches the oracle again.

No wait is starved on purpose here: the kernels run their normal pipelines and only the
limit is cut, so the first wait that does not succeed at once gives up."""

import numpy as np
import pytest
import torch

import workloads as W
from oracle import step as ostep

pytestmark = pytest.mark.gpu

TOL = {"bf16": 1e-2, "fp8_e4m3": 5e-2}
DERR_TIMEOUT = 0x200


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.fixture(autouse=True)
def _default_limit_after():
    yield
    import prefix_shared_kv_token_gb300 as pkv
    pkv.set_wait_limit_ns(0)


def _workloads():
    return {
        # extend: gather + tcgen05 extend kernel (two-tile, split and packed items) + merge
        "extend": W.fewshot_extend(seed=91, n_req=6, prefix=300, suffix=150, num_slots=8192),
        # decode: tensor-core span pass (a 700-key prefix shared by 40 requests), precise
        # items for the short contexts, the persistent bulk-copy decode kernel, the merge
        "decode": W.batched_decode(seed=92, n_req=40, prefix=700, lo=1, hi=300, num_slots=40000),
        # fp8 pool, both kinds in one step
        "fp8": W.tot_mixed(seed=93, root_len=512, depth=2, branch=3, seg=128, n_new_branches=3, num_slots=8192),
    }


@pytest.mark.parametrize("name", ["extend", "decode", "fp8"])
def test_short_wait_limit_gives_up_and_the_next_call_is_exact(name):
    import prefix_shared_kv_token_gb300 as pkv
    from prefix_shared_kv_token_gb300.runtime import PrefixCache

    w = _workloads()[name]
    pc = PrefixCache(w)
    pc.populate()
    calls = [pc.prepare(k) for k in ("extend", "decode") if any(r.kind == k for r in w.requests)]
    for c in calls:
        c.store()
    torch.cuda.synchronize()
    assert pkv.get_device_error(pc.err) == 0

    pkv.set_wait_limit_ns(1)
    assert pkv.get_wait_limit_ns() == 1
    for c in calls:
        c.attend()
    torch.cuda.synchronize()               # the kernels returned on their own
    pkv.set_wait_limit_ns(0)
    for c in calls:
        word = pkv.get_device_error(c.workspace)
        assert word & DERR_TIMEOUT, (c.kind, hex(word))

    # the context is still usable: a clean workspace and the default limit give exact results
    for c in calls:
        c.workspace.zero_()
        c.o.zero_()
        c.attend()
    torch.cuda.synchronize()
    for c in calls:
        assert pkv.get_device_error(c.workspace) == 0
        want = ostep.expected_outputs(w, c.kind)
        got = c.o.float().cpu().numpy().astype(np.float64)
        err = float(np.max(np.abs(got - want)))
        assert err <= TOL[w.dtype], (c.kind, err)
