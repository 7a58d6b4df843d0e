"""pkv_attn_decode_noalloc: the decode entry point for callers that cannot allocate device
memory (its scratch is a fixed array inside the library), called through the C ABI and
checked against pkv_attn_decode with a caller-provided workspace, on two calls in a row.

This file is collected last on purpose: if it fails, a run that stops at the first failure
has already run every other test.  It also passes on its own in a fresh process.
"""

import ctypes as C

import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def test_noalloc_decode_matches_workspace_decode_twice():
    import prefix_shared_kv_token_gb300 as pkv
    from prefix_shared_kv_token_gb300 import _lib
    from prefix_shared_kv_token_gb300.runtime import PrefixCache

    # a cascade plan with split tails, so the partial-state records in scratch are used
    w = W.batched_decode(seed=77, n_req=11, prefix=300, lo=100, hi=700, num_slots=20000)
    pc = PrefixCache(w)
    pc.populate()
    call = pc.prepare("decode", cascade=True, opts={"chunk_keys": 128})
    assert call.plan.info.num_records > 0
    assert call.plan.info.workspace_bytes <= 32 << 20
    call.run()                                   # reference: caller-provided workspace
    torch.cuda.synchronize()
    assert pkv.get_device_error(call.workspace) == 0
    ref = call.o.clone()

    pool, batch = call.pool.c(), call.batch.c()
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(2):
        out = torch.full_like(call.o, float("nan"))
        rc = _lib.lib.pkv_attn_decode_noalloc(C.byref(pool), C.byref(batch), call.q.data_ptr(), out.data_ptr(),
                                              C.c_float(call.sm_scale), C.byref(call.plan.info),
                                              call.plan_dev.data_ptr(), stream)
        assert rc == 0, _lib.ERRORS.get(rc, rc)
        torch.cuda.synchronize()
        diff = (out.float() - ref.float()).abs().max().item()
        assert np.isfinite(diff) and diff <= 1e-2


def test_noalloc_rejects_oversized_plan():
    from prefix_shared_kv_token_gb300 import _lib
    info = _lib.PkvPlanInfo()
    info.op = 1
    info.workspace_bytes = (32 << 20) + 1
    rc = _lib.lib.pkv_attn_decode_noalloc(None, None, None, None, C.c_float(1.0), C.byref(info), None, None)
    assert rc == -3   # PKV_E_WORKSPACE, nothing launched
