"""pkv_attn_decode_noalloc: the decode entry point for callers that cannot allocate device
memory -- a serving loop that froze its device-memory budget after start-up, or a host
program embedding the library without a device allocator of its own.  Its scratch is a fixed
array inside the library.  Called through the C ABI on two calls in a row, it must give
bit-for-bit the output of pkv_attn_decode with a caller-provided workspace (same plan, same
kernels), leave its error word clear, and match the oracle within the bf16 tolerance.

This file is collected last on purpose: if it fails, a run that stops at the first failure
has already run every other test.  It also passes on its own in a fresh process.
"""

import ctypes as C

import numpy as np
import pytest
import torch

import workloads as W
from oracle import step as ostep

pytestmark = pytest.mark.gpu

TOL_BF16 = 1e-2


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
    want = ostep.expected_outputs(w, "decode")
    assert float(np.max(np.abs(ref.float().cpu().numpy() - want))) <= TOL_BF16

    pool, batch = call.pool.c(), call.batch.c()
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(2):
        out = torch.full_like(call.o, float("nan"))
        rc = _lib.lib.pkv_attn_decode_noalloc(C.byref(pool), C.byref(batch), call.q.data_ptr(), out.data_ptr(),
                                              C.c_float(call.sm_scale), C.byref(call.plan.info),
                                              call.plan_dev.data_ptr(), stream)
        assert rc == 0, _lib.ERRORS.get(rc, rc)
        raw = C.c_int32(-1)
        rc = _lib.lib.pkv_get_noalloc_device_error(stream, C.byref(raw))   # synchronises the stream
        assert rc == 0 and raw.value == 0, (rc, raw.value)
        assert torch.equal(out, ref)             # same plan and kernels: identical bits
        err = float(np.max(np.abs(out.float().cpu().numpy() - want)))
        assert err <= TOL_BF16, err


def test_noalloc_error_word_reports_a_bad_slot():
    import prefix_shared_kv_token_gb300 as pkv
    from prefix_shared_kv_token_gb300 import _lib
    from prefix_shared_kv_token_gb300.runtime import PrefixCache

    # a host-made table with one slot outside the pool: read as zeros and flagged, never faulted
    w = W.batched_decode(seed=78, n_req=3, prefix=40, lo=20, hi=60, num_slots=4096)
    pc = PrefixCache(w)
    pc.populate()
    call = pc.prepare("decode", cascade=False)
    call.run()
    torch.cuda.synchronize()
    assert pkv.get_device_error(call.workspace) == 0
    ref = call.o.clone()
    pool, batch = call.pool.c(), call.batch.c()
    stream = torch.cuda.current_stream().cuda_stream
    rt = call.batch.req_to_token
    good = int(rt[0, 5].item())

    def noalloc(out):
        return _lib.lib.pkv_attn_decode_noalloc(C.byref(pool), C.byref(batch), call.q.data_ptr(), out.data_ptr(),
                                                C.c_float(call.sm_scale), C.byref(call.plan.info),
                                                call.plan_dev.data_ptr(), stream)

    rt[0, 5] = w.num_slots + 7
    out = torch.empty_like(ref)
    assert noalloc(out) == 0
    assert pkv.get_noalloc_device_error() & 0x100   # PKV_DERR_SLOT_RANGE
    # the next call clears the word before it launches
    rt[0, 5] = good
    assert noalloc(out) == 0
    assert pkv.get_noalloc_device_error() == 0
    assert torch.equal(out, ref)


def test_noalloc_rejects_oversized_plan():
    from prefix_shared_kv_token_gb300 import _lib
    info = _lib.PkvPlanInfo()
    info.op = 1
    info.workspace_bytes = (32 << 20) + 1
    rc = _lib.lib.pkv_attn_decode_noalloc(None, None, None, None, C.c_float(1.0), C.byref(info), None, None)
    assert rc == -3   # PKV_E_WORKSPACE, nothing launched
