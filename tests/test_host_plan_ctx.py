"""Context-buffer extend plans (chunked prefill over a caller-kept context buffer), on the host:
every query token attends to exactly the rows of its own request's positions 0..its own
position, found at ctx_row0[r] + position; nothing is gathered; the new tokens' rows are
listed for the store in q order; bad row layouts are rejected."""

import numpy as np
import pytest

import prefix_shared_kv_token_gb300 as pkv

EXT = np.dtype([("g", "<i4"), ("tok0", "<i4"), ("ntok", "<i4"), ("qpos0", "<i4"), ("pos0", "<i4"),
                ("nseg", "<i4"), ("rec", "<i4"), ("flags", "<i4"), ("key0", "<i4", 4), ("nkeys", "<i4", 4)])


def _sections(plan, dtype, n, off):
    return np.frombuffer(plan.blob[off:off + n * dtype.itemsize].tobytes(), dtype=dtype)


@pytest.mark.parametrize("hq,hkv", [(32, 8), (8, 8), (16, 2)])
def test_ctx_plan_covers_each_request_through_its_rows(hq, hkv):
    # three requests extending chunks after 0, 512 and 1000 cached positions; rows laid out
    # with gaps (room for later chunks) and not in request order
    pre = np.array([0, 512, 1000], np.int32)
    ext = np.array([256, 300, 17], np.int32)
    seq = pre + ext
    qo = np.concatenate([[0], np.cumsum(ext)]).astype(np.int32)
    row0 = np.array([5000, 0, 2000], np.int32)
    rows = 6000
    plan = pkv.plan_extend_ctx(seq, ext, qo, row0, rows, hq, hkv, 128)
    info = plan.info
    assert info.op == 2 and int(info.offsets[16]) == 1 and int(info.offsets[6]) == rows
    assert int(info.offsets[5]) == 0                    # no gather
    assert int(info.workspace_bytes) == 256            # header only: no records, no gathered keys
    T = int(qo[-1])
    tok_row = np.frombuffer(plan.blob[info.offsets[15]:info.offsets[15] + 4 * T].tobytes(), np.int32)
    want_rows = np.concatenate([row0[r] + np.arange(pre[r], seq[r]) for r in range(3)])
    assert np.array_equal(tok_row, want_rows)
    items = _sections(plan, EXT, info.num_items, info.offsets[0])
    req_of_tok = np.repeat(np.arange(3), ext)
    pos_of_tok = np.concatenate([np.arange(pre[r], seq[r]) for r in range(3)])
    cover = np.zeros((T, hkv, rows), np.int32)
    for it in items:
        assert it["nseg"] == 1 and it["rec"] == -1 and not (it["flags"] & 4)
        for t in range(it["ntok"]):
            tok = it["tok0"] + t
            r = req_of_tok[tok]
            assert it["key0"][0] == row0[r] and it["pos0"] == 0
            for k in range(it["nkeys"][0]):
                if k <= it["qpos0"] + t:
                    cover[tok, it["g"], it["key0"][0] + k] += 1
    for tok in range(T):
        r = req_of_tok[tok]
        want = np.zeros(rows, np.int32)
        want[row0[r]:row0[r] + pos_of_tok[tok] + 1] = 1
        for g in range(hkv):
            assert np.array_equal(cover[tok, g], want), (tok, g)


def test_ctx_plan_rejects_bad_row_layouts():
    seq = np.array([100, 100], np.int32)
    ext = np.array([10, 10], np.int32)
    qo = np.array([0, 10, 20], np.int32)
    with pytest.raises(pkv.PkvError):            # rows of the two requests overlap
        pkv.plan_extend_ctx(seq, ext, qo, np.array([0, 50], np.int32), 1000, 32, 8, 128)
    with pytest.raises(pkv.PkvError):            # past the end of the arrays
        pkv.plan_extend_ctx(seq, ext, qo, np.array([0, 950], np.int32), 1000, 32, 8, 128)
    with pytest.raises(pkv.PkvError):            # negative row
        pkv.plan_extend_ctx(seq, ext, qo, np.array([-1, 200], np.int32), 1000, 32, 8, 128)
    pkv.plan_extend_ctx(seq, ext, qo, np.array([0, 100], np.int32), 200, 32, 8, 128)   # exactly fits
