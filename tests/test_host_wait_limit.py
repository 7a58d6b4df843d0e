"""The wait-limit hook of the attention kernels (host side): the value set is the value the
next launches get, and 0 restores the 2 s default."""

import prefix_shared_kv_token_gb300 as pkv


def test_wait_limit_set_get_and_default():
    assert pkv.get_wait_limit_ns() == 2_000_000_000
    try:
        pkv.set_wait_limit_ns(1)
        assert pkv.get_wait_limit_ns() == 1
        pkv.set_wait_limit_ns(5_000_000_000)
        assert pkv.get_wait_limit_ns() == 5_000_000_000
    finally:
        pkv.set_wait_limit_ns(0)
    assert pkv.get_wait_limit_ns() == 2_000_000_000
