"""Failure detection on the GPU without a fault: the bounded wait every kernel
uses gives up on a barrier nothing arrives on, records PA_ERR_TIMEOUT, and the
context stays usable for the next launch."""

import time

import pytest
import torch

from gpu_util import assert_matches_oracle, device_tables, oracle_decode
from workloads import tiny_decode

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_reports(lib):
    from paged_kv_cache_317_gb300 import binding as B
    rec = B.new_error_record()
    t0 = time.perf_counter()
    B.pa_selftest_bounded_wait(rec, arrive=False, limit_ns=2_000_000)   # 2 ms, nothing arrives
    assert B.pa_error_read(rec) == [B.STATUS_CODE["PA_ERR_TIMEOUT"], 1, 0, 0]
    assert time.perf_counter() - t0 < 5.0
    B.pa_error_clear(rec)
    B.pa_selftest_bounded_wait(rec, arrive=True, limit_ns=2_000_000)    # the phase completes
    assert B.pa_error_read(rec) == [0, 0, 0, 0]
    # the context is still usable: a decode runs and matches the oracle
    b = tiny_decode(seed=1, device="cuda", with_append=False)
    bt, sl = device_tables(b)
    out = B.paged_attn_decode(b.q, b.k_cache, b.v_cache, bt, sl, b.scale, error_record=rec)
    torch.cuda.synchronize()
    assert B.pa_error_read(rec) == [0, 0, 0, 0]
    assert_matches_oracle(out, oracle_decode(b), "decode after a timeout")


def test_selftest_rejects_bad_limits(lib):
    from paged_kv_cache_317_gb300 import binding as B
    rec = B.new_error_record()
    for bad in (0, 2_000_000_000):
        with pytest.raises(B.PagedKVError):
            B.pa_selftest_bounded_wait(rec, arrive=False, limit_ns=bad)
