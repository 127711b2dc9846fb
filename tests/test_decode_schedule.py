"""Host-side decode schedule (pa_decode_partition_tokens, pa_decode_work_items):
pure host code, so it runs here without a GPU."""

import ctypes

import numpy as np
import pytest

from paged_kv_cache_317_gb300 import binding as B


def rule(lens, num_heads, heads_per_cta, num_sms):
    """The balance rule as the header states it."""
    G = heads_per_cta or (2 if num_heads % 2 == 0 else 1)
    work = int(np.sum(lens)) * (num_heads // G)
    longest = int(np.max(lens)) if len(lens) else 0
    for pt, c in ((512, 3.5), (256, 3.5), (128, 2.0)):
        if min(pt, longest) * num_sms * c <= work:
            return pt
    return 64


def test_partition_choice_follows_the_balance_rule():
    rng = np.random.default_rng(0)
    for trial in range(400):
        n = int(rng.integers(1, 300))
        median = float(np.exp(rng.uniform(np.log(8), np.log(20000))))
        lens = np.clip(np.round(np.exp(np.log(median) + 0.75 * rng.standard_normal(n))), 0, 1 << 17)
        H = int(rng.choice([8, 12, 32, 40, 64, 7]))
        G = int(rng.choice([0, 1]))
        sms = int(rng.choice([1, 76, 148, 152]))
        got = B.decode_partition_tokens(lens, H, G, sms)
        assert got == rule(lens, H, G, sms), (trial, n, median, H, G, sms)


def test_partition_choice_at_the_ends():
    big = np.full(256, 350)
    assert B.decode_partition_tokens(big, 40, 0, 152) == 512      # plenty of work per SM
    assert B.decode_partition_tokens([350], 40, 0, 152) == 64     # one short sequence
    assert B.decode_partition_tokens([1024] * 4, 40, 0, 152) == 128
    assert B.decode_partition_tokens([], 40, 0, 152) == 512       # nothing to balance
    # a long batch keeps 512 even with one huge sequence, since the heaviest
    # block is a partition, not the sequence
    assert B.decode_partition_tokens([100000] + [300] * 255, 40, 0, 152) == 512
    # the boundary itself: work exactly 3.5 x SMs x heaviest keeps the partition
    # (7 x 512 tokens x 2 heads = 3.5 x 4 SMs x 512)
    assert B.decode_partition_tokens([512] * 7, 2, 1, 4) == 512
    assert B.decode_partition_tokens([512] * 6, 2, 1, 4) == 256
    # 128 needs only half the work per SM: 2 x 4 SMs x 128 = 1024 = 4 x 128 x 2 heads
    assert B.decode_partition_tokens([128] * 4, 2, 1, 4) == 128
    assert B.decode_partition_tokens([128] * 3, 2, 1, 4) == 64


def test_partition_choice_rejects_bad_arguments():
    with pytest.raises(B.PagedKVError, match="INVALID_ARG"):
        B.decode_partition_tokens([5, -1], 40, 0, 152)
    with pytest.raises(B.PagedKVError, match="INVALID_ARG"):
        B.decode_partition_tokens([5], 40, 3, 152)                 # 3 does not divide 40
    with pytest.raises(B.PagedKVError, match="INVALID_ARG"):
        B.decode_partition_tokens([5], 32, 16, 152)                # above 8 heads per block
    with pytest.raises(B.PagedKVError, match="INVALID_ARG"):
        B.decode_partition_tokens([5], 0, 0, 152)
    with pytest.raises(B.PagedKVError, match="INVALID_ARG"):
        B.decode_partition_tokens([5], 8, 0, -1)


def _items_by_formula(lens, pt, MB, bs, order=None):
    lens = np.asarray(lens, np.int64)
    P = max(1, -(-MB * bs // pt))
    order = sorted(range(len(lens)), key=lambda i: (-lens[i], i)) if order is None else order
    return np.array([i * P + p for i in order for p in range(max(1, -(-int(lens[i]) // pt)))],
                    dtype=np.int32)


def test_work_items_match_their_definition():
    rng = np.random.default_rng(1)
    for trial in range(200):
        n = int(rng.integers(0, 60))
        bs = int(rng.choice([16, 32]))
        MB = int(rng.integers(1, 200))
        lens = rng.integers(0, MB * bs + 1, size=n)
        lens[rng.random(n) < 0.1] = 0
        pt = int(rng.choice([0, 16, 64, 128, 512, 2048]))
        order = None if trial % 3 else list(rng.permutation(n))
        got = B.partition_work_items(lens, pt, MB, bs, order=order)
        want = _items_by_formula(lens, pt or 512, MB, bs, order)
        assert got.dtype == np.int32
        assert np.array_equal(got, want), trial


def test_work_items_reject_bad_arguments():
    lib = B.load_library()
    lens = (ctypes.c_int32 * 3)(10, 40, 20)
    n = ctypes.c_int32(-1)
    buf = (ctypes.c_int32 * 8)()
    # a count query, then a buffer one short: the count comes back, nothing is written
    assert lib.pa_decode_work_items(lens, 3, 16, 4, 16, None, None, 0, ctypes.byref(n)) == 0
    assert n.value == 1 + 3 + 2
    buf[0] = 12345
    assert lib.pa_decode_work_items(lens, 3, 16, 4, 16, None, buf, 5, ctypes.byref(n)) == 1
    assert n.value == 6 and buf[0] == 12345
    assert lib.pa_decode_work_items(lens, 3, 16, 4, 16, None, buf, 8, ctypes.byref(n)) == 0
    assert list(buf[:6]) == [1 * 4 + 0, 1 * 4 + 1, 1 * 4 + 2, 2 * 4 + 0, 2 * 4 + 1, 0]
    with pytest.raises(B.PagedKVError, match="INVALID_ARG"):
        B.partition_work_items([10, 40, 20], 16, 4, 16, order=[0, 0, 2])   # not a permutation
    with pytest.raises(B.PagedKVError, match="INVALID_ARG"):
        B.partition_work_items([10, 65, 20], 16, 4, 16)                   # longer than 4 blocks
    with pytest.raises(B.PagedKVError, match="INVALID_ARG"):
        B.partition_work_items([10], 24, 4, 16)                          # not a multiple of 16
    with pytest.raises(ValueError):
        B.partition_work_items([10, 20], 16, 4, 16, order=[0])
