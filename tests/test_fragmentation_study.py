"""Fragmentation study on the library's allocator: the pool occupancy it
reports matches the oracle's wasted-slot arithmetic, and on the synthetic
workload lengths paging wastes under the page's 4 % while a contiguous
max-length reservation wastes 60-80 % (PagedAttention, zeroshotmind.com page,
"The memory you allocate but never use" and "The fragmentation arithmetic")."""

import json
import os

import numpy as np
import pytest

from oracle.allocator_model import BlockAllocatorModel
from oracle.fragmentation import contiguous_waste, paged_waste
from workloads import lognormal_lengths

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                     "fragmentation_pages.json")))


def _lengths_13b(n=256, seed=2):
    return lognormal_lengths(np.random.default_rng(seed), n, 350.0, 0.75, 16, 2048)


def _lengths_mixed(n=512, seed=5):
    rng = np.random.default_rng(seed)
    is_long = np.zeros(n, dtype=bool)
    is_long[: int(round(0.3 * n))] = True
    rng.shuffle(is_long)
    return np.where(is_long, rng.integers(1024, 4097, size=n),
                    rng.integers(32, 257, size=n)).astype(np.int64)


@pytest.mark.parametrize("lens_fn,max_len", [(_lengths_13b, 2048), (_lengths_mixed, 4096)])
def test_library_allocator_occupancy_matches_the_arithmetic(lib, lens_fn, max_len):
    from paged_kv_cache_317_gb300.binding import BlockAllocator
    bs = GOLDEN["default_block_size"]["block_size"]
    lens = lens_fn()
    nb = int((-(-lens // bs)).sum()) + 8
    a = BlockAllocator(nb, bs, np.random.default_rng(0).permutation(nb))
    for i, L in enumerate(lens):
        a.add(i, int(L))
    st = a.stats()
    frac, slack = paged_waste(lens, bs)
    assert st["tokens_logical"] == int(lens.sum())
    assert st["slots_logical"] == int(lens.sum() + slack.sum())
    assert st["slots_filled"] == st["tokens_logical"]          # no sharing: every row once
    assert st["blocks_used"] * bs == st["slots_logical"]
    lib_frac = 1 - st["tokens_logical"] / st["slots_logical"]
    assert abs(lib_frac - frac) < 1e-12
    assert lib_frac < GOLDEN["paged_waste_bound"]["max_fraction"]
    contig, _ = contiguous_waste(lens, max_len)
    lo, hi = GOLDEN["contiguous_waste_range"]["low"], GOLDEN["contiguous_waste_range"]["high"]
    assert lo <= contig <= hi


def test_sharing_stores_a_prefix_once():
    """Eight samples of one partly filled prompt: logically 8 copies, physically one
    prefix plus the seven copied tail blocks."""
    from paged_kv_cache_317_gb300.binding import BlockAllocator
    bs, prompt = 16, 1029
    a = BlockAllocator(200, bs)
    model = BlockAllocatorModel(200, bs)
    a.add(0, prompt)
    model.add(0, prompt)
    for s in range(1, 8):
        a.fork(0, s)
        model.fork(0, s)
    for s in range(8):
        a.append(s)
        model.append(s)
    st = a.stats()
    assert st["tokens_logical"] == 8 * (prompt + 1)
    full, tail = prompt // bs, prompt % bs + 1
    assert st["blocks_used"] == full + 8                        # shared full blocks + 8 tails
    assert st["slots_filled"] == full * bs + 8 * tail
    assert st["blocks_used"] == sum(1 for r in model.refcount if r > 0)
