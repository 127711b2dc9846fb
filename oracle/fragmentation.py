"""Wasted KV slots: contiguous max-length reservation versus paged blocks.
TEST INFRASTRUCTURE ONLY.

PagedAttention, zeroshotmind.com page:

* "The memory you allocate but never use": a contiguous scheme reserves
  ``max_seq_len`` slots per request; whatever the request does not fill is
  internal fragmentation (its example: capped at 2048, stops after 128, so
  1920 slots sit unused).
* "The fragmentation arithmetic": with paging, the only waste is the unfilled
  part of each sequence's last block, at most ``block_size - 1`` slots (15 at
  block size 16).

External fragmentation (holes between slabs of different sizes) depends on an
arrival/departure history the pages do not give; it is not modelled, so the
contiguous figure here is the internal part only, a lower bound on that
scheme's waste.
"""

from __future__ import annotations

import numpy as np


def paged_slots(lens, block_size: int) -> np.ndarray:
    """Slots reserved per sequence under paging: whole blocks, ceil(len / bs) of them."""
    lens = np.asarray(lens, dtype=np.int64)
    return -(-lens // block_size) * block_size


def paged_waste(lens, block_size: int):
    """(wasted fraction of reserved slots, per-sequence slack array)."""
    lens = np.asarray(lens, dtype=np.int64)
    reserved = paged_slots(lens, block_size)
    slack = reserved - lens
    total = reserved.sum()
    return (float(slack.sum() / total) if total else 0.0), slack


def contiguous_waste(lens, max_seq_len: int):
    """(wasted fraction, per-sequence unused slots) when every sequence reserves
    ``max_seq_len`` contiguous slots."""
    lens = np.asarray(lens, dtype=np.int64)
    if (lens > max_seq_len).any():
        raise ValueError("a sequence is longer than its reservation")
    unused = max_seq_len - lens
    total = max_seq_len * lens.shape[0]
    return (float(unused.sum() / total) if total else 0.0), unused
