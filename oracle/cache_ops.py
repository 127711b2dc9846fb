"""Element-by-element reference for the two kernels that keep the paged cache
consistent.  TEST INFRASTRUCTURE ONLY (see the package docstring).

* Append (PagedAttention, zeroshotmind.com page, "Paging the cache": blocks are
  filled as the sequence grows): token ``t``'s key and value go to slot
  ``slot_mapping[t]``, i.e. row ``slot % block_size`` of physical block
  ``slot // block_size``, for every head.  A negative slot marks a padding
  token that is not written.
* Block copy (same page, "Sharing a prefix without copying it": copy-on-write
  duplicates just the one block about to be written): for each ``(src, dst)``
  pair, every key and value element of block ``dst`` becomes that of ``src``.

Both are bit copies: they operate on the stored representation (uint16 bit
patterns or float16) and never convert values.
"""

from __future__ import annotations

import numpy as np


def kv_append(k_cache: np.ndarray, v_cache: np.ndarray, k: np.ndarray, v: np.ndarray,
              slot_mapping, block_size: int) -> None:
    """In place.  Caches ``[B, H, bs, D]``; k, v ``[T, H, D]``; slot_mapping ``[T]``."""
    for t in range(len(slot_mapping)):
        slot = int(slot_mapping[t])
        if slot < 0:
            continue
        block, row = divmod(slot, block_size)
        for h in range(k_cache.shape[1]):
            k_cache[block, h, row, :] = k[t, h, :]
            v_cache[block, h, row, :] = v[t, h, :]


def block_copy(k_caches, v_caches, pairs) -> None:
    """In place, over every layer's pair of caches.  ``pairs`` is ``[n, 2]`` of
    (source block, destination block), applied in order; the pair (-1, -1) is
    padding and copies nothing (a library convention, not from the sources)."""
    for src, dst in np.asarray(pairs).reshape(-1, 2):
        if src == -1 and dst == -1:
            continue
        for kc, vc in zip(k_caches, v_caches):
            kc[int(dst)] = kc[int(src)].copy()
            vc[int(dst)] = vc[int(src)].copy()
