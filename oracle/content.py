"""Logical token contents of sequences.  TEST INFRASTRUCTURE ONLY.

The attention a sequence computes depends only on its tokens in logical order
(PagedAttention, zeroshotmind.com page, "Block tables: logical order, physical
scatter"); where those tokens physically sit is the allocator's business.  This
model therefore tracks, per sequence, the list of *origins* of its tokens (an
integer naming the row of a value store that produced the token), under the
operations a serving loop performs:

* add: a sequence starts with a run of tokens;
* fork: the child starts with exactly the parent's tokens ("Sharing a prefix
  without copying it": parallel samples share everything up to where they
  differ);
* append: one more token at the end;
* free: the sequence ends.

The oracle reads a sequence's keys and values by looking its origins up in the
value stores; no block table, slot or copy is involved, so the model shares
nothing with the allocator it is used to check.
"""

from __future__ import annotations

from typing import Dict, List

import numpy as np


class LogicalSequences:
    def __init__(self):
        self.origins: Dict[int, List[int]] = {}

    def add(self, seq: int, origins) -> None:
        assert seq not in self.origins
        self.origins[seq] = [int(o) for o in origins]

    def fork(self, parent: int, child: int) -> None:
        assert child not in self.origins
        self.origins[child] = list(self.origins[parent])

    def append(self, seq: int, origin: int) -> None:
        self.origins[seq].append(int(origin))

    def free(self, seq: int) -> None:
        del self.origins[seq]

    def __len__(self) -> int:
        return len(self.origins)

    def length(self, seq: int) -> int:
        return len(self.origins[seq])

    def rows(self, seq: int) -> np.ndarray:
        return np.asarray(self.origins[seq], dtype=np.int64)
