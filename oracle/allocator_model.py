"""Reference model of the paged-cache block allocator.  TEST INFRASTRUCTURE ONLY.

Rules, from PagedAttention (zeroshotmind.com page):

* "Paging the cache": blocks hold ``block_size`` tokens; a sequence is granted
  one block at a time, only when it grows into it, so it holds exactly
  ceil(len / block_size) blocks with at most one partly filled tail block.
* "Block tables": each sequence keeps the list of its physical blocks in
  logical order.
* "Sharing a prefix without copying it": sequences may point at the same
  physical blocks; a block's reference count is the number of sequences that
  depend on it.  A sequence about to write into a block that others also hold
  gets its own copy of just that block (copy-on-write): a fresh block, its
  table entry repointed, and the original's count decremented.

Policy choices the pages leave open, fixed here so that two allocators given the
same ``free_order`` produce the same tables: the free list is a stack, blocks
are first handed out in ``free_order`` order, and a freed block goes back on
top (last in, first out).  A block whose count drops to zero is freed.  A write
into a full block never happens (the next token opens a new block), so full
shared blocks are never copied.
"""

from __future__ import annotations

from typing import Dict, List, Optional, Tuple


class AllocatorError(Exception):
    pass


class BlockAllocatorModel:
    def __init__(self, num_blocks: int, block_size: int, free_order=None):
        if num_blocks <= 0 or block_size <= 0:
            raise AllocatorError("num_blocks and block_size must be positive")
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)
        order = list(range(num_blocks)) if free_order is None else [int(b) for b in free_order]
        if sorted(order) != list(range(num_blocks)):
            raise AllocatorError("free_order must be a permutation of the pool")
        self.free: List[int] = list(reversed(order))   # top of the stack = end of the list
        self.refcount: List[int] = [0] * num_blocks
        self.tables: Dict[int, List[int]] = {}
        self.lens: Dict[int, int] = {}

    # -- helpers ---------------------------------------------------------
    def _take(self) -> int:
        if not self.free:
            raise AllocatorError("out of blocks")
        b = self.free.pop()
        self.refcount[b] = 1
        return b

    def _release(self, b: int) -> None:
        if self.refcount[b] <= 0:
            raise AllocatorError(f"refcount underflow on block {b}")
        self.refcount[b] -= 1
        if self.refcount[b] == 0:
            self.free.append(b)

    # -- operations ------------------------------------------------------
    def add(self, seq: int, num_tokens: int) -> None:
        """A new sequence holding ``num_tokens`` tokens: ceil(n / bs) fresh blocks."""
        if seq in self.tables:
            raise AllocatorError(f"sequence {seq} exists")
        need = -(-int(num_tokens) // self.block_size)
        if need > len(self.free):
            raise AllocatorError("out of blocks")
        self.tables[seq] = [self._take() for _ in range(need)]
        self.lens[seq] = int(num_tokens)

    def fork(self, parent: int, child: int) -> None:
        """``child`` shares every block of ``parent``; each block's count goes up by one."""
        if parent not in self.tables:
            raise AllocatorError(f"no sequence {parent}")
        if child in self.tables:
            raise AllocatorError(f"sequence {child} exists")
        self.tables[child] = list(self.tables[parent])
        self.lens[child] = self.lens[parent]
        for b in self.tables[child]:
            self.refcount[b] += 1

    def append(self, seq: int) -> Tuple[int, Optional[Tuple[int, int]]]:
        """Reserve the slot of the sequence's next token.

        Returns ``(slot, cow)`` where ``slot = block * bs + row`` and ``cow`` is the
        ``(src, dst)`` block pair to copy before the token is written, or None.
        """
        if seq not in self.tables:
            raise AllocatorError(f"no sequence {seq}")
        pos = self.lens[seq]
        j, row = divmod(pos, self.block_size)
        table = self.tables[seq]
        cow = None
        if row == 0:
            table.append(self._take())
        else:
            b = table[j]
            if self.refcount[b] > 1:
                d = self._take()
                self.refcount[b] -= 1
                table[j] = d
                cow = (b, d)
        self.lens[seq] = pos + 1
        return table[j] * self.block_size + row, cow

    def free_seq(self, seq: int) -> None:
        if seq not in self.tables:
            raise AllocatorError(f"no sequence {seq}")
        for b in self.tables.pop(seq):
            self._release(b)
        del self.lens[seq]

    # -- invariants ------------------------------------------------------
    def check(self) -> None:
        """Raise if any invariant the pages fix is broken."""
        bs = self.block_size
        holders = [0] * self.num_blocks
        for seq, table in self.tables.items():
            L = self.lens[seq]
            if len(table) != -(-L // bs):
                raise AllocatorError(f"seq {seq}: {len(table)} blocks for {L} tokens")
            if len(table) * bs - L > bs - 1:
                raise AllocatorError(f"seq {seq}: more than {bs - 1} slack slots")
            for b in table:
                holders[b] += 1
        if holders != self.refcount:
            raise AllocatorError("refcount differs from the number of holders")
        if len(set(self.free)) != len(self.free):
            raise AllocatorError("block on the free list twice")
        used = {b for b in range(self.num_blocks) if holders[b] > 0}
        if used & set(self.free):
            raise AllocatorError("a held block is on the free list")
        if len(used) + len(self.free) != self.num_blocks:
            raise AllocatorError("blocks leaked")
