"""Pins for the allocator reference model: worked scenarios derived by hand from
the pages' rules, and the invariants after random operation sequences."""

import numpy as np
import pytest

from oracle.allocator_model import AllocatorError, BlockAllocatorModel
from oracle.content import LogicalSequences


def test_add_grants_ceil_len_over_block_size_blocks_in_free_order():
    a = BlockAllocatorModel(10, 4, free_order=[7, 2, 9, 0, 1, 3, 4, 5, 6, 8])
    a.add(100, 6)            # 6 tokens at 4 per block -> 2 blocks, 2 slack slots
    assert a.tables[100] == [7, 2]
    a.add(101, 4)            # exactly one full block
    assert a.tables[101] == [9]
    a.add(102, 0)            # nothing yet
    assert a.tables[102] == []
    a.check()


def test_append_opens_a_block_only_when_the_tail_is_full():
    a = BlockAllocatorModel(8, 4, free_order=range(8))
    a.add(1, 3)
    slot, cow = a.append(1)               # position 3: row 3 of block 0
    assert (slot, cow) == (3, None)
    slot, cow = a.append(1)               # position 4: new block 1, row 0
    assert (slot, cow) == (4, None) and a.tables[1] == [0, 1]
    a.check()


def test_fork_then_divergent_write_copies_exactly_one_block():
    a = BlockAllocatorModel(8, 4, free_order=range(8))
    a.add(1, 6)                           # blocks [0, 1]; tail block 1 holds 2 tokens
    a.fork(1, 2)
    assert a.refcount[0] == 2 and a.refcount[1] == 2
    slot, cow = a.append(2)               # child writes into shared tail -> copy block 1 to 2
    assert cow == (1, 2) and slot == 2 * 4 + 2
    assert a.tables[2] == [0, 2] and a.tables[1] == [0, 1]
    assert a.refcount[1] == 1 and a.refcount[2] == 1 and a.refcount[0] == 2
    slot, cow = a.append(1)               # parent now sole holder: writes in place
    assert cow is None and slot == 1 * 4 + 2
    a.check()


def test_fork_at_block_boundary_needs_no_copy():
    a = BlockAllocatorModel(8, 4, free_order=range(8))
    a.add(1, 8)                           # two full blocks
    a.fork(1, 2)
    s1, c1 = a.append(1)
    s2, c2 = a.append(2)
    assert c1 is None and c2 is None
    assert a.tables[1][:2] == a.tables[2][:2] and a.tables[1][2] != a.tables[2][2]
    a.check()


def test_free_returns_blocks_last_in_first_out():
    a = BlockAllocatorModel(6, 4, free_order=range(6))
    a.add(1, 8)                           # blocks 0, 1
    a.fork(1, 2)
    a.free_seq(1)                         # counts drop to 1: nothing freed
    assert len(a.free) == 4
    a.free_seq(2)                         # both freed, 1 then 0 pushed... in table order
    assert len(a.free) == 6
    a.add(3, 4)
    assert a.tables[3] == [1]             # last block released is first handed out
    a.check()


def test_out_of_blocks_and_misuse_raise():
    a = BlockAllocatorModel(2, 4)
    a.add(1, 8)
    with pytest.raises(AllocatorError):
        a.add(2, 1)
    with pytest.raises(AllocatorError):
        a.append(1)                       # needs a third block
    with pytest.raises(AllocatorError):
        a.free_seq(99)
    with pytest.raises(AllocatorError):
        a.fork(1, 1)


@pytest.mark.parametrize("partial,expected_copies", [(True, 7), (False, 0)])
def test_parallel_sampling_copy_count(partial, expected_copies):
    """One prompt shared by 8 samples; each sample appends once in sample order.
    A partly filled shared tail is copied by the first 7 writers; the 8th, then
    the sole holder, writes in place.  A block-aligned prompt needs no copy."""
    bs = 16
    a = BlockAllocatorModel(200, bs)
    a.add(0, 1024 + (5 if partial else 0))
    for s in range(1, 8):
        a.fork(0, s)
    copies = [a.append(s)[1] for s in range(8)]
    real = [c for c in copies if c is not None]
    assert len(real) == expected_copies
    assert len({c[1] for c in real}) == len(real)            # each copy gets its own block
    assert len({c[0] for c in real}) <= 1                    # all copy the same shared tail
    a.check()


def test_random_operation_sequences_keep_the_invariants():
    rng = np.random.default_rng(42)
    for trial in range(20):
        bs = int(rng.choice([1, 4, 16]))
        a = BlockAllocatorModel(300, bs, free_order=rng.permutation(300))
        content = LogicalSequences()
        next_id, origin = 0, 0
        for _ in range(400):
            op = rng.integers(0, 4)
            live = list(a.tables)
            try:
                if op == 0 or not live:
                    n = int(rng.integers(0, 40))
                    a.add(next_id, n)
                    content.add(next_id, range(origin, origin + n))
                    origin += n
                    next_id += 1
                elif op == 1:
                    p = live[rng.integers(len(live))]
                    a.fork(p, next_id)
                    content.fork(p, next_id)
                    next_id += 1
                elif op == 2:
                    s = live[rng.integers(len(live))]
                    held_before = {b: a.refcount[b] for b in a.tables[s]}
                    slot, cow = a.append(s)
                    content.append(s, origin)
                    origin += 1
                    if cow is not None:
                        assert held_before[cow[0]] > 1                 # only shared blocks copy
                        assert a.refcount[cow[0]] == held_before[cow[0]] - 1
                    assert slot // bs == a.tables[s][(a.lens[s] - 1) // bs]
                else:
                    s = live[rng.integers(len(live))]
                    a.free_seq(s)
                    content.free(s)
            except AllocatorError as e:
                assert "out of blocks" in str(e)
            a.check()
            for s in a.tables:
                assert a.lens[s] == content.length(s)
        for s in list(a.tables):
            a.free_seq(s)
        a.check()
        assert len(a.free) == 300


def test_logical_content_of_fork_and_append():
    c = LogicalSequences()
    c.add(1, [10, 11, 12])
    c.fork(1, 2)
    c.append(2, 99)
    c.append(1, 50)
    assert c.rows(1).tolist() == [10, 11, 12, 50]
    assert c.rows(2).tolist() == [10, 11, 12, 99]
    c.free(1)
    assert len(c) == 1
