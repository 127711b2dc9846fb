"""Pins for the append and block-copy oracles: brute force over flat memory,
and the invariants that the untouched parts of the pool keep their bytes."""

import numpy as np

from oracle import cache_ops as C


def _flat_index(block, head, row, d, H, bs, D):
    # Row-major offset in a [B, H, bs, D] pool, written out independently.
    return ((block * H + head) * bs + row) * D + d


def test_append_matches_flat_memory_brute_force():
    rng = np.random.default_rng(0)
    B, H, bs, D, T = 6, 3, 4, 5, 9
    kc = rng.integers(0, 1 << 16, size=(B, H, bs, D), dtype=np.uint32).astype(np.uint16)
    vc = rng.integers(0, 1 << 16, size=(B, H, bs, D), dtype=np.uint32).astype(np.uint16)
    k = rng.integers(0, 1 << 16, size=(T, H, D), dtype=np.uint32).astype(np.uint16)
    v = rng.integers(0, 1 << 16, size=(T, H, D), dtype=np.uint32).astype(np.uint16)
    slots = np.array([0, 5, -1, 23, 7, -3, 12, 1, 20], dtype=np.int64)
    fk, fv = kc.reshape(-1).copy(), vc.reshape(-1).copy()
    for t, s in enumerate(slots):
        if s < 0:
            continue
        for h in range(H):
            for d in range(D):
                fk[_flat_index(s // bs, h, s % bs, d, H, bs, D)] = k[t, h, d]
                fv[_flat_index(s // bs, h, s % bs, d, H, bs, D)] = v[t, h, d]
    C.kv_append(kc, vc, k, v, slots, bs)
    assert np.array_equal(kc.reshape(-1), fk) and np.array_equal(vc.reshape(-1), fv)


def test_append_skips_negative_slots_and_leaves_the_rest():
    kc = np.zeros((2, 1, 4, 2), np.uint16)
    vc = np.zeros_like(kc)
    k = np.full((2, 1, 2), 7, np.uint16)
    C.kv_append(kc, vc, k, k, [-1, 6], 4)
    assert kc[1, 0, 2].tolist() == [7, 7]
    kc[1, 0, 2] = 0
    assert not kc.any()


def test_block_copy_duplicates_exactly_the_listed_blocks():
    rng = np.random.default_rng(1)
    layers = [rng.integers(0, 1000, size=(5, 2, 4, 3)).astype(np.uint16) for _ in range(3)]
    vlayers = [x + 1 for x in layers]
    before_k = [x.copy() for x in layers]
    before_v = [x.copy() for x in vlayers]
    C.block_copy(layers, vlayers, np.array([[1, 3], [4, 0]]))
    for L in range(3):
        for src, dst in ((1, 3), (4, 0)):
            assert np.array_equal(layers[L][dst], before_k[L][src])
            assert np.array_equal(vlayers[L][dst], before_v[L][src])
        for untouched in (1, 2, 4):
            assert np.array_equal(layers[L][untouched], before_k[L][untouched])


def test_block_copy_padding_pairs_copy_nothing():
    rng = np.random.default_rng(2)
    kc = rng.integers(0, 1000, size=(4, 2, 4, 3)).astype(np.uint16)
    vc = kc + 1
    before_k, before_v = kc.copy(), vc.copy()
    C.block_copy([kc], [vc], np.array([[-1, -1], [2, 0], [-1, -1]]))
    assert np.array_equal(kc[0], before_k[2]) and np.array_equal(vc[0], before_v[2])
    for untouched in (1, 2, 3):
        assert np.array_equal(kc[untouched], before_k[untouched])
        assert np.array_equal(vc[untouched], before_v[untouched])
