"""Pins for the attention oracle: brute force, closed forms and invariants.

None of these re-types the oracle's formula: the brute force walks the pool
with its own index arithmetic in pure Python, and the closed forms come from
the mathematics of softmax.
"""

import math

import numpy as np
import pytest
import torch

from oracle import attention as A
from workloads import random_decode_batch, tiny_decode


def _bf16_bits(x: torch.Tensor) -> np.ndarray:
    return x.contiguous().view(torch.int16).numpy().view(np.uint16)


def _storage(t: torch.Tensor):
    if t.dtype == torch.bfloat16:
        return _bf16_bits(t), "bf16"
    return t.numpy(), "f16"


def brute_force(pool_k, pool_v, table, L, bs, q, scale):
    """Pure-Python triple loop over a tiny pool given as nested lists of floats."""
    H, D = len(q), len(q[0])
    out = [[0.0] * D for _ in range(H)]
    for h in range(H):
        scores = []
        for t in range(L):
            blk, row = table[t // bs], t % bs
            scores.append(scale * sum(q[h][d] * pool_k[blk][h][row][d] for d in range(D)))
        if L == 0:
            continue
        mx = max(scores)
        ws = [math.exp(s - mx) for s in scores]
        tot = sum(ws)
        for t in range(L):
            blk, row = table[t // bs], t % bs
            for d in range(D):
                out[h][d] += ws[t] / tot * pool_v[blk][h][row][d]
    return out


def test_bf16_upcast_matches_torch_and_known_values():
    bits = np.array([0x3F80, 0xC000, 0x3F81, 0x0000, 0x8000, 0x7F7F, 0x0001], dtype=np.uint16)
    got = A.to_float64(bits, "bf16")
    assert got[0] == 1.0 and got[1] == -2.0 and got[2] == 1.0078125
    assert got[3] == 0.0 and got[4] == 0.0 and math.copysign(1, got[4]) == -1
    rng = np.random.default_rng(0)
    raw = rng.integers(0, 1 << 16, size=10000, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(raw.view(np.int16)).view(torch.bfloat16).double().numpy()
    mine = A.to_float64(raw, "bf16")
    same = (ref == mine) | (np.isnan(ref) & np.isnan(mine))
    assert same.all()


@pytest.mark.parametrize("seed,H,D,bs,lens", [
    (11, 2, 8, 4, [1, 5, 9, 16]),
    (12, 1, 4, 16, [40, 3]),
    (13, 2, 6, 8, [17, 8, 24]),
])
def test_matches_brute_force_on_tiny_inputs(seed, H, D, bs, lens):
    b = random_decode_batch(seed, lens, H, D, bs, dtype="f16", pool_factor=2.0)
    kc, vc = b.k_cache.double().tolist(), b.v_cache.double().tolist()
    q = b.q.double()
    got = A.paged_decode_attention(b.q.numpy(), b.k_cache.numpy(), b.v_cache.numpy(),
                                   b.block_tables, b.context_lens, b.scale, bs, "f16")
    for i, L in enumerate(lens):
        ref = brute_force(kc, vc, b.block_tables[i].tolist(), L, bs, q[i].tolist(), b.scale)
        assert np.max(np.abs(got[i] - np.array(ref))) <= 1e-12


def test_identical_keys_give_mean_of_values():
    rng = np.random.default_rng(1)
    L, H, D = 37, 3, 16
    k = np.repeat(rng.standard_normal((1, H, D)), L, axis=0)
    v = rng.standard_normal((L, H, D))
    q = rng.standard_normal((H, D))
    out = A.attention(q, k, v, 0.7)
    np.testing.assert_allclose(out, v.mean(axis=0), rtol=0, atol=1e-14)


def test_zero_query_gives_mean_of_values():
    rng = np.random.default_rng(2)
    k, v = rng.standard_normal((50, 2, 8)), rng.standard_normal((50, 2, 8))
    out = A.attention(np.zeros((2, 8)), k, v, 1.0)
    np.testing.assert_allclose(out, v.mean(axis=0), rtol=0, atol=1e-14)


def test_single_token_returns_its_value_exactly():
    rng = np.random.default_rng(3)
    k, v = rng.standard_normal((1, 4, 8)), rng.standard_normal((1, 4, 8))
    out = A.attention(rng.standard_normal((4, 8)) * 30, k, v, 0.125)
    assert np.array_equal(out, v[0])


def test_two_token_closed_form():
    # scores ln 3 and 0 -> weights 3/4 and 1/4 (independent of the shift).
    q = np.array([[1.0, 0.0]])
    k = np.array([[[math.log(3.0) + 5.0, 0.0]], [[5.0, 0.0]]])
    v = np.array([[[4.0, -8.0]], [[0.0, 8.0]]])
    out = A.attention(q, k, v, 1.0)
    np.testing.assert_allclose(out, [[3.0, -4.0]], rtol=0, atol=1e-14)


def test_scale_is_applied_to_the_scores():
    # With scale 2 the same keys give scores 2 ln 3 and 0 -> weights 9/10, 1/10.
    q = np.array([[1.0, 0.0]])
    k = np.array([[[math.log(3.0), 0.0]], [[0.0, 0.0]]])
    v = np.array([[[10.0, 0.0]], [[0.0, 10.0]]])
    out = A.attention(q, k, v, 2.0)
    np.testing.assert_allclose(out, [[9.0, 1.0]], rtol=0, atol=1e-13)


def test_large_scores_do_not_overflow():
    # One key dominates by ~1e4 in the exponent: the output is its value.
    q = np.array([[100.0]])
    k = np.array([[[100.0]], [[0.0]], [[-50.0]]])
    v = np.array([[[1.5]], [[-7.0]], [[3.0]]])
    out = A.attention(q, k, v, 1.0)
    assert np.isfinite(out).all()
    np.testing.assert_allclose(out, [[1.5]], rtol=0, atol=0)


def test_empty_sequence_is_zero():
    out = A.attention(np.ones((2, 4)), np.zeros((0, 2, 4)), np.zeros((0, 2, 4)), 1.0)
    assert out.shape == (2, 4) and not out.any()


def test_permuting_physical_placement_changes_nothing():
    b = tiny_decode(seed=1, with_append=False)
    kc, vc = b.k_cache.numpy(), b.v_cache.numpy()
    base = A.paged_decode_attention(b.q.numpy(), kc, vc, b.block_tables, b.context_lens,
                                    b.scale, b.block_size, "f16")
    perm = np.random.default_rng(9).permutation(b.num_blocks)       # new home of block p
    kc2, vc2 = np.empty_like(kc), np.empty_like(vc)
    kc2[perm], vc2[perm] = kc, vc
    tables2 = np.where(b.block_tables >= 0, perm[np.maximum(b.block_tables, 0)], -1)
    moved = A.paged_decode_attention(b.q.numpy(), kc2, vc2, tables2, b.context_lens,
                                     b.scale, b.block_size, "f16")
    assert np.array_equal(base, moved)


def test_poisoned_unused_slots_are_never_read():
    b = tiny_decode(seed=1, with_append=False)
    out = A.paged_decode_attention(b.q.numpy(), b.k_cache.numpy(), b.v_cache.numpy(),
                                   b.block_tables, b.context_lens, b.scale, b.block_size, "f16")
    assert np.isfinite(out).all()
    assert np.isnan(b.k_cache.numpy()).any()      # the poison is there to be missed


def test_bf16_path_matches_brute_force():
    b = random_decode_batch(21, [7, 19], 2, 8, 4, dtype="bf16", pool_factor=2.0)
    qs, dt = _storage(b.q)
    got = A.paged_decode_attention(qs, _bf16_bits(b.k_cache), _bf16_bits(b.v_cache),
                                   b.block_tables, b.context_lens, b.scale, 4, dt)
    kc, vc = b.k_cache.double().tolist(), b.v_cache.double().tolist()
    for i, L in enumerate([7, 19]):
        ref = brute_force(kc, vc, b.block_tables[i].tolist(), L, 4, b.q[i].double().tolist(), b.scale)
        assert np.max(np.abs(got[i] - np.array(ref))) <= 1e-12


@pytest.mark.parametrize("part", [1, 3, 16, 64, 1000])
def test_merged_partitions_equal_unsplit_attention(part):
    rng = np.random.default_rng(part)
    L, H, D = 200, 3, 16
    q, k, v = rng.standard_normal((H, D)), rng.standard_normal((L, H, D)), rng.standard_normal((L, H, D))
    m, l, acc = A.partition_partials(q, k, v, 0.3, part)
    assert m.shape == (-(-L // part), H)
    np.testing.assert_allclose(A.merge_partials(m, l, acc), A.attention(q, k, v, 0.3),
                               rtol=0, atol=1e-12)


def test_merge_of_uneven_pieces_equals_unsplit_attention():
    """The split a prefix record makes (a partition's shared first chunks, then
    each member's own rest, merged as two partials alongside the other
    partitions) is a regrouping of the same sum: partials over any cut of the
    tokens into consecutive pieces merge to the unsplit attention."""
    rng = np.random.default_rng(17)
    L, H, D = 300, 2, 16
    q, k, v = rng.standard_normal((H, D)), rng.standard_normal((L, H, D)), rng.standard_normal((L, H, D))
    for cuts in ([0, 128, 176, 256, 300], [0, 16, 300], [0, 299, 300], [0, 1, 2, 3, 300]):
        parts = [A.partition_partials(q, k[a:b], v[a:b], 0.7, b - a) for a, b in zip(cuts, cuts[1:])]
        m, l, acc = (np.concatenate([x[i] for x in parts]) for i in range(3))
        np.testing.assert_allclose(A.merge_partials(m, l, acc), A.attention(q, k, v, 0.7),
                                   rtol=0, atol=1e-12)


def test_single_partition_partials_normalise_to_attention():
    rng = np.random.default_rng(5)
    q, k, v = rng.standard_normal((2, 8)), rng.standard_normal((30, 2, 8)), rng.standard_normal((30, 2, 8))
    m, l, acc = A.partition_partials(q, k, v, 1.0, 64)
    np.testing.assert_allclose(acc[0] / l[0][:, None], A.attention(q, k, v, 1.0), rtol=0, atol=1e-13)
    s = np.einsum("hd,lhd->hl", q, k)
    np.testing.assert_array_equal(m[0], s.max(axis=1))


def _brute_prefill(pool_k, pool_v, table, L, n_q, bs, q_rows, scale):
    """Pure-Python causal multi-query attention: query j at position L - n_q + j."""
    H, D = len(q_rows[0]), len(q_rows[0][0])
    out = []
    for j in range(n_q):
        p = L - n_q + j
        row = [[0.0] * D for _ in range(H)]
        for h in range(H):
            sc = []
            for t in range(p + 1):
                blk, r = table[t // bs], t % bs
                sc.append(scale * sum(q_rows[j][h][d] * pool_k[blk][h][r][d] for d in range(D)))
            mx = max(sc)
            ws = [math.exp(x - mx) for x in sc]
            tot = sum(ws)
            for t in range(p + 1):
                blk, r = table[t // bs], t % bs
                for d in range(D):
                    row[h][d] += ws[t] / tot * pool_v[blk][h][r][d]
        out.append(row)
    return out


def test_prefill_matches_brute_force():
    lens, nq = [9, 20, 5], [3, 20, 1]
    b = random_decode_batch(31, lens, 2, 4, 4, dtype="f16", pool_factor=2.0)
    gen = torch.Generator().manual_seed(5)
    q = torch.randn(sum(nq), 2, 4, generator=gen).half()
    starts = np.concatenate([[0], np.cumsum(nq)])
    got = A.paged_prefill_attention(q.numpy(), b.k_cache.numpy(), b.v_cache.numpy(),
                                    b.block_tables, b.context_lens, starts, 0.6, 4, "f16")
    kc, vc = b.k_cache.double().tolist(), b.v_cache.double().tolist()
    for i in range(3):
        ref = _brute_prefill(kc, vc, b.block_tables[i].tolist(), lens[i], nq[i], 4,
                             q[starts[i]:starts[i + 1]].double().tolist(), 0.6)
        assert np.max(np.abs(got[starts[i]:starts[i + 1]] - np.array(ref))) <= 1e-12


def test_prefill_single_query_is_decode_and_last_query_sees_everything():
    lens = [33, 70]
    b = random_decode_batch(32, lens, 3, 8, 16, dtype="f16")
    dec = A.paged_decode_attention(b.q.numpy(), b.k_cache.numpy(), b.v_cache.numpy(),
                                   b.block_tables, b.context_lens, 0.4, 16, "f16")
    one = A.paged_prefill_attention(b.q.numpy(), b.k_cache.numpy(), b.v_cache.numpy(),
                                    b.block_tables, b.context_lens, [0, 1, 2], 0.4, 16, "f16")
    assert np.array_equal(one, dec)
    # query j of a chunk = decode of the first p + 1 tokens with that query
    q = np.repeat(b.q.numpy()[1:2], 5, axis=0)
    many = A.paged_prefill_attention(q, b.k_cache.numpy(), b.v_cache.numpy(), b.block_tables[1:],
                                     b.context_lens[1:], [0, 5], 0.4, 16, "f16")
    for j in range(5):
        p = 70 - 5 + j
        short = A.paged_decode_attention(b.q.numpy()[1:2], b.k_cache.numpy(), b.v_cache.numpy(),
                                         b.block_tables[1:], np.array([p + 1]), 0.4, 16, "f16")
        assert np.array_equal(many[j], short[0])
