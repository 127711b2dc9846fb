"""GPU parity of paged decode attention against the fp64 oracle, through the C ABI."""

import numpy as np
import pytest
import torch

from gpu_util import (assert_matches_oracle, device_tables, oracle_decode, storage)
from oracle import attention as OA
from workloads import random_decode_batch, tiny_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B(lib):
    from paged_kv_cache_317_gb300 import binding
    return binding


def run_decode(B, batch, out_dtype=torch.float32, **kw):
    bt, sl = device_tables(batch)
    if batch.has_append:
        B.kv_cache_append(batch.new_k, batch.new_v,
                          torch.from_numpy(batch.slot_mapping).cuda(), batch.k_cache,
                          batch.v_cache)
    out = B.paged_attn_decode(batch.q, batch.k_cache, batch.v_cache, bt, sl, batch.scale,
                              out_dtype=out_dtype, **kw)
    torch.cuda.synchronize()
    return out


def test_tiny_config_append_then_decode(B):
    b = tiny_decode(seed=1, device="cuda")
    ref = oracle_decode(b)
    rec = B.new_error_record()
    bt, sl = device_tables(b)
    B.kv_cache_append(b.new_k, b.new_v, torch.from_numpy(b.slot_mapping).cuda(), b.k_cache,
                      b.v_cache, error_record=rec)
    out = B.paged_attn_decode(b.q, b.k_cache, b.v_cache, bt, sl, b.scale, error_record=rec)
    assert B.pa_error_read(rec) == [0, 0, 0, 0]
    assert_matches_oracle(out, ref, "tiny")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("bs", [8, 16, 32])
def test_decode_sweep_ragged_lengths(B, dtype, D, bs):
    lens = [1, 2, 15, 16, 17, 31, 33, 100, 255, 511, 512, 513, 700, 1025, 0, 3]
    b = random_decode_batch(1000 + D + bs, lens, 4, D, bs, dtype=dtype, device="cuda")
    ref = oracle_decode(b)
    for pt in (0, 64, 16):
        out = run_decode(B, b, partition_tokens=pt)
        assert_matches_oracle(out, ref, f"{dtype} D{D} bs{bs} pt{pt}")


@pytest.mark.parametrize("out_dtype", [torch.float16, torch.bfloat16])
def test_half_precision_outputs(B, out_dtype):
    b = random_decode_batch(7, [5, 40, 300, 900], 8, 128, 16, dtype="bf16", device="cuda")
    ref = oracle_decode(b)
    for pt in (0, 128):
        assert_matches_oracle(run_decode(B, b, out_dtype=out_dtype, partition_tokens=pt), ref)


@pytest.mark.parametrize("G,S", [(1, 2), (2, 3), (4, 2), (8, 2), (5, 4), (4, 6)])
def test_launch_shapes_agree(B, G, S):
    b = random_decode_batch(8, [1, 77, 640, 1500, 16], 40, 128, 16, dtype="bf16", device="cuda")
    ref = oracle_decode(b)
    assert_matches_oracle(run_decode(B, b, heads_per_cta=G, stages=S), ref, f"G{G} S{S}")


@pytest.mark.parametrize("bs", [8, 16])
def test_permuted_placement_is_bit_identical(B, bs):
    b = random_decode_batch(9, [3, 64, 129, 800], 8, 128, bs, dtype="f16", device="cuda",
                            pool_factor=2.0)
    base = run_decode(B, b)
    perm = torch.from_numpy(np.random.default_rng(3).permutation(b.num_blocks)).cuda()
    k2, v2 = torch.empty_like(b.k_cache), torch.empty_like(b.v_cache)
    k2[perm], v2[perm] = b.k_cache, b.v_cache
    t = torch.from_numpy(b.block_tables).cuda().long()
    t2 = torch.where(t >= 0, perm[t.clamp(min=0)], t).int()
    out2 = B.paged_attn_decode(b.q, k2, v2, t2, torch.from_numpy(b.context_lens).cuda(), b.scale)
    torch.cuda.synchronize()
    assert torch.equal(base, out2)


def test_single_token_returns_its_value_exactly(B):
    b = random_decode_batch(10, [1, 1, 1], 8, 128, 16, dtype="bf16", device="cuda")
    out = run_decode(B, b)
    for i in range(3):
        blk = int(b.block_tables[i, 0])
        assert torch.equal(out[i], b.v_cache[blk, :, 0, :].float())


def test_empty_sequence_gives_zeros(B):
    b = random_decode_batch(11, [0, 5, 0], 4, 64, 16, dtype="f16", device="cuda")
    out = run_decode(B, b)
    assert not out[0].any() and not out[2].any() and torch.isfinite(out).all()


def test_identical_keys_give_mean_of_values(B):
    b = random_decode_batch(12, [300, 47], 4, 128, 16, dtype="bf16", device="cuda")
    for i in range(2):
        nb = -(-int(b.context_lens[i]) // 16)
        for j in range(nb):
            b.k_cache[int(b.block_tables[i, j])] = b.k_cache[int(b.block_tables[0, 0]), :, 0:1, :]
    out = run_decode(B, b, partition_tokens=64)
    for i in range(2):
        L = int(b.context_lens[i])
        v, dt = storage(b.v_cache)
        rows = OA.gather_sequence(v, b.block_tables[i], L, 16)
        mean = OA.to_float64(rows, dt).mean(axis=0)
        assert_matches_oracle(out[i], mean, "identical keys")


def test_split_partials_match_oracle_partitions(B):
    """Phase 1 alone leaves per-partition (m, l, acc) in the workspace in log2 units."""
    lens = [600, 1030, 100]
    H, D, bs, pt = 4, 128, 16, 256
    b = random_decode_batch(13, lens, H, D, bs, dtype="bf16", device="cuda")
    bt, sl = device_tables(b)
    N, MB = len(lens), b.max_blocks_per_seq
    P = -(-MB * bs // pt)
    need = B.paged_attn_workspace_size(N, H, D, bs, MB, pt)
    ws = torch.zeros(need // 4, dtype=torch.float32, device="cuda")
    out = torch.zeros(N, H, D, device="cuda")
    B.paged_attn_decode(b.q, b.k_cache, b.v_cache, bt, sl, b.scale, out=out, partition_tokens=pt,
                        workspace=ws, phases=1)
    torch.cuda.synchronize()
    acc = ws[: N * H * P * D].view(N, H, P, D).double().cpu().numpy()
    ml = ws[N * H * P * D:].view(N, H, P, 2).double().cpu().numpy()
    kc, dt = storage(b.k_cache)
    vc, _ = storage(b.v_cache)
    qs, _ = storage(b.q)
    log2e = 1.0 / np.log(2.0)
    for i, L in enumerate(lens):
        k = OA.to_float64(OA.gather_sequence(kc, b.block_tables[i], L, bs), dt)
        v = OA.to_float64(OA.gather_sequence(vc, b.block_tables[i], L, bs), dt)
        m, l, a = OA.partition_partials(OA.to_float64(qs[i], dt), k, v, b.scale, pt)
        n = m.shape[0]
        if n == 1:
            continue            # single partition: written straight to out
        np.testing.assert_allclose(ml[i, :, :n, 0], (m * log2e).T, rtol=0, atol=1e-4)
        np.testing.assert_allclose(ml[i, :, :n, 1], l.T, rtol=1e-5, atol=1e-5)
        np.testing.assert_allclose(acc[i, :, :n, :], a.transpose(1, 0, 2), rtol=1e-5, atol=1e-4)
    # phase 2 alone completes the output
    B.paged_attn_decode(b.q, b.k_cache, b.v_cache, bt, sl, b.scale, out=out, partition_tokens=pt,
                        workspace=ws, phases=2)
    torch.cuda.synchronize()
    assert_matches_oracle(out[:2], oracle_decode(b, [0, 1]), "phase 2")


def test_bad_block_entry_is_recorded_and_clamped(B):
    b = random_decode_batch(14, [40, 20], 4, 64, 16, dtype="f16", device="cuda", poison=False)
    bt, sl = device_tables(b)
    bt[1, 0] = b.num_blocks + 5
    rec = B.new_error_record()
    out = B.paged_attn_decode(b.q, b.k_cache, b.v_cache, bt, sl, b.scale, error_record=rec)
    r = B.pa_error_read(rec)
    assert r[0] == 4 and r[1] >= 1 and r[2] == 1 and r[3] == b.num_blocks + 5
    assert torch.isfinite(out).all()
    assert_matches_oracle(out[:1], oracle_decode(b, [0]), "unaffected sequence")


def test_bad_seq_len_is_recorded_and_clamped(B):
    b = random_decode_batch(15, [40, 20], 4, 64, 16, dtype="f16", device="cuda", poison=False)
    bt, sl = device_tables(b)
    bt[1, :] = bt[1, 0]          # every entry valid, so the clamped length reads real blocks
    sl[0] = -3
    sl[1] = 10 ** 6
    rec = B.new_error_record()
    out = B.paged_attn_decode(b.q, b.k_cache, b.v_cache, bt[:, :], sl, b.scale, error_record=rec,
                              partition_tokens=16)
    r = B.pa_error_read(rec)
    assert r[0] == 6 and r[1] == 2
    assert not out[0].any()


def test_seq_order_changes_nothing_but_the_schedule(B):
    b = random_decode_batch(16, [5, 900, 33, 1500, 64, 700, 2, 1100], 8, 128, 16, dtype="bf16",
                            device="cuda", with_append=True)
    bt, sl = device_tables(b)
    order = torch.from_numpy(np.argsort(-b.context_lens, kind="stable").astype(np.int32)).cuda()
    k1, v1, k2, v2 = b.k_cache.clone(), b.v_cache.clone(), b.k_cache.clone(), b.v_cache.clone()
    plain = B.paged_attn_decode_append(b.q, b.new_k, b.new_v, k1, v1, bt, sl, b.scale)
    ordered = B.paged_attn_decode_append(b.q, b.new_k, b.new_v, k2, v2, bt, sl, b.scale,
                                         seq_order=order)
    torch.cuda.synchronize()
    assert torch.equal(plain, ordered)
    assert torch.equal(k1.view(torch.int16), k2.view(torch.int16))
    assert_matches_oracle(ordered, oracle_decode(b), "ordered")


def test_bad_seq_order_entry_is_recorded_and_skipped(B):
    b = random_decode_batch(17, [40, 20, 60], 4, 64, 16, dtype="f16", device="cuda", poison=False)
    bt, sl = device_tables(b)
    order = torch.tensor([2, 7, 0], dtype=torch.int32, device="cuda")
    rec = B.new_error_record()
    out = torch.zeros(3, 4, 64, device="cuda")
    B.paged_attn_decode(b.q, b.k_cache, b.v_cache, bt, sl, b.scale, out=out, seq_order=order,
                        error_record=rec)
    assert B.pa_error_read(rec) == [6, 1, 1, 7]
    ref = oracle_decode(b, [0, 2])
    assert_matches_oracle(out[[0, 2]], ref, "valid entries")
    assert not out[1].any()                 # sequence 1 was not scheduled


def test_shared_prefix_equals_private_copy_bit_exact(B):
    """A sequence whose leading blocks are shared with another sequence decodes
    bit-identically to the same sequence holding private copies of those blocks
    (PagedAttention, "Sharing a prefix without copying it": sharing changes only
    the table, never what attention reads)."""
    lens = [700, 900, 40]
    bs = 16
    b = random_decode_batch(18, lens, 8, 128, bs, dtype="bf16", device="cuda", pool_factor=3.0,
                            poison=False)
    bt = b.block_tables.copy()
    n = lens[0] // bs                          # full blocks of sequence 0
    shared = bt.copy()
    shared[1, :n] = bt[0, :n]
    used = {int(x) for x in bt[bt >= 0]}
    free = [x for x in range(b.num_blocks) if x not in used][:n]
    assert len(free) == n
    pairs = torch.tensor([[int(bt[0, j]), free[j]] for j in range(n)], dtype=torch.int64,
                         device="cuda")
    B.block_copy([b.k_cache], [b.v_cache], pairs)
    private = bt.copy()
    private[1, :n] = free
    sl = torch.from_numpy(b.context_lens).cuda()
    for pt in (0, 64):
        out_s = B.paged_attn_decode(b.q, b.k_cache, b.v_cache, torch.from_numpy(shared).cuda(), sl,
                                    b.scale, partition_tokens=pt)
        out_p = B.paged_attn_decode(b.q, b.k_cache, b.v_cache, torch.from_numpy(private).cuda(),
                                    sl, b.scale, partition_tokens=pt)
        torch.cuda.synchronize()
        assert torch.equal(out_s, out_p)
    kc, dt = storage(b.k_cache)
    vc, _ = storage(b.v_cache)
    qs, _ = storage(b.q)
    k = OA.to_float64(OA.gather_sequence(kc, shared[1], lens[1], bs), dt)
    v = OA.to_float64(OA.gather_sequence(vc, shared[1], lens[1], bs), dt)
    ref = OA.attention(OA.to_float64(qs[1], dt), k, v, b.scale)
    assert_matches_oracle(out_s[1], ref, "shared prefix")


def test_work_items_change_nothing_but_the_schedule(B):
    """Running only the (sequence, partition) items that hold tokens, in any order,
    gives the same bits as the full grid; fused append included."""
    from paged_kv_cache_317_gb300.binding import partition_work_items
    lens = [5, 900, 2048, 1500, 64, 513, 2, 1100, 1, 512]
    b = random_decode_batch(22, lens, 8, 128, 16, dtype="bf16", device="cuda", with_append=True)
    bt, sl = device_tables(b)
    MB = b.max_blocks_per_seq
    for pt in (0, 256):
        k1, v1 = b.k_cache.clone(), b.v_cache.clone()
        plain = B.paged_attn_decode_append(b.q, b.new_k, b.new_v, k1, v1, bt, sl, b.scale,
                                           partition_tokens=pt)
        items = partition_work_items(b.context_lens, pt, MB, 16)
        for perm in (None, np.random.default_rng(pt).permutation(len(items))):
            it = items if perm is None else items[perm]
            k2, v2 = b.k_cache.clone(), b.v_cache.clone()
            got = B.paged_attn_decode_append(b.q, b.new_k, b.new_v, k2, v2, bt, sl, b.scale,
                                             partition_tokens=pt,
                                             work_items=torch.from_numpy(it).cuda())
            torch.cuda.synchronize()
            assert torch.equal(plain, got)
            assert torch.equal(k1.view(torch.int16), k2.view(torch.int16))
    assert_matches_oracle(plain, oracle_decode(b), "work items")


def test_bad_work_item_is_recorded_and_skipped(B):
    from paged_kv_cache_317_gb300.binding import partition_work_items
    b = random_decode_batch(23, [40, 20, 60], 4, 64, 16, dtype="f16", device="cuda", poison=False)
    bt, sl = device_tables(b)
    items = partition_work_items(b.context_lens, 0, b.max_blocks_per_seq, 16, order=[0, 1, 2])
    P = 1
    bad = np.array([items[0], 3 * P + 5, items[2]], dtype=np.int32)   # sequence 1 replaced
    rec = B.new_error_record()
    out = torch.zeros(3, 4, 64, device="cuda")
    B.paged_attn_decode(b.q, b.k_cache, b.v_cache, bt, sl, b.scale, out=out,
                        work_items=torch.from_numpy(bad).cuda(), error_record=rec)
    assert B.pa_error_read(rec) == [6, 1, 1, 3 * P + 5]
    assert_matches_oracle(out[[0, 2]], oracle_decode(b, [0, 2]), "valid items")
    assert not out[1].any()


@pytest.mark.parametrize("lens", [[1500], [900, 3, 2048, 40], [1, 17, 64, 65, 300] * 8, [95, 3, 191],
                                  [700] * 40 + [5, 2000]])
def test_host_schedule_matches_oracle(B, lens):
    """The partition length and work list the host schedule picks (short partitions
    for small batches) give the oracle's outputs, fused append included."""
    b = random_decode_batch(31 + len(lens), lens, 8, 128, 16, dtype="bf16", device="cuda",
                            with_append=True)
    pt = B.decode_partition_tokens(b.context_lens, 8)
    assert pt in (32, 64, 128, 256, 512)
    items = B.partition_work_items(b.context_lens, pt, b.max_blocks_per_seq, 16)
    bt, sl = device_tables(b)
    rec = B.new_error_record()
    out = B.paged_attn_decode_append(b.q, b.new_k, b.new_v, b.k_cache, b.v_cache, bt, sl,
                                     b.scale, out_dtype=torch.float32, partition_tokens=pt,
                                     work_items=torch.from_numpy(items).cuda(), error_record=rec)
    torch.cuda.synchronize()
    assert B.pa_error_read(rec) == [0, 0, 0, 0]
    assert_matches_oracle(out, oracle_decode(b), f"host schedule pt {pt}")


def test_bad_block_entry_in_the_second_half_of_a_chunk(B):
    """8-token blocks: a 16-token chunk reads two table entries; a bad second one is
    recorded and clamped too, and the other sequence is unaffected."""
    b = random_decode_batch(15, [40, 20], 4, 64, 8, dtype="f16", device="cuda", poison=False)
    bt, sl = device_tables(b)
    bt[1, 1] = b.num_blocks + 7           # tokens 8-15 of sequence 1
    rec = B.new_error_record()
    out = B.paged_attn_decode(b.q, b.k_cache, b.v_cache, bt, sl, b.scale, error_record=rec)
    r = B.pa_error_read(rec)
    assert r[0] == 4 and r[1] >= 1 and r[2] == 1 and r[3] == b.num_blocks + 7
    assert torch.isfinite(out).all()
    assert_matches_oracle(out[:1], oracle_decode(b, [0]), "unaffected sequence")


def test_largest_batch_the_call_takes(B):
    """65535 sequences (the most one call takes), short ragged lengths with one
    partition of 16 tokens each, fused append, host schedule (work list): sampled
    sequences against the oracle, every appended row bit-exact."""
    rng = np.random.default_rng(65535)
    lens = rng.integers(1, 41, 65535)
    b = random_decode_batch(9, lens, 2, 64, 16, dtype="f16", device="cuda", with_append=True,
                            poison=False)
    bt, sl = device_tables(b)
    pt = B.decode_partition_tokens(b.context_lens, 2)
    items = B.partition_work_items(b.context_lens, pt, b.max_blocks_per_seq, 16)
    assert len(items) == 65535                   # one item per sequence: the list's limit too
    rec = B.new_error_record()
    out = B.paged_attn_decode_append(b.q, b.new_k, b.new_v, b.k_cache, b.v_cache, bt, sl,
                                     b.scale, out_dtype=torch.float32, partition_tokens=pt,
                                     work_items=torch.from_numpy(items).cuda(),
                                     error_record=rec)
    torch.cuda.synchronize()
    assert B.pa_error_read(rec) == [0, 0, 0, 0]
    seqs = sorted(set(rng.choice(65535, 48, replace=False).tolist()) | {0, 65534})
    assert_matches_oracle(out[seqs], oracle_decode(b, seqs), "65535 sequences")
    slots = torch.from_numpy(b.slot_mapping).cuda()
    blk, row = slots // 16, slots % 16
    assert torch.equal(b.k_cache[blk, :, row], b.new_k) and torch.equal(b.v_cache[blk, :, row], b.new_v)
    with pytest.raises(B.PagedKVError):                     # one more sequence is refused
        B.paged_attn_decode(torch.cat([b.q, b.q[:1]]), b.k_cache, b.v_cache,
                            torch.cat([bt, bt[:1]]), torch.cat([sl, sl[:1]]), b.scale)
