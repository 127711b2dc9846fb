"""GPU parity on the five workloads at their full sizes.

The library (C++ allocator + kernels) runs each workload; the oracle recomputes
sampled outputs in fp64 from the generator's tensors.  For the sharing and
serving workloads the oracle does not look at block tables at all: it tracks
each sequence's tokens in logical order (oracle.content) and reads their values
from the generator's stores, so a wrong table, slot, copy or fork shows up as a
mismatch.
"""

import math

import numpy as np
import pytest
import torch

from gpu_util import assert_matches_oracle, device_tables, oracle_decode, storage
from oracle import attention as OA
from oracle.content import LogicalSequences
from workloads import decode_13b, long_context, mixed_serving, parallel_sampling

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B(lib):
    from paged_kv_cache_317_gb300 import binding
    return binding


def _sample(n, k, seed, always=()):
    rng = np.random.default_rng(seed)
    pick = set(int(i) for i in always)
    pick.update(int(i) for i in rng.choice(n, size=min(n, k), replace=False))
    return sorted(pick)


# --------------------------------------------------------------- 13B-shaped
def test_13b_decode_with_append(B):
    b = decode_13b(device="cuda")
    ref = oracle_decode(b)                            # reads the generator's pool before the append
    k0, v0 = b.k_cache.clone(), b.v_cache.clone()
    bt, sl = device_tables(b)
    slots = torch.from_numpy(b.slot_mapping).cuda()
    rec = B.new_error_record()
    B.kv_cache_append(b.new_k, b.new_v, slots, b.k_cache, b.v_cache, error_record=rec)
    out = B.paged_attn_decode(b.q, b.k_cache, b.v_cache, bt, sl, b.scale, error_record=rec)
    assert B.pa_error_read(rec) == [0, 0, 0, 0]
    assert torch.isfinite(out).all()
    # append: the slots hold the new rows bit for bit; every other slot is unchanged
    blk, row = slots // 16, slots % 16
    assert torch.equal(b.k_cache[blk, :, row, :].view(torch.int16), b.new_k.view(torch.int16))
    assert torch.equal(b.v_cache[blk, :, row, :].view(torch.int16), b.new_v.view(torch.int16))
    k0[blk, :, row, :] = b.new_k
    v0[blk, :, row, :] = b.new_v
    assert torch.equal(k0.view(torch.int16), b.k_cache.view(torch.int16))
    assert torch.equal(v0.view(torch.int16), b.v_cache.view(torch.int16))
    assert_matches_oracle(out, ref, "13B, all 256 sequences")


def test_13b_single_pass_and_split_agree_with_oracle(B):
    b = decode_13b(device="cuda", num_seqs=64, seed=22)
    ref = oracle_decode(b)
    bt, sl = device_tables(b)
    B.kv_cache_append(b.new_k, b.new_v, torch.from_numpy(b.slot_mapping).cuda(), b.k_cache,
                      b.v_cache)
    for pt in (0, 256, 4096):
        out = B.paged_attn_decode(b.q, b.k_cache, b.v_cache, bt, sl, b.scale, partition_tokens=pt)
        assert_matches_oracle(out, ref, f"13B pt{pt}")


# ------------------------------------------------------------- long context
@pytest.mark.parametrize("bs", [16, 32])
def test_long_context_split_k(B, bs):
    b = long_context(device="cuda", block_size=bs)
    bt, sl = device_tables(b)
    rec = B.new_error_record()
    out = B.paged_attn_decode(b.q, b.k_cache, b.v_cache, bt, sl, b.scale, partition_tokens=512,
                              error_record=rec)
    assert B.pa_error_read(rec) == [0, 0, 0, 0]
    assert torch.isfinite(out).all()
    # the first and last sequence (the first and last blocks of the launch) and
    # six more drawn at random: 8 of 32
    inner = np.random.default_rng(40 + bs).choice(np.arange(1, b.num_seqs - 1), 6, replace=False)
    seqs = sorted({0, b.num_seqs - 1, *(int(i) for i in inner)})
    assert len(seqs) == 8
    assert_matches_oracle(out[seqs], oracle_decode(b, seqs), f"long bs{bs}")


# ------------------------------------------------- shared prompts + CoW copies
def _gather(stores, origins, device="cuda"):
    """Rows of concatenated value stores: stores = [(base, tensor), ...] in base order."""
    o = torch.from_numpy(origins).to(device)
    out = torch.empty((len(origins),) + tuple(stores[0][1].shape[1:]), dtype=stores[0][1].dtype,
                      device=device)
    for j, (base, t) in enumerate(stores):
        hi = stores[j + 1][0] if j + 1 < len(stores) else None
        m = (o >= base) if hi is None else ((o >= base) & (o < hi))
        if m.any():
            out[m] = t[o[m] - base]
    return out


def _oracle_logical(q_row, content, seq, k_stores, v_stores, scale):
    origins = content.rows(seq)
    k, dt = storage(_gather(k_stores, origins))
    v, _ = storage(_gather(v_stores, origins))
    qs, _ = storage(q_row)
    return OA.attention(OA.to_float64(qs, dt), OA.to_float64(k, dt), OA.to_float64(v, dt), scale)


@pytest.mark.parametrize("partial", [True, False])
def test_parallel_sampling_with_copy_on_write(B, partial):
    from paged_kv_cache_317_gb300.binding import BlockAllocator
    plan = parallel_sampling(device="cuda", partial_prefix=partial)
    P, S, H, D, bs = plan.num_prompts, plan.samples, plan.num_heads, plan.head_dim, plan.block_size
    N = plan.num_seqs
    alloc = BlockAllocator(plan.num_blocks, bs, plan.free_order)
    kc = torch.full((plan.num_blocks, H, bs, D), float("nan"), dtype=plan.dtype, device="cuda")
    vc = torch.full_like(kc, float("nan"))
    content = LogicalSequences()
    tail_base = int(plan.prompt_offsets[-1])
    rec = B.new_error_record()
    # prompts, written once each through the append kernel
    for k in range(P):
        a, e = int(plan.prompt_offsets[k]), int(plan.prompt_offsets[k + 1])
        alloc.add(k * S, e - a)
        slots = torch.from_numpy(alloc.slots(k * S, 0, e - a)).cuda()
        B.kv_cache_append(plan.prompt_k[a:e], plan.prompt_v[a:e], slots, kc, vc, error_record=rec)
        content.add(k * S, range(a, e))
    for k in range(P):
        for s in range(1, S):
            alloc.fork(k * S, k * S + s)
            content.fork(k * S, k * S + s)
    # first divergent token of every sample, in sample order
    ids = list(range(N))
    slots, pairs = alloc.batch_append(ids)
    expected_copies = P * (S - 1) if partial else 0
    assert len(pairs) == expected_copies
    if len(pairs):
        B.block_copy([kc], [vc], torch.from_numpy(pairs).cuda(), error_record=rec)
    first = plan.tail_offsets[:-1].astype(np.int64)
    fi = torch.from_numpy(first).cuda()
    B.kv_cache_append(plan.tail_k[fi], plan.tail_v[fi], torch.from_numpy(slots).cuda(), kc, vc,
                      error_record=rec)
    for i in ids:
        content.append(i, tail_base + int(first[i]))
    # the rest of each tail
    rest_rows, rest_slots = [], []
    for i in ids:
        for t in range(1, int(plan.tail_lens[i])):
            slot, cow = alloc.append(i)
            assert cow is None                  # tails are private
            rest_rows.append(int(plan.tail_offsets[i]) + t)
            rest_slots.append(slot)
            content.append(i, tail_base + rest_rows[-1])
    rows = torch.tensor(rest_rows, dtype=torch.long, device="cuda")
    B.kv_cache_append(plan.tail_k[rows], plan.tail_v[rows],
                      torch.tensor(rest_slots, dtype=torch.int64, device="cuda"), kc, vc,
                      error_record=rec)
    alloc.check()
    # every sample of a prompt shares its full prefix blocks
    for k in range(P):
        base_t = alloc.block_table(k * S)
        full = int(plan.prompt_lens[k]) // bs
        for s in range(1, S):
            assert alloc.block_table(k * S + s)[:full] == base_t[:full]
            assert alloc.refcount(base_t[0]) == S
    mb = max(len(alloc.block_table(i)) for i in ids)
    tables, lens = alloc.batch_block_tables(ids, mb)
    out = B.paged_attn_decode(plan.q, kc, vc, torch.from_numpy(tables).cuda(),
                              torch.from_numpy(lens).cuda(), plan.scale, error_record=rec)
    assert B.pa_error_read(rec) == [0, 0, 0, 0]
    assert torch.isfinite(out).all()
    k_st = [(0, plan.prompt_k), (tail_base, plan.tail_k)]
    v_st = [(0, plan.prompt_v), (tail_base, plan.tail_v)]
    seqs = _sample(N, 40, 3, always=range(S))
    # the same decode reading each prompt's shared partitions once for all samples
    items, recs = B.share_plan(tables, lens, 512, bs, fused_append=False)
    assert len(recs) == P * 2 and (recs[:, 1] == S).all()      # tokens 0..1023 of each prompt
    out_sh = B.paged_attn_decode(plan.q, kc, vc, torch.from_numpy(tables).cuda(),
                                 torch.from_numpy(lens).cuda(), plan.scale, partition_tokens=512,
                                 work_items=torch.from_numpy(items).cuda(),
                                 shared_records=torch.from_numpy(recs).cuda(), error_record=rec)
    assert B.pa_error_read(rec) == [0, 0, 0, 0]
    for i in seqs:
        assert lens[i] == content.length(i)
        ref = _oracle_logical(plan.q[i], content, i, k_st, v_st, plan.scale)
        assert_matches_oracle(out[i], ref, f"sampling seq {i}")
        assert_matches_oracle(out_sh[i], ref, f"sampling seq {i}, shared partitions")


# --------------------------------------------------------------- mixed serving
def _run_mixed(B, plan, check_every, sample_per_step, full_steps):
    from paged_kv_cache_317_gb300.binding import BlockAllocator
    N, H, D, bs = plan.num_seqs, plan.num_heads, plan.head_dim, plan.block_size
    alloc = BlockAllocator(plan.num_blocks, bs, plan.free_order)
    kc = torch.full((plan.num_blocks, H, bs, D), float("nan"), dtype=plan.dtype, device="cuda")
    vc = torch.full_like(kc, float("nan"))
    content = LogicalSequences()
    rec = B.new_error_record()
    ids = list(range(N))
    next_id = N
    all_slots = []
    for b in range(N):
        a, e = int(plan.init_offsets[b]), int(plan.init_offsets[b + 1])
        alloc.add(b, e - a)
        all_slots.append(alloc.slots(b, 0, e - a))
        content.add(b, range(a, e))
    B.kv_cache_append(plan.init_k, plan.init_v, torch.from_numpy(np.concatenate(all_slots)).cuda(),
                      kc, vc, error_record=rec)
    step_base = int(plan.init_offsets[-1])
    step_k = torch.empty((plan.steps * N, H, D), dtype=plan.dtype, device="cuda")
    step_v = torch.empty_like(step_k)
    max_blocks = int(math.ceil((plan.init_lens.max() + plan.steps) / bs))
    copies = 0
    for s in range(plan.steps):
        for a, b in plan.fork_pairs[s]:
            alloc.free(ids[b])
            content.free(ids[b])
            alloc.fork(ids[a], next_id)
            content.fork(ids[a], next_id)
            ids[b] = next_id
            next_id += 1
        slots, pairs = alloc.batch_append(ids)
        copies += len(pairs)
        if len(pairs):
            B.block_copy([kc], [vc], torch.from_numpy(pairs).cuda(), error_record=rec)
        q, k, v = plan.step_tokens(s)
        step_k[s * N:(s + 1) * N] = k
        step_v[s * N:(s + 1) * N] = v
        B.kv_cache_append(k, v, torch.from_numpy(slots).cuda(), kc, vc, error_record=rec)
        for b in range(N):
            content.append(ids[b], step_base + s * N + b)
        tables, lens = alloc.batch_block_tables(ids, max_blocks)
        out = B.paged_attn_decode(q, kc, vc, torch.from_numpy(tables).cuda(),
                                  torch.from_numpy(lens).cuda(), plan.scale, error_record=rec)
        if s % check_every == 0 or s in full_steps:
            torch.cuda.synchronize()
            assert torch.isfinite(out).all(), f"step {s}"
            picks = range(N) if s in full_steps else _sample(N, sample_per_step, 1000 + s)
            k_st = [(0, plan.init_k), (step_base, step_k)]
            v_st = [(0, plan.init_v), (step_base, step_v)]
            for b in picks:
                assert lens[b] == content.length(ids[b])
                ref = _oracle_logical(q[b], content, ids[b], k_st, v_st, plan.scale)
                assert_matches_oracle(out[b], ref, f"step {s} slot {b}")
    alloc.check()
    assert B.pa_error_read(rec) == [0, 0, 0, 0]
    return copies


def test_mixed_serving_small_every_output(B):
    plan = mixed_serving(device="cuda", num_seqs=48, steps=12, long=(300, 700), seed=55)
    copies = _run_mixed(B, plan, check_every=1, sample_per_step=48, full_steps=set(range(12)))
    assert copies > 0


def test_mixed_serving_full_size(B):
    plan = mixed_serving(device="cuda")
    copies = _run_mixed(B, plan, check_every=1, sample_per_step=3, full_steps={0, 49, 99})
    assert copies > 0
