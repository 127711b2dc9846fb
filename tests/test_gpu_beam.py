"""Beam-search-style churn through the library: every step each beam group keeps
the survivors of a random score draw (forks of their parents; the old beams
end), every beam appends a token (copy-on-write of shared tails, batched into
one block_copy), and all beams decode.  The oracle tracks each beam's tokens
in logical order and recomputes every output (PagedAttention, zeroshotmind.com
page, "Sharing a prefix without copying it": candidates share everything up to
where they differ)."""

import pytest
import torch

from gpu_util import assert_matches_oracle
from oracle.content import LogicalSequences
from test_gpu_workloads import _oracle_logical
from workloads import beam_search

pytestmark = pytest.mark.gpu


def test_beam_search_churn(lib):
    from paged_kv_cache_317_gb300 import binding as B
    plan = beam_search(device="cuda")
    G, W, H, D, bs = plan.groups, plan.width, plan.num_heads, plan.head_dim, plan.block_size
    alloc = B.BlockAllocator(plan.num_blocks, bs, plan.free_order)
    kc = torch.full((plan.num_blocks, H, bs, D), float("nan"), dtype=plan.dtype, device="cuda")
    vc = torch.full_like(kc, float("nan"))
    content = LogicalSequences()
    rec = B.new_error_record()
    next_id = 0
    beams = []
    for g in range(G):
        a, e = int(plan.prompt_offsets[g]), int(plan.prompt_offsets[g + 1])
        root = next_id
        next_id += 1
        alloc.add(root, e - a)
        B.kv_cache_append(plan.prompt_k[a:e], plan.prompt_v[a:e],
                          torch.from_numpy(alloc.slots(root, 0, e - a)).cuda(), kc, vc,
                          error_record=rec)
        content.add(root, range(a, e))
        group = []
        for _ in range(W):
            alloc.fork(root, next_id)
            content.fork(root, next_id)
            group.append(next_id)
            next_id += 1
        alloc.free(root)
        content.free(root)
        beams.append(group)
    base = int(plan.prompt_offsets[-1])
    step_k = torch.empty((plan.steps * G * W, H, D), dtype=plan.dtype, device="cuda")
    step_v = torch.empty_like(step_k)
    max_blocks = int(-(-(plan.prompt_lens.max() + plan.steps + 1) // bs))
    total_copies = 0
    shared_parts = 0
    free_start = alloc.num_free()
    for s in range(plan.steps):
        new_beams = []
        for g in range(G):
            group = []
            for j in range(W):
                parent = beams[g][int(plan.parents[s, g, j])]
                alloc.fork(parent, next_id)
                content.fork(parent, next_id)
                group.append(next_id)
                next_id += 1
            for old in beams[g]:
                alloc.free(old)
                content.free(old)
            new_beams.append(group)
        beams = new_beams
        ids = [i for grp in beams for i in grp]
        slots, pairs = alloc.batch_append(ids)
        total_copies += len(pairs)
        if len(pairs):
            B.block_copy([kc], [vc], torch.from_numpy(pairs).cuda(), error_record=rec)
        q, k, v = plan.step_tokens(s)
        step_k[s * G * W:(s + 1) * G * W] = k
        step_v[s * G * W:(s + 1) * G * W] = v
        B.kv_cache_append(k, v, torch.from_numpy(slots).cuda(), kc, vc, error_record=rec)
        for n, i in enumerate(ids):
            content.append(i, base + s * G * W + n)
        tables, lens = alloc.batch_block_tables(ids, max_blocks)
        out = B.paged_attn_decode(q, kc, vc, torch.from_numpy(tables).cuda(),
                                  torch.from_numpy(lens).cuda(), plan.scale, error_record=rec)
        # and with the partitions the beams share read once per group
        items, recs = B.share_plan(tables, lens, 64, bs, fused_append=False)
        shared_parts += len(recs)
        out_sh = B.paged_attn_decode(q, kc, vc, torch.from_numpy(tables).cuda(),
                                     torch.from_numpy(lens).cuda(), plan.scale,
                                     partition_tokens=64, work_items=torch.from_numpy(items).cuda(),
                                     shared_records=torch.from_numpy(recs).cuda(),
                                     error_record=rec)
        alloc.check()
        if s % 5 == 4 or s == plan.steps - 1:
            k_st = [(0, plan.prompt_k), (base, step_k)]
            v_st = [(0, plan.prompt_v), (base, step_v)]
            for n, i in enumerate(ids):
                assert lens[n] == content.length(i)
                ref = _oracle_logical(q[n], content, i, k_st, v_st, plan.scale)
                assert_matches_oracle(out[n], ref, f"step {s} beam {i}")
                assert_matches_oracle(out_sh[n], ref, f"step {s} beam {i}, shared partitions")
    assert B.pa_error_read(rec) == [0, 0, 0, 0]
    assert total_copies > 0 and shared_parts > 0
    for grp in beams:
        for i in grp:
            alloc.free(i)
    assert alloc.num_free() == plan.num_blocks                 # nothing leaked
