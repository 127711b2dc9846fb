"""GPU parity of the fused append + decode call: bit-identical to append then
decode, within tolerance of the oracle, and the cache bit-exact."""

import numpy as np
import pytest
import torch

from gpu_util import assert_matches_oracle, bits, device_tables, oracle_decode
from oracle import cache_ops as OC
from workloads import decode_13b, random_decode_batch, tiny_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B(lib):
    from paged_kv_cache_317_gb300 import binding
    return binding


def _both(B, b, **kw):
    """(fused out, caches after fused) and (unfused out, caches after unfused)."""
    bt, sl = device_tables(b)
    k1, v1 = b.k_cache.clone(), b.v_cache.clone()
    rec = B.new_error_record()
    fused = B.paged_attn_decode_append(b.q, b.new_k, b.new_v, k1, v1, bt, sl, b.scale,
                                       error_record=rec, **kw)
    k2, v2 = b.k_cache.clone(), b.v_cache.clone()
    B.kv_cache_append(b.new_k, b.new_v, torch.from_numpy(b.slot_mapping).cuda(), k2, v2)
    plain = B.paged_attn_decode(b.q, k2, v2, bt, sl, b.scale, **kw)
    torch.cuda.synchronize()
    assert B.pa_error_read(rec) == [0, 0, 0, 0]
    return fused, (k1, v1), plain, (k2, v2)


@pytest.mark.parametrize("pt", [0, 16, 64])
def test_fused_tiny_matches_oracle_and_unfused(B, pt):
    b = tiny_decode(seed=1, device="cuda")
    ref = oracle_decode(b)
    fused, (k1, v1), plain, (k2, v2) = _both(B, b, partition_tokens=pt)
    assert torch.equal(fused, plain)
    assert_matches_oracle(fused, ref, "fused tiny")
    ek, ev = bits(b.k_cache), bits(b.v_cache)
    OC.kv_append(ek, ev, bits(b.new_k), bits(b.new_v), b.slot_mapping, b.block_size)
    assert np.array_equal(bits(k1), ek) and np.array_equal(bits(v1), ev)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("D,bs", [(64, 16), (128, 32), (256, 16), (128, 8), (64, 8)])
def test_fused_ragged_lengths(B, dtype, D, bs):
    lens = [1, 2, 16, 17, 32, 33, 511, 512, 513, 1000]
    b = random_decode_batch(300 + D + bs, lens, 4, D, bs, dtype=dtype, device="cuda",
                            with_append=True)
    ref = oracle_decode(b)
    for pt in (0, 32):
        fused, (k1, v1), plain, (k2, v2) = _both(B, b, partition_tokens=pt)
        assert torch.equal(fused, plain)
        assert torch.equal(k1.view(torch.int16), k2.view(torch.int16))
        assert torch.equal(v1.view(torch.int16), v2.view(torch.int16))
        assert_matches_oracle(fused, ref, f"fused {dtype} D{D} bs{bs} pt{pt}")


def test_fused_13b_full_size(B):
    b = decode_13b(device="cuda")
    seqs = list(range(0, 256, 11))
    ref = oracle_decode(b, seqs)
    fused, _, plain, _ = _both(B, b, out_dtype=torch.bfloat16)
    assert torch.equal(fused, plain)
    assert_matches_oracle(fused[seqs], ref, "fused 13B")



def test_bench_step_configuration(B):
    """The step bench.py times, on the batch it times: 13B-shaped lengths (seed 2),
    fused append, (sequence, partition) work items longest first, 512-token
    partitions, bf16 output, partition pass then merge pass with a preallocated
    workspace.  Every sequence against the oracle; appended rows bit for bit."""
    import numpy as np
    from paged_kv_cache_317_gb300.binding import partition_work_items
    b = decode_13b(seed=2, device="cuda", poison=False)
    N, H, D, bs, MB, pt = b.num_seqs, b.num_heads, b.head_dim, b.block_size, \
        b.max_blocks_per_seq, 512
    lens = b.context_lens
    ref = oracle_decode(b)
    bt = torch.from_numpy(b.block_tables).cuda()
    sl = torch.from_numpy(lens).cuda()
    items = torch.from_numpy(partition_work_items(
        lens, pt, MB, bs, order=np.argsort(-lens, kind="stable"))).cuda()
    out = torch.empty((N, H, D), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(B.paged_attn_workspace_size(N, H, D, bs, MB, pt), dtype=torch.uint8,
                     device="cuda")
    rec = B.new_error_record()
    for phases in (1, 2):
        B.paged_attn_decode_append(b.q, b.new_k, b.new_v, b.k_cache, b.v_cache, bt, sl, b.scale,
                                   out=out, partition_tokens=pt, workspace=ws, error_record=rec,
                                   phases=phases, work_items=items if phases == 1 else None)
    torch.cuda.synchronize()
    assert B.pa_error_read(rec) == [0, 0, 0, 0]
    slots = torch.from_numpy(b.slot_mapping).cuda()
    blk, row = slots // bs, slots % bs
    assert torch.equal(b.k_cache[blk, :, row, :].view(torch.int16), b.new_k.view(torch.int16))
    assert torch.equal(b.v_cache[blk, :, row, :].view(torch.int16), b.new_v.view(torch.int16))
    assert_matches_oracle(out, ref, "bench step, all 256 sequences")


def test_early_inputs_changes_nothing_eager_and_in_a_graph(B):
    """early_inputs lets the call's first kernel read its work item, length, table
    entries and query before the preceding kernel has completed; the caches, the
    shared workspace and `out` are still touched only after it.  Back-to-back calls
    on three batches that share one workspace (each call's partition pass writes
    the partials the previous call's merge reads), eagerly and replayed from a
    CUDA graph, give the same bits as without it."""
    batches = [random_decode_batch(900 + j, [1, 40, 300, 700, 1500 + 100 * j, 17], 8, 128, 16,
                                   dtype="bf16", device="cuda", with_append=True, poison=False)
               for j in range(3)]
    pt = 64
    ws = torch.empty(max(B.paged_attn_workspace_size(6, 8, 128, 16, b.max_blocks_per_seq, pt)
                         for b in batches), dtype=torch.uint8, device="cuda")
    tabs = [device_tables(b) for b in batches]
    items = [torch.from_numpy(B.partition_work_items(b.context_lens, pt, b.max_blocks_per_seq,
                                                     16)).cuda() for b in batches]

    def run(early, graph):
        caches = [(b.k_cache.clone(), b.v_cache.clone()) for b in batches]
        outs = [torch.empty(b.q.shape, dtype=torch.float32, device="cuda") for b in batches]

        def step():
            for _ in range(4):
                for b, (kc, vc), (bt, sl), it, o in zip(batches, caches, tabs, items, outs):
                    B.paged_attn_decode_append(b.q, b.new_k, b.new_v, kc, vc, bt, sl, b.scale,
                                               out=o, partition_tokens=pt, workspace=ws,
                                               work_items=it, early_inputs=early)
        if graph:
            step()                                   # warm-up outside the capture
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                step()
            for _ in range(3):
                g.replay()
        else:
            step()
        torch.cuda.synchronize()
        return outs, caches

    ref_outs, ref_caches = run(False, False)
    for early, graph in ((True, False), (True, True), (False, True)):
        outs, caches = run(early, graph)
        for o, r in zip(outs, ref_outs):
            assert torch.equal(o, r), (early, graph)
        for (k, v), (rk, rv) in zip(caches, ref_caches):
            assert torch.equal(k.view(torch.int16), rk.view(torch.int16))
            assert torch.equal(v.view(torch.int16), rv.view(torch.int16))
    for b, o in zip(batches, ref_outs):
        assert_matches_oracle(o, oracle_decode(b), "early-input chain")
