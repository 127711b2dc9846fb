"""GPU parity of the tensor-core chunked prefill against the fp64 oracle."""

import numpy as np
import pytest
import torch

from gpu_util import assert_matches_oracle, storage
from oracle import attention as OA
from workloads import random_decode_batch
from workloads.gen import _torch_gen, randn_rounded

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B(lib):
    from paged_kv_cache_317_gb300 import binding
    return binding


def _case(seed, lens, nq, H, bs, dtype, poison=True, D=128):
    b = random_decode_batch(seed, lens, H, D, bs, dtype=dtype, device="cuda", poison=poison)
    g = _torch_gen(seed + 7, "cuda")
    q = randn_rounded((int(sum(nq)), H, D), b.dtype, g, "cuda")
    starts = np.concatenate([[0], np.cumsum(nq)]).astype(np.int32)
    return b, q, starts


def _run(B, b, q, starts, out_dtype=torch.float32, rec=None):
    return B.paged_attn_prefill(q, torch.from_numpy(starts).cuda(), int(np.diff(starts).max()),
                                b.k_cache, b.v_cache, torch.from_numpy(b.block_tables).cuda(),
                                torch.from_numpy(b.context_lens).cuda(), b.scale,
                                out_dtype=out_dtype, error_record=rec)


def _oracle(b, q, starts, seqs=None):
    qs, dt = storage(q)
    kc, _ = storage(b.k_cache)
    vc, _ = storage(b.v_cache)
    return OA.paged_prefill_attention(qs, kc, vc, b.block_tables, b.context_lens, starts, b.scale,
                                      b.block_size, dt, seqs)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("bs", [8, 16, 32])
def test_prefill_small_cases(B, dtype, bs):
    lens = [5, 300, 1000, 17, 129, 64]
    nq = [5, 64, 200, 1, 129, 3]            # whole-sequence prefill, chunks, one query
    b, q, starts = _case(40 + bs, lens, nq, 2, bs, dtype)
    rec = B.new_error_record()
    out = _run(B, b, q, starts, rec=rec)
    torch.cuda.synchronize()
    assert B.pa_error_read(rec) == [0, 0, 0, 0]
    assert_matches_oracle(out, _oracle(b, q, starts), f"prefill {dtype} bs{bs}")


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float16])
def test_prefill_half_outputs(B, out_dtype, D):
    """16-bit outputs leave through the staging buffer as 32 columns per 64-byte
    piece (fp32 ones as 16): every head_dim's column count."""
    b, q, starts = _case(50, [200, 90], [130, 90], 4, 16, "bf16", D=D)
    assert_matches_oracle(_run(B, b, q, starts, out_dtype=out_dtype), _oracle(b, q, starts))


def test_single_query_prefill_matches_decode(B):
    lens = [1, 40, 513, 2000]
    b = random_decode_batch(60, lens, 8, 128, 16, dtype="bf16", device="cuda")
    starts = np.arange(len(lens) + 1, dtype=np.int32)
    out = _run(B, b, b.q, starts)
    dec = B.paged_attn_decode(b.q, b.k_cache, b.v_cache, torch.from_numpy(b.block_tables).cuda(),
                              torch.from_numpy(b.context_lens).cuda(), b.scale)
    torch.cuda.synchronize()
    assert (out - dec).abs().max().item() <= 2e-3
    assert_matches_oracle(out, _oracle(b, b.q, starts))


def test_prefill_13b_shaped_chunks_sampled(B):
    """16 sequences x 40 heads; each appends a 512-token chunk to a context of up to
    2048 tokens.  The oracle checks two sequences in full and sampled rows of others."""
    rng = np.random.default_rng(70)
    lens = rng.integers(512, 2049, size=16)
    nq = np.full(16, 512)
    b, q, starts = _case(70, lens, nq, 40, 16, "bf16", poison=False)
    out = _run(B, b, q, starts)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all()
    qs, dt = storage(q)
    kc, _ = storage(b.k_cache)
    vc, _ = storage(b.v_cache)
    for i in (0, 9):
        a, e = starts[i], starts[i + 1]
        ref = OA.paged_prefill_attention(qs, kc, vc, b.block_tables, b.context_lens, starts,
                                         b.scale, 16, dt, seqs=[i])
        assert_matches_oracle(out[a:e], ref, f"seq {i}")
    for i in (3, 15):
        L = int(lens[i])
        k = OA.to_float64(OA.gather_sequence(kc, b.block_tables[i], L, 16), dt)
        v = OA.to_float64(OA.gather_sequence(vc, b.block_tables[i], L, 16), dt)
        for j in (0, 1, 127, 128, 255, 300, 511):
            p = L - 512 + j
            ref = OA.attention(OA.to_float64(qs[starts[i] + j], dt), k[: p + 1], v[: p + 1],
                               b.scale)
            assert_matches_oracle(out[starts[i] + j], ref, f"seq {i} row {j}")


def test_prefill_bad_query_range_is_recorded_and_skipped(B):
    b, q, starts = _case(80, [50, 60], [10, 20], 2, 16, "bf16", poison=False)
    bad = starts.copy()
    bad[1] = 45                              # sequence 0 claims 45 queries > nothing wrong yet
    bad[2] = 30 + 60                         # sequence 1 range past the end of q
    rec = B.new_error_record()
    out = torch.zeros((q.shape[0], 2, 128), device="cuda")
    B.paged_attn_prefill(q, torch.from_numpy(bad).cuda(), 60, b.k_cache, b.v_cache,
                         torch.from_numpy(b.block_tables).cuda(),
                         torch.from_numpy(b.context_lens).cuda(), b.scale, out=out,
                         error_record=rec)
    r = B.pa_error_read(rec)
    assert r[0] == 6 and r[1] >= 1


def test_prefill_is_deterministic_across_launches(B):
    """Repeated launches give bit-identical outputs (a race on a TMEM or shared
    buffer would show up as run-to-run differences)."""
    rng = np.random.default_rng(90)
    lens = rng.integers(200, 1500, size=24)
    nq = np.minimum(lens, rng.integers(1, 400, size=24))
    b, q, starts = _case(90, lens, nq, 8, 16, "bf16", poison=False)
    first = _run(B, b, q, starts)
    for _ in range(4):
        again = _run(B, b, q, starts)
        torch.cuda.synchronize()
        assert torch.equal(first, again)
    assert_matches_oracle(first[: starts[3]], _oracle(b, q, starts, seqs=[0, 1, 2]), "determinism")


def test_prefill_long_context_many_tiles(B):
    """16K-token contexts: every ring and barrier phase wraps around many times."""
    lens = [16384, 12001]
    nq = [200, 77]
    b, q, starts = _case(95, lens, nq, 4, 32, "bf16", poison=True)
    rec = B.new_error_record()
    out = _run(B, b, q, starts, rec=rec)
    torch.cuda.synchronize()
    assert B.pa_error_read(rec) == [0, 0, 0, 0]
    assert_matches_oracle(out, _oracle(b, q, starts), "long prefill")


def test_prefill_sequences_without_queries_are_skipped(B):
    """Sequences with no queries in the launch (query_start[i] == query_start[i+1])
    write nothing; the others are unaffected."""
    lens = [300, 120, 0, 900]
    nq = [40, 0, 0, 130]
    b, q, starts = _case(97, lens, nq, 4, 16, "bf16")
    rec = B.new_error_record()
    out = _run(B, b, q, starts, rec=rec)
    torch.cuda.synchronize()
    assert B.pa_error_read(rec) == [0, 0, 0, 0]
    assert_matches_oracle(out, _oracle(b, q, starts, seqs=[0, 3]), "skipped sequences")


def test_prefill_bad_block_entry_is_recorded_and_clamped(B):
    b, q, starts = _case(98, [200, 150], [64, 50], 2, 16, "bf16", poison=False)
    bt = torch.from_numpy(b.block_tables).cuda()
    bt[1, 2] = b.num_blocks + 9
    rec = B.new_error_record()
    out = B.paged_attn_prefill(q, torch.from_numpy(starts).cuda(), 64, b.k_cache, b.v_cache, bt,
                               torch.from_numpy(b.context_lens).cuda(), b.scale,
                               error_record=rec)
    torch.cuda.synchronize()
    r = B.pa_error_read(rec)
    assert r[0] == 4 and r[1] >= 1 and r[2] == 1 and r[3] == b.num_blocks + 9
    assert torch.isfinite(out).all()
    assert_matches_oracle(out[: starts[1]], _oracle(b, q, starts, seqs=[0]), "unaffected sequence")


@pytest.mark.parametrize("D", [64, 256])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_prefill_other_head_dims(B, D, dtype):
    """head_dim 64 (two blocks per SM) and 256 (512 TMEM columns, one block per SM)."""
    lens = [5, 300, 1000, 17, 129, 700]
    nq = [5, 64, 200, 1, 129, 256]
    b, q, starts = _case(60 + D, lens, nq, 3, 16, dtype, D=D)
    rec = B.new_error_record()
    out = _run(B, b, q, starts, rec=rec)
    torch.cuda.synchronize()
    assert B.pa_error_read(rec) == [0, 0, 0, 0]
    assert_matches_oracle(out, _oracle(b, q, starts), f"prefill D{D} {dtype}")
    again = _run(B, b, q, starts)
    torch.cuda.synchronize()
    assert torch.equal(out, again)


def test_prefill_seq_order_changes_nothing_but_the_schedule(B):
    rng = np.random.default_rng(99)
    lens = rng.integers(200, 1500, size=9)
    nq = np.minimum(lens, rng.integers(1, 300, size=9))
    b, q, starts = _case(99, lens, nq, 4, 16, "bf16", poison=False)
    plain = _run(B, b, q, starts)
    for order in (np.argsort(-lens, kind="stable"), rng.permutation(9)):
        got = B.paged_attn_prefill(q, torch.from_numpy(starts).cuda(), int(nq.max()), b.k_cache,
                                   b.v_cache, torch.from_numpy(b.block_tables).cuda(),
                                   torch.from_numpy(b.context_lens).cuda(), b.scale,
                                   seq_order=torch.from_numpy(order.astype(np.int32)).cuda())
        torch.cuda.synchronize()
        assert torch.equal(plain, got)
    bad = torch.tensor([0, 1, 2, 3, 40, 5, 6, 7, 8], dtype=torch.int32, device="cuda")
    rec = B.new_error_record()
    out = torch.zeros_like(plain)
    B.paged_attn_prefill(q, torch.from_numpy(starts).cuda(), int(nq.max()), b.k_cache, b.v_cache,
                         torch.from_numpy(b.block_tables).cuda(),
                         torch.from_numpy(b.context_lens).cuda(), b.scale, out=out,
                         seq_order=bad, error_record=rec)
    torch.cuda.synchronize()
    assert B.pa_error_read(rec) == [6, 1, 4, 40]
    assert not out[starts[4]:starts[5]].any()                # sequence 4 was not dispatched
    assert torch.equal(out[: starts[4]], plain[: starts[4]])


def test_prefill_many_items_per_block(B):
    """Far more (sequence, query tile, head) items than resident blocks: each block
    runs ~30 items in turn, many of them empty (query tiles past a short chunk),
    so every barrier's phase is carried across items of different lengths."""
    rng = np.random.default_rng(101)
    n = 600
    lens = rng.integers(20, 700, size=n)
    nq = np.minimum(lens, rng.choice([1, 3, 64, 128, 129, 200, 256], size=n))
    b, q, starts = _case(101, lens, nq, 8, 16, "bf16", poison=True)
    rec = B.new_error_record()
    out = _run(B, b, q, starts, rec=rec)
    again = _run(B, b, q, starts)
    torch.cuda.synchronize()
    assert B.pa_error_read(rec) == [0, 0, 0, 0]
    assert torch.equal(out, again)
    seqs = sorted({0, 1, n - 1} | set(rng.choice(n, size=12, replace=False).tolist()))
    ref = _oracle(b, q, starts, seqs=seqs)
    rows = np.concatenate([np.arange(starts[i], starts[i + 1]) for i in seqs])
    assert_matches_oracle(out[torch.from_numpy(rows).cuda()], ref, "many items per block")


def test_prefill_bad_ranges_between_good_items(B):
    """Sequences whose query range is invalid (more queries than tokens) are
    recorded and skipped by every role of the block alike: the items around them,
    in the same blocks, stay correct."""
    rng = np.random.default_rng(103)
    n = 400
    lens = rng.integers(100, 600, size=n)
    nq = np.minimum(lens, rng.integers(1, 200, size=n))
    b, q, starts = _case(103, lens, nq, 4, 16, "bf16", poison=False)
    bad = np.arange(5, n, 7)
    seen = b.context_lens.copy()
    seen[bad] = nq[bad] - 1                   # fewer tokens than queries: invalid
    rec = B.new_error_record()
    out = torch.zeros((q.shape[0], 4, 128), device="cuda")
    B.paged_attn_prefill(q, torch.from_numpy(starts).cuda(), int(nq.max()), b.k_cache,
                         b.v_cache, torch.from_numpy(b.block_tables).cuda(),
                         torch.from_numpy(seen).cuda(), b.scale, out=out, error_record=rec)
    torch.cuda.synchronize()
    r = B.pa_error_read(rec)
    assert r[0] == 6 and r[2] in set(bad.tolist())
    for i in bad[:5]:
        assert not out[starts[i]:starts[i + 1]].any()
    good = [i for i in range(n) if i % 7 != 5]
    seqs = sorted(set(rng.choice(good, size=14, replace=False).tolist()) | {good[0], good[-1]})
    ref = _oracle(b, q, starts, seqs=seqs)
    rows = np.concatenate([np.arange(starts[i], starts[i + 1]) for i in seqs])
    assert_matches_oracle(out[torch.from_numpy(rows).cuda()], ref, "good items among bad")
