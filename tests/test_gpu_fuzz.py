"""Seeded randomized parity sweep: decode and prefill on random shapes, dtypes,
block sizes, launch shapes and schedules, each checked against the oracle."""

import numpy as np
import pytest
import torch

from gpu_util import assert_matches_oracle, device_tables, oracle_decode, storage
from oracle import attention as OA
from workloads import random_decode_batch
from workloads.gen import _torch_gen, randn_rounded

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B(lib):
    from paged_kv_cache_317_gb300 import binding
    return binding


@pytest.mark.parametrize("seed", range(48))
def test_decode_random_configuration(B, seed):
    _random_decode_case(B, seed)


@pytest.mark.parametrize("seed", range(16))
def test_decode_random_configuration_8_token_blocks(B, seed):
    """8-token blocks: every 16-token chunk spans two blocks."""
    _random_decode_case(B, 500 + seed, block_size=8)


def _random_decode_case(B, seed, block_size=None):
    from paged_kv_cache_317_gb300.binding import partition_work_items
    rng = np.random.default_rng(1000 + seed)
    D = int(rng.choice([64, 128, 256]))
    bs = int(rng.choice([16, 32, 48]))
    if block_size is not None:
        bs = block_size
    H = int(rng.choice([1, 2, 3, 4, 8, 12]))
    N = int(rng.integers(1, 12))
    dtype = str(rng.choice(["f16", "bf16"]))
    lens = [int(x) for x in rng.integers(0, 1500, size=N)]
    append = bool(rng.integers(0, 2))
    if append:
        lens = [max(1, L) for L in lens]
    b = random_decode_batch(2000 + seed, lens, H, D, bs, dtype=dtype, device="cuda",
                            with_append=append, pool_factor=float(rng.uniform(1.2, 3.0)))
    bt, sl = device_tables(b)
    # launch shapes whose shared-memory ring fits a block (S stages x G heads x K+V chunks)
    shapes = [(g, s_) for g in (1, 2, 3, 4, 8) for s_ in (2, 3, 4)
              if H % g == 0 and 256 + s_ * g * 2 * 16 * D * 2 <= 227 * 1024]
    G, S = shapes[int(rng.integers(0, len(shapes)))]
    pt = int(rng.choice([0, 16, 64, 256, 512]))
    out_dtype = [torch.float32, torch.float16, torch.bfloat16][int(rng.integers(0, 3))]
    sched = {}
    choice = int(rng.integers(0, 4))
    if choice == 1:
        sched["seq_order"] = torch.from_numpy(rng.permutation(N).astype(np.int32)).cuda()
    elif choice == 2:
        items = partition_work_items(b.context_lens, pt, b.max_blocks_per_seq, bs)
        sched["work_items"] = torch.from_numpy(rng.permutation(items).astype(np.int32)).cuda()
    elif choice == 3:
        # the host schedule; a random SM count spreads its choice over 64..512
        pt = B.decode_partition_tokens(b.context_lens, H, G, int(rng.choice([1, 4, 152])))
        items = partition_work_items(b.context_lens, pt, b.max_blocks_per_seq, bs)
        sched["work_items"] = torch.from_numpy(items).cuda()
    rec = B.new_error_record()
    if append:
        out = B.paged_attn_decode_append(b.q, b.new_k, b.new_v, b.k_cache, b.v_cache, bt, sl,
                                         b.scale, out_dtype=out_dtype, partition_tokens=pt,
                                         heads_per_cta=G, stages=S, error_record=rec, **sched)
    else:
        out = B.paged_attn_decode(b.q, b.k_cache, b.v_cache, bt, sl, b.scale,
                                  out_dtype=out_dtype, partition_tokens=pt, heads_per_cta=G,
                                  stages=S, error_record=rec, **sched)
    torch.cuda.synchronize()
    assert B.pa_error_read(rec) == [0, 0, 0, 0]
    assert_matches_oracle(out, oracle_decode(b),
                          f"seed {seed}: D{D} bs{bs} H{H} N{N} {dtype} G{G} S{S} pt{pt} "
                          f"append={append} sched={list(sched)}")


@pytest.mark.parametrize("seed", range(32))
def test_prefill_random_configuration(B, seed):
    _random_prefill_case(B, seed)


@pytest.mark.parametrize("seed", range(8))
def test_prefill_random_configuration_8_token_blocks(B, seed):
    """8-token blocks: every 16-key chunk is loaded as two 8-row boxes."""
    _random_prefill_case(B, 500 + seed, block_size=8)


def _random_prefill_case(B, seed, block_size=None):
    rng = np.random.default_rng(3000 + seed)
    D = int(rng.choice([64, 128, 256]))
    bs = int(rng.choice([16, 32]))
    if block_size is not None:
        bs = block_size
    H = int(rng.integers(1, 5))
    N = int(rng.integers(1, 5))
    dtype = str(rng.choice(["f16", "bf16"]))
    lens = [int(x) for x in rng.integers(1, 900, size=N)]
    nq = [min(L, int(rng.integers(0, 257))) if rng.random() < 0.8 else min(L, 300) for L in lens]
    b = random_decode_batch(4000 + seed, lens, H, D, bs, dtype=dtype, device="cuda")
    q = randn_rounded((max(1, sum(nq)), H, D), b.dtype, _torch_gen(5000 + seed, "cuda"),
                      "cuda")
    starts = np.concatenate([[0], np.cumsum(nq)]).astype(np.int32)
    out_dtype = [torch.float32, torch.float16, torch.bfloat16][int(rng.integers(0, 3))]
    rec = B.new_error_record()
    out = B.paged_attn_prefill(q, torch.from_numpy(starts).cuda(), max(1, max(nq)), b.k_cache,
                               b.v_cache, torch.from_numpy(b.block_tables).cuda(),
                               torch.from_numpy(b.context_lens).cuda(), b.scale,
                               out_dtype=out_dtype, error_record=rec)
    torch.cuda.synchronize()
    assert B.pa_error_read(rec) == [0, 0, 0, 0]
    qs, dt = storage(q)
    kc, _ = storage(b.k_cache)
    vc, _ = storage(b.v_cache)
    ref = OA.paged_prefill_attention(qs, kc, vc, b.block_tables, b.context_lens, starts, b.scale,
                                     bs, dt)
    assert_matches_oracle(out[: starts[-1]], ref,
                          f"seed {seed}: D{D} bs{bs} H{H} N{N} {dtype} nq={nq} lens={lens}")
