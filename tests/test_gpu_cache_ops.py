"""GPU parity of kv_cache_append and block_copy: bit-exact against the oracle's
element-wise copies over the whole pool (untouched bytes included)."""

import numpy as np
import pytest
import torch

from gpu_util import bits
from oracle import cache_ops as OC
from workloads.gen import _torch_gen, randn_rounded

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B(lib):
    from paged_kv_cache_317_gb300 import binding
    return binding


def _pool(seed, nb, H, bs, D, dtype):
    g = _torch_gen(seed, "cuda")
    return (randn_rounded((nb, H, bs, D), dtype, g, "cuda"),
            randn_rounded((nb, H, bs, D), dtype, g, "cuda"))


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("H,D,bs,T", [(8, 64, 16, 37), (40, 128, 16, 256), (32, 128, 32, 512),
                                      (3, 8, 16, 5), (2, 256, 48, 100)])
def test_append_is_bit_exact(B, dtype, H, D, bs, T):
    nb = max(8, 3 * T // bs + 4)
    kc, vc = _pool(1, nb, H, bs, D, dtype)
    g = _torch_gen(2, "cuda")
    k = randn_rounded((T, H, D), dtype, g, "cuda")
    v = randn_rounded((T, H, D), dtype, g, "cuda")
    rng = np.random.default_rng(T)
    slots = rng.choice(nb * bs, size=T, replace=False).astype(np.int64)
    slots[rng.random(T) < 0.1] = -1                    # padding tokens
    ek, ev = bits(kc), bits(vc)
    OC.kv_append(ek, ev, bits(k), bits(v), slots, bs)
    rec = B.new_error_record()
    B.kv_cache_append(k, v, torch.from_numpy(slots).cuda(), kc, vc, error_record=rec)
    assert B.pa_error_read(rec) == [0, 0, 0, 0]
    assert np.array_equal(bits(kc), ek) and np.array_equal(bits(vc), ev)


def test_append_out_of_range_slot_is_recorded_and_skipped(B):
    kc, vc = _pool(3, 4, 2, 16, 64, torch.float16)
    k = torch.ones(3, 2, 64, dtype=torch.float16, device="cuda")
    before_k, before_v = bits(kc), bits(vc)
    slots = torch.tensor([5, 4 * 16, 7], dtype=torch.int64, device="cuda")
    rec = B.new_error_record()
    B.kv_cache_append(k, k, slots, kc, vc, error_record=rec)
    assert B.pa_error_read(rec) == [5, 1, 1, 64]
    OC.kv_append(before_k, before_v, bits(k), bits(k), [5, -1, 7], 16)
    assert np.array_equal(bits(kc), before_k) and np.array_equal(bits(vc), before_v)


@pytest.mark.parametrize("layers", [1, 3])
@pytest.mark.parametrize("H,D,bs", [(40, 128, 16), (8, 64, 32), (2, 8, 16)])
def test_block_copy_is_bit_exact(B, layers, H, D, bs):
    nb = 64
    pools = [_pool(10 + l, nb, H, bs, D, torch.bfloat16) for l in range(layers)]
    ks, vs = [p[0] for p in pools], [p[1] for p in pools]
    rng = np.random.default_rng(layers * 7 + H)
    pick = rng.choice(nb, size=2 * 20, replace=False)
    pairs = np.stack([pick[:20], pick[20:]], axis=1).astype(np.int64)
    ek, ev = [bits(x) for x in ks], [bits(x) for x in vs]
    OC.block_copy(ek, ev, pairs)
    rec = B.new_error_record()
    B.block_copy(ks, vs, torch.from_numpy(pairs).cuda(), error_record=rec)
    assert B.pa_error_read(rec) == [0, 0, 0, 0]
    for l in range(layers):
        assert np.array_equal(bits(ks[l]), ek[l]) and np.array_equal(bits(vs[l]), ev[l])


def test_block_copy_bad_pair_is_recorded_and_skipped(B):
    kc, vc = _pool(20, 8, 4, 16, 64, torch.float16)
    pairs = torch.tensor([[1, 2], [3, 99], [4, 5]], dtype=torch.int64, device="cuda")
    ek, ev = bits(kc), bits(vc)
    rec = B.new_error_record()
    B.block_copy([kc], [vc], pairs, error_record=rec)
    assert B.pa_error_read(rec) == [4, 1, 1, 99]
    OC.block_copy([ek], [ev], [[1, 2], [4, 5]])
    assert np.array_equal(bits(kc), ek) and np.array_equal(bits(vc), ev)


def test_block_copy_padding_pairs_are_skipped_silently(B):
    kc, vc = _pool(21, 8, 4, 16, 64, torch.bfloat16)
    pairs = np.array([[-1, -1], [1, 2], [-1, -1], [4, 5], [-1, -1]], dtype=np.int64)
    ek, ev = bits(kc), bits(vc)
    rec = B.new_error_record()
    B.block_copy([kc], [vc], torch.from_numpy(pairs).cuda(), error_record=rec)
    assert B.pa_error_read(rec) == [0, 0, 0, 0]
    OC.block_copy([ek], [ev], pairs)
    assert np.array_equal(bits(kc), ek) and np.array_equal(bits(vc), ev)
