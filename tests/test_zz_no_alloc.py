"""The allocation-free decode entry point, checked against the regular one.

paged_attn_decode_noalloc serves callers that cannot allocate device memory
(code inside another runtime's memory pool, loops that must never block in the
allocator, fixed memory budgets): it takes its split-K scratch from an array
compiled into the library instead of a caller-provided workspace.  This file is
collected last so that a failure here stops a ``-x`` run only after every other
test has run; it also passes when run on its own in a fresh process.
"""

import ctypes

import pytest
import torch

from gpu_util import ATOL
from workloads import decode_13b

pytestmark = pytest.mark.gpu


def _args(b, bt, sl, out, pt=0):
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    return (p(b.q), p(b.k_cache), p(b.v_cache), p(bt), p(sl), b.num_seqs, b.num_heads,
            b.head_dim, b.block_size, bt.shape[1], b.num_blocks, b.scale, 1, p(out), 2, pt)


def test_noalloc_matches_the_regular_entry_point_on_two_calls(lib):
    from paged_kv_cache_317_gb300 import binding as B
    b = decode_13b(device="cuda", num_seqs=64, seed=31)
    bt = torch.from_numpy(b.block_tables).cuda()
    sl = torch.from_numpy(b.context_lens).cuda()
    B.kv_cache_append(b.new_k, b.new_v, torch.from_numpy(b.slot_mapping).cuda(), b.k_cache,
                      b.v_cache)
    ref = B.paged_attn_decode(b.q, b.k_cache, b.v_cache, bt, sl, b.scale)
    need = lib.paged_attn_workspace_size(b.num_seqs, b.num_heads, b.head_dim, b.block_size,
                                         bt.shape[1], 0)
    assert 0 < need <= B.NOALLOC_SCRATCH_BYTES          # split-K: the scratch is really used
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):
        out = torch.full_like(ref, float("nan"))
        rec = B.new_error_record()
        st = lib.paged_attn_decode_noalloc(*_args(b, bt, sl, out), ctypes.c_void_p(rec.data_ptr()),
                                           stream)
        assert st == 0
        torch.cuda.synchronize()
        assert B.pa_error_read(rec) == [0, 0, 0, 0]
        assert (out - ref).abs().max().item() <= ATOL


def test_noalloc_rejects_sizes_beyond_its_scratch(lib):
    from paged_kv_cache_317_gb300 import binding as B
    b = decode_13b(device="cuda", num_seqs=4, seed=32)
    big_mb = 1 << 14                                     # 262144-token capacity per sequence
    bt = torch.zeros((b.num_seqs, big_mb), dtype=torch.int32, device="cuda")
    sl = torch.from_numpy(b.context_lens).cuda()
    out = torch.zeros((b.num_seqs, b.num_heads, b.head_dim), device="cuda")
    assert lib.paged_attn_workspace_size(b.num_seqs, b.num_heads, b.head_dim, b.block_size,
                                         big_mb, 0) > B.NOALLOC_SCRATCH_BYTES
    st = lib.paged_attn_decode_noalloc(*_args(b, bt, sl, out), None,
                                       ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert B.STATUS[st] == "PA_ERR_INVALID_ARG"
