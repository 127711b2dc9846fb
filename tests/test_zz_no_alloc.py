"""The allocation-free decode entry point, checked against the regular one and
against the oracle.

paged_attn_decode_noalloc serves callers that cannot allocate device memory
(code inside another runtime's memory pool, loops that must never block in the
allocator, fixed memory budgets): it takes its split-K scratch from an array
compiled into the library instead of a caller-provided workspace.  This file is
collected last so that a failure here stops a ``-x`` run only after every other
test has run; it also passes when run on its own in a fresh process.
"""

import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

from gpu_util import ATOL, assert_matches_oracle, oracle_decode
from workloads import decode_13b, random_decode_batch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "paged_kv_cache_317_gb300")


def _args(b, bt, sl, out, pt=0):
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    dtype = {torch.float16: 0, torch.bfloat16: 1}[b.q.dtype]
    return (p(b.q), p(b.k_cache), p(b.v_cache), p(bt), p(sl), b.num_seqs, b.num_heads,
            b.head_dim, b.block_size, bt.shape[1], b.num_blocks, b.scale, dtype, p(out), 2, pt)


def _noalloc(lib, b, bt, sl, pt):
    from paged_kv_cache_317_gb300 import binding as B
    out = torch.full((b.num_seqs, b.num_heads, b.head_dim), float("nan"), device="cuda")
    rec = B.new_error_record()
    st = lib.paged_attn_decode_noalloc(*_args(b, bt, sl, out, pt), ctypes.c_void_p(rec.data_ptr()),
                                       ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, B.STATUS[st]
    torch.cuda.synchronize()
    assert B.pa_error_read(rec) == [0, 0, 0, 0]
    return out


def test_noalloc_matches_the_regular_entry_point_and_the_oracle_on_two_calls(lib):
    from paged_kv_cache_317_gb300 import binding as B
    b = decode_13b(device="cuda", num_seqs=64, seed=31)
    ref = oracle_decode(b)                               # append-then-decode, from the generator
    bt = torch.from_numpy(b.block_tables).cuda()
    sl = torch.from_numpy(b.context_lens).cuda()
    B.kv_cache_append(b.new_k, b.new_v, torch.from_numpy(b.slot_mapping).cuda(), b.k_cache,
                      b.v_cache)
    regular = B.paged_attn_decode(b.q, b.k_cache, b.v_cache, bt, sl, b.scale)
    need = lib.paged_attn_workspace_size(b.num_seqs, b.num_heads, b.head_dim, b.block_size,
                                         bt.shape[1], 0)
    assert 0 < need <= B.NOALLOC_SCRATCH_BYTES          # split-K: the scratch is really used
    for _ in range(2):
        out = _noalloc(lib, b, bt, sl, 0)
        assert (out - regular).abs().max().item() <= ATOL
        assert_matches_oracle(out, ref, "noalloc, 64 sequences")


def test_noalloc_smaller_call_after_a_larger_one(lib):
    """A call with fewer, shorter sequences and 256-token partitions right after
    a larger call: the array still holds the larger call's partials, and none of
    them may leak into this call's output."""
    from paged_kv_cache_317_gb300 import binding as B
    big = decode_13b(device="cuda", num_seqs=96, seed=33, poison=False)
    bt = torch.from_numpy(big.block_tables).cuda()
    sl = torch.from_numpy(big.context_lens).cuda()
    _noalloc(lib, big, bt, sl, 0)
    lens = [1, 15, 255, 256, 257, 600, 1023]
    small = random_decode_batch(34, lens, 8, 128, 16, dtype="bf16", device="cuda")
    sbt = torch.from_numpy(small.block_tables).cuda()
    ssl = torch.from_numpy(small.context_lens).cuda()
    assert lib.paged_attn_workspace_size(small.num_seqs, small.num_heads, small.head_dim,
                                         small.block_size, sbt.shape[1], 256) > 0
    out = _noalloc(lib, small, sbt, ssl, 256)
    regular = B.paged_attn_decode(small.q, small.k_cache, small.v_cache, sbt, ssl, small.scale,
                                  partition_tokens=256, out_dtype=torch.float32)
    assert torch.equal(out, regular)                    # same kernels, same partitions
    assert_matches_oracle(out, oracle_decode(small), "noalloc after a larger call")


def test_noalloc_before_and_after_a_device_reset(lib, tmp_path):
    """In a process of its own (a reset ends every context of the process):
    the C program decodes through paged_attn_decode_noalloc and through
    paged_attn_decode, resets the device and does it again."""
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    exe = str(tmp_path / "noalloc_after_reset")
    cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17",
           "-I", os.path.join(ROOT, "include"),
           os.path.join(ROOT, "tests", "noalloc_after_reset.cu"), "-L", PKG, "-lpagedkv",
           "-Xlinker", "-rpath," + PKG, "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "ok:" in r.stdout


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
