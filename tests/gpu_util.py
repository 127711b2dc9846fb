"""Helpers for the GPU parity tests: hand generator tensors to the oracle and
compare the library's outputs with the oracle's within the stated bounds.

Tolerance: attention outputs in fp32 must be within 2e-3 (max abs) of the fp64
oracle.  Half-precision outputs carry their own rounding on top, so for them the
bound is 2e-3 plus half an ulp of the output type at the oracle's value.
Append, copy and every index operation must be bit-exact.
"""

from __future__ import annotations

import numpy as np
import torch

from oracle import attention as OA
from oracle import cache_ops as OC

ATOL = 2e-3


def storage(t: torch.Tensor):
    """Host copy of stored values in the form the oracle takes, plus its dtype tag."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16).copy(), "bf16"
    if t.dtype == torch.float16:
        return t.numpy().copy(), "f16"
    raise TypeError(t.dtype)


def bits(t: torch.Tensor) -> np.ndarray:
    """Raw 16-bit patterns (for bit-exact comparison, NaN included)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy()


def half_ulp(x: np.ndarray, dtype: torch.dtype) -> np.ndarray:
    mant = {torch.float16: 10, torch.bfloat16: 7}[dtype]
    emin = {torch.float16: -14, torch.bfloat16: -126}[dtype]
    _, e = np.frexp(np.abs(x))
    e = np.maximum(e - 1, emin)
    return 0.5 * np.ldexp(1.0, e - mant)


def assert_matches_oracle(out: torch.Tensor, ref: np.ndarray, what: str = "") -> float:
    got = out.detach().double().cpu().numpy()
    assert got.shape == ref.shape, (got.shape, ref.shape)
    bound = ATOL if out.dtype == torch.float32 else ATOL + half_ulp(ref, out.dtype)
    err = np.abs(got - ref)
    bad = ~(err <= bound)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {bad.sum()} elements off; max err {np.nanmax(err)}; "
                             f"first {idx.tolist()} got {got[tuple(idx[0])]} ref {ref[tuple(idx[0])]}")
    return float(err.max()) if err.size else 0.0


def compact_pool(k_cache, v_cache, tables, lens, block_size, seqs):
    """Host copies of just the blocks the listed sequences use, with their tables
    relabelled to the compact pool (physical placement does not change attention)."""
    used = []
    rows = []
    for i in seqs:
        nb = -(-int(lens[i]) // block_size)
        used.extend(int(b) for b in tables[i][:nb])
    uniq = sorted(set(used))
    remap = {b: j for j, b in enumerate(uniq)}
    idx = torch.tensor(uniq if uniq else [0], dtype=torch.long, device=k_cache.device)
    kc, dt = storage(k_cache.index_select(0, idx))
    vc, _ = storage(v_cache.index_select(0, idx))
    for i in seqs:
        nb = -(-int(lens[i]) // block_size)
        row = [remap[int(b)] for b in tables[i][:nb]]
        rows.append(row + [-1] * (tables.shape[1] - nb))
    return kc, vc, np.array(rows, dtype=np.int64).reshape(len(seqs), -1), dt, remap


def oracle_decode(batch, seqs=None) -> np.ndarray:
    """fp64 expected output of append-then-decode for a workloads.DecodeBatch,
    computed from the generator's tensors only."""
    seqs = list(range(batch.num_seqs)) if seqs is None else list(seqs)
    lens = batch.context_lens
    kc, vc, tables, dt, remap = compact_pool(batch.k_cache, batch.v_cache, batch.block_tables,
                                             lens, batch.block_size, seqs)
    q, _ = storage(batch.q[torch.tensor(seqs, device=batch.q.device)])
    if batch.has_append:
        bs = batch.block_size
        sel = torch.tensor(seqs, device=batch.new_k.device)
        nk, _ = storage(batch.new_k[sel])
        nv, _ = storage(batch.new_v[sel])
        slots = []
        for i in seqs:
            s = int(batch.slot_mapping[i])
            slots.append(remap[s // bs] * bs + s % bs)
        OC.kv_append(kc, vc, nk, nv, np.array(slots), bs)
    return OA.paged_decode_attention(q, kc, vc, tables, lens[seqs], batch.scale,
                                     batch.block_size, dt)


def device_tables(batch, device="cuda"):
    bt = torch.from_numpy(np.ascontiguousarray(batch.block_tables)).to(device)
    sl = torch.from_numpy(np.ascontiguousarray(batch.context_lens.astype(np.int32))).to(device)
    return bt, sl
