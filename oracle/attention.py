"""fp64 reference for single-query decode attention through a block table.

TEST INFRASTRUCTURE ONLY (see the package docstring).

What it computes (PagedAttention, zeroshotmind.com page, section "Block tables:
logical order, physical scatter"): each sequence's keys and values are the rows
found by walking its logical blocks 0, 1, 2, ... in order, following each
through the block table to a physical block, and keeping the first ``seq_len``
rows.  The attention over that contiguous logical sequence is the textbook one:

    s_t = scale * <q, k_t>,   w = softmax(s),   out = sum_t w_t v_t

Stored half-precision values are upcast exactly to float64 before any
arithmetic, so the only error left in a comparison is the GPU's.
"""

from __future__ import annotations

import numpy as np


def to_float64(x, dtype: str) -> np.ndarray:
    """Exact upcast of stored values.

    ``f16``: an array of numpy float16.  ``bf16``: an array of uint16 bit
    patterns, each the upper 16 bits of an IEEE-754 binary32 (so the value is
    the binary32 whose low 16 bits are zero).  ``f32``/``f64``: floats.
    """
    if dtype == "f16":
        return np.asarray(x, dtype=np.float16).astype(np.float64)
    if dtype == "bf16":
        bits = np.asarray(x, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
        return bits.view(np.float32).astype(np.float64)
    if dtype in ("f32", "f64"):
        return np.asarray(x, dtype=np.float64)
    raise ValueError(f"unknown dtype {dtype!r}")


def gather_sequence(cache: np.ndarray, table_row, seq_len: int, block_size: int) -> np.ndarray:
    """Reassemble one sequence from a paged pool.

    ``cache`` is ``[num_blocks, H, block_size, D]``.  Logical block ``j`` of the
    sequence sits in physical block ``table_row[j]``; token ``t`` is row
    ``t % block_size`` of logical block ``t // block_size``.  Returns
    ``[seq_len, H, D]`` in the cache's own storage type.
    """
    n_blocks = -(-int(seq_len) // block_size)
    if n_blocks == 0:
        return np.zeros((0, cache.shape[1], cache.shape[3]), dtype=cache.dtype)
    logical = [cache[int(table_row[j])] for j in range(n_blocks)]    # each [H, bs, D]
    stacked = np.concatenate(logical, axis=1)                         # [H, n_blocks*bs, D]
    return np.ascontiguousarray(stacked[:, :seq_len, :].transpose(1, 0, 2))


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float) -> np.ndarray:
    """softmax(scale * q k^T) v for every head, in float64.

    q ``[H, D]``, k and v ``[L, H, D]``.  An empty sequence (L = 0) has no
    softmax; its output is defined as zeros.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    if k.shape[0] == 0:
        return np.zeros((q.shape[0], v.shape[2]), dtype=np.float64)
    s = np.einsum("hd,lhd->hl", q, k) * float(scale)
    s = s - s.max(axis=1, keepdims=True)
    w = np.exp(s)
    w = w / w.sum(axis=1, keepdims=True)
    return np.einsum("hl,lhd->hd", w, v)


def paged_decode_attention(q, k_cache, v_cache, block_tables, seq_lens, scale: float,
                           block_size: int, dtype: str, seqs=None) -> np.ndarray:
    """Decode attention for every sequence (or the listed ``seqs``), float64 ``[n, H, D]``.

    ``q`` is ``[N, H, D]`` and the caches ``[num_blocks, H, block_size, D]``, all in
    the storage representation that ``to_float64`` accepts for ``dtype``.
    """
    idx = range(len(seq_lens)) if seqs is None else seqs
    out = []
    for i in idx:
        L = int(seq_lens[i])
        k = to_float64(gather_sequence(k_cache, block_tables[i], L, block_size), dtype)
        v = to_float64(gather_sequence(v_cache, block_tables[i], L, block_size), dtype)
        out.append(attention(to_float64(q[i], dtype), k, v, scale))
    return np.stack(out) if out else np.zeros((0,) + tuple(np.shape(q)[1:]), dtype=np.float64)


def partition_partials(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float,
                       partition_tokens: int):
    """Split a sequence into consecutive partitions of ``partition_tokens`` tokens
    (the last may be shorter) and return, per partition p,

        m_p   = max_t s_t
        l_p   = sum_t exp(s_t - m_p)
        acc_p = sum_t exp(s_t - m_p) v_t

    over the tokens t of p, with ``s_t = scale * <q, k_t>``.  Shapes: m, l
    ``[P, H]``, acc ``[P, H, D]``, float64.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    L = k.shape[0]
    ms, ls, accs = [], [], []
    for start in range(0, L, partition_tokens):
        kp, vp = k[start:start + partition_tokens], v[start:start + partition_tokens]
        s = np.einsum("hd,lhd->hl", q, kp) * float(scale)
        m = s.max(axis=1)
        e = np.exp(s - m[:, None])
        ms.append(m)
        ls.append(e.sum(axis=1))
        accs.append(np.einsum("hl,lhd->hd", e, vp))
    return np.array(ms), np.array(ls), np.array(accs)


def merge_partials(m: np.ndarray, l: np.ndarray, acc: np.ndarray) -> np.ndarray:
    """Combine per-partition partials into the full softmax-weighted mean:

        M = max_p m_p,   out = sum_p exp(m_p - M) acc_p / sum_p exp(m_p - M) l_p
    """
    M = m.max(axis=0)
    w = np.exp(m - M[None, :])
    return (w[:, :, None] * acc).sum(axis=0) / (w * l).sum(axis=0)[:, None]


def paged_prefill_attention(q, k_cache, v_cache, block_tables, seq_lens, query_start,
                            scale: float, block_size: int, dtype: str, seqs=None):
    """Several query tokens per sequence, each attending causally through the block table.

    Sequence i holds ``seq_lens[i]`` tokens; its last ``Q_i = query_start[i+1] -
    query_start[i]`` are the queries, stored at rows ``query_start[i] .. query_start[i+1]``
    of ``q`` (``[total, H, D]``).  Query j of sequence i sits at position
    ``p = seq_lens[i] - Q_i + j`` and attends over tokens ``0 .. p`` (itself included),
    exactly as a single-query decode of the sequence's first ``p + 1`` tokens would.
    Returns float64 ``[total, H, D]`` (or only the rows of ``seqs``, in order).
    """
    idx = range(len(seq_lens)) if seqs is None else seqs
    rows = []
    for i in idx:
        L = int(seq_lens[i])
        a, b = int(query_start[i]), int(query_start[i + 1])
        n_q = b - a
        k = to_float64(gather_sequence(k_cache, block_tables[i], L, block_size), dtype)
        v = to_float64(gather_sequence(v_cache, block_tables[i], L, block_size), dtype)
        for j in range(n_q):
            p = L - n_q + j
            rows.append(attention(to_float64(q[a + j], dtype), k[: p + 1], v[: p + 1], scale))
    if not rows:
        return np.zeros((0,) + tuple(np.shape(q)[1:]), dtype=np.float64)
    return np.stack(rows)
