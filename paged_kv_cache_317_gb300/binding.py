"""Thin ctypes binding over libpagedkv.so, with the C ABI's names.

Argument marshalling only: tensors are passed by ``data_ptr()``, sizes are read
off their shapes, and the stream is the caller's current CUDA stream.  Every
step of the path runs in the library's kernels; there is no fallback.  If the
library is missing, loading it raises.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

from . import _build

c_int, c_int32, c_int64, c_float, c_size_t, c_void_p = (
    ctypes.c_int, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t, ctypes.c_void_p)
P_int32 = ctypes.POINTER(ctypes.c_int32)
P_int64 = ctypes.POINTER(ctypes.c_int64)

PA_F16, PA_BF16, PA_F32 = 0, 1, 2
_DTYPE = {torch.float16: PA_F16, torch.bfloat16: PA_BF16, torch.float32: PA_F32}

STATUS = {
    0: "PA_OK", 1: "PA_ERR_INVALID_ARG", 2: "PA_ERR_UNSUPPORTED", 3: "PA_ERR_CUDA",
    4: "PA_ERR_BAD_BLOCK", 5: "PA_ERR_BAD_SLOT", 6: "PA_ERR_BAD_SEQ_LEN", 7: "PA_ERR_TIMEOUT",
    8: "PA_ERR_OOM", 9: "PA_ERR_NO_SEQ", 10: "PA_ERR_SEQ_EXISTS", 11: "PA_ERR_REFCOUNT",
}
STATUS_CODE = {v: k for k, v in STATUS.items()}


class pa_prefill_opts(ctypes.Structure):
    _fields_ = [("seq_order", c_void_p)]


class pa_decode_opts(ctypes.Structure):
    _fields_ = [("heads_per_cta", c_int), ("stages", c_int), ("phases", c_int),
                ("seq_order", c_void_p), ("work_items", c_void_p), ("num_work_items", c_int),
                ("shared_records", c_void_p), ("num_shared", c_int), ("early_inputs", c_int),
                ("tail_start", c_void_p), ("counts", c_void_p)]


ABI_VERSION = 3             # PAGEDKV_VERSION of include/pagedkv.h
PA_SHARE_MAX_MEMBERS = 8
PA_SHARE_RECORD_WORDS = 2 + PA_SHARE_MAX_MEMBERS


def _decode_opts(heads_per_cta, stages, phases, seq_order, work_items, shared_records=None,
                 early_inputs=False, tail_start=None, counts=None):
    if seq_order is not None:
        _need(seq_order, "seq_order", torch.int32)
    if work_items is not None:
        _need(work_items, "work_items", torch.int32)
    if tail_start is not None:
        _need(tail_start, "tail_start", torch.int32)
    if counts is not None:
        _need(counts, "counts", torch.int32)
        if counts.numel() < 2:
            raise ValueError("counts must hold two entries (work items, records)")
    if shared_records is not None:
        _need(shared_records, "shared_records", torch.int32)
        if shared_records.dim() != 2 or shared_records.shape[1] != PA_SHARE_RECORD_WORDS:
            raise ValueError(f"shared_records must be [n, {PA_SHARE_RECORD_WORDS}]")
    items_ptr = None if work_items is None else work_items.data_ptr()
    if work_items is not None and not items_ptr and shared_records is not None:
        items_ptr = shared_records.data_ptr() or None   # an empty list still counts as given
    return pa_decode_opts(heads_per_cta, stages, phases,
                          None if seq_order is None else seq_order.data_ptr(),
                          items_ptr,
                          0 if work_items is None else int(work_items.numel()),
                          None if shared_records is None else shared_records.data_ptr(),
                          0 if shared_records is None else int(shared_records.shape[0]),
                          int(bool(early_inputs)),
                          None if tail_start is None else tail_start.data_ptr(),
                          None if counts is None else counts.data_ptr())


def _host_int32(values, name: str) -> "np.ndarray":
    import numpy as np
    if isinstance(values, np.ndarray) and values.dtype == np.int32 and values.ndim == 1 \
            and values.flags.c_contiguous:
        return values
    a = np.asarray(values, dtype=np.int64).reshape(-1)
    if a.size and (a.min() < -2**31 or a.max() >= 2**31):
        raise ValueError(f"{name}: values do not fit int32")
    return np.ascontiguousarray(a, dtype=np.int32)


def decode_partition_tokens(seq_lens, num_heads: int, heads_per_cta: int = 0,
                            num_sms: int = 0) -> int:
    """Split-K partition length for a decode over these (host) lengths, chosen by
    pa_decode_partition_tokens: 512 for batches with plenty of work per SM, down
    to 32 for a few short sequences.  num_sms 0 asks the current device."""
    lens = _host_int32(seq_lens, "seq_lens")
    out = ctypes.c_int32()
    _check(load_library().pa_decode_partition_tokens(
        lens.ctypes.data, len(lens), num_heads, heads_per_cta, num_sms,
        ctypes.byref(out)), "pa_decode_partition_tokens")
    return out.value


def partition_work_items(seq_lens, partition_tokens: int, max_blocks_per_seq: int,
                         block_size: int, order=None) -> "np.ndarray":
    """The (sequence, partition) work list of a decode launch, item = i * P + p,
    sequences in the given order (default: longest first); built by
    pa_decode_work_items."""
    import numpy as np
    lens = _host_int32(seq_lens, "seq_lens")
    ordp = None
    if order is not None:
        ordarr = _host_int32(order, "order")
        if ordarr.shape != lens.shape:
            raise ValueError("order must hold one entry per sequence")
        ordp = ordarr.ctypes.data
    lib, n = load_library(), ctypes.c_int32()
    args = (lens.ctypes.data, len(lens), partition_tokens, max_blocks_per_seq,
            block_size, ordp)
    _check(lib.pa_decode_work_items(*args, None, 0, ctypes.byref(n)), "pa_decode_work_items")
    items = np.empty(n.value, dtype=np.int32)
    _check(lib.pa_decode_work_items(*args, items.ctypes.data, n.value,
                                    ctypes.byref(n)), "pa_decode_work_items")
    return items


def share_plan(block_tables, seq_lens, partition_tokens: int, block_size: int,
               fused_append: bool = True, order=None, out=None):
    """Work list and shared-partition records (pa_decode_share_plan) for a decode
    over host tables [N, max_blocks] and lengths: (work_items int32 [n],
    shared_records int32 [r, PA_SHARE_RECORD_WORDS]).  out: optional int32
    buffers (items [cap], records [cap, PA_SHARE_RECORD_WORDS]) to fill in place
    (a pinned staging buffer, say); the results are then views of them."""
    return _share_plan(block_tables, seq_lens, partition_tokens, block_size, fused_append,
                       order, False, None if out is None else (*out[:2], None))[:2]


def share_plan_prefix(block_tables, seq_lens, partition_tokens: int, block_size: int,
                      fused_append: bool = True, order=None, out=None):
    """The same plan with prefix records (pa_decode_share_plan_ex): partitions a
    group shares only in part are read once up to where the members diverge.
    Returns (work_items, shared_records, tail_start int32 [N]); pass tail_start to
    the decode with the other two.  out: optional (items, records, tail_start)
    buffers to fill in place."""
    return _share_plan(block_tables, seq_lens, partition_tokens, block_size, fused_append,
                       order, True, out)


def _out_buffer(buf, name, shape_tail=()):
    import numpy as np
    if (not isinstance(buf, np.ndarray) or buf.dtype != np.int32 or
            not buf.flags.c_contiguous or buf.shape[1:] != tuple(shape_tail)):
        raise ValueError(f"{name} must be a C-contiguous int32 array of shape [n, *{shape_tail}]")
    return buf


def _share_plan(block_tables, seq_lens, partition_tokens, block_size, fused_append, order,
                prefixes, out=None):
    import numpy as np
    tables = np.ascontiguousarray(block_tables, dtype=np.int32)
    if tables.ndim != 2:
        raise ValueError("block_tables must be [num_seqs, max_blocks]")
    lens = _host_int32(seq_lens, "seq_lens")
    if len(lens) != tables.shape[0]:
        raise ValueError("one length per table row")
    ordp = None
    if order is not None:
        ordarr = _host_int32(order, "order")
        if ordarr.shape != lens.shape:
            raise ValueError("order must hold one entry per sequence")
        ordp = ordarr.ctypes.data
    lib, ni, nr = load_library(), ctypes.c_int32(), ctypes.c_int32()
    args = (tables.ctypes.data, lens.ctypes.data, len(lens),
            tables.shape[1], block_size, partition_tokens, int(bool(fused_append)), ordp)
    # one call with room for every (sequence, partition) pair; records hold >= 2 each
    pt = partition_tokens or 512
    pairs = len(lens) * max(1, -(-tables.shape[1] * block_size // pt)) if pt > 0 else 0
    if out is None:
        items = np.empty(pairs, dtype=np.int32)
        recs = np.empty((pairs // 2, PA_SHARE_RECORD_WORDS), dtype=np.int32)
        tails = np.empty(len(lens), dtype=np.int32)
    else:
        if len(out) not in (2, 3):
            raise ValueError("out must be (items, records) or (items, records, tail_start)")
        items = _out_buffer(out[0], "items")
        recs = _out_buffer(out[1], "records", (PA_SHARE_RECORD_WORDS,))
        tails = out[2] if len(out) == 3 else None
        if tails is None:
            tails = np.empty(len(lens), dtype=np.int32)
        elif _out_buffer(tails, "tail_start").shape[0] != len(lens):
            raise ValueError("tail_start must hold one entry per sequence")
    _check(lib.pa_decode_share_plan_ex(*args, int(bool(prefixes)), items.ctypes.data,
                                       len(items), ctypes.byref(ni), recs.ctypes.data,
                                       len(recs), ctypes.byref(nr), tails.ctypes.data),
           "pa_decode_share_plan_ex")
    return items[: ni.value], recs[: nr.value], tails


# name -> (restype, argtypes); mirrors include/pagedkv.h
SIGNATURES = {
    "pa_version": (c_int, []),
    "pa_status_string": (ctypes.c_char_p, [c_int]),
    "pa_error_clear": (c_int, [c_void_p, c_void_p]),
    "pa_error_read": (c_int, [c_void_p, P_int32, c_void_p]),
    "pa_selftest_bounded_wait": (c_int, [c_void_p, c_int, ctypes.c_ulonglong, c_void_p]),
    "paged_attn_workspace_size": (c_size_t, [c_int] * 6),
    "paged_attn_workspace_size_tails": (c_size_t, [c_int] * 6),
    "paged_attn_decode": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int,
                                  c_int, c_int, c_int, c_int, c_float, c_int, c_void_p, c_int,
                                  c_int, c_void_p, c_size_t, c_void_p, c_void_p]),
    "paged_attn_decode_ex": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int,
                                     c_int, c_int, c_int, c_int, c_int, c_float, c_int, c_void_p,
                                     c_int, c_int, c_void_p, c_size_t, c_void_p, c_void_p,
                                     ctypes.POINTER(pa_decode_opts)]),
    "paged_attn_decode_append": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                         c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int,
                                         c_int, c_float, c_int, c_void_p, c_int, c_int, c_void_p,
                                         c_size_t, c_void_p, c_void_p,
                                         ctypes.POINTER(pa_decode_opts)]),
    "paged_attn_prefill": (c_int, [c_void_p, c_void_p, c_int, c_int, c_void_p, c_void_p,
                                   c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int, c_int,
                                   c_float, c_int, c_void_p, c_int, c_void_p, c_void_p]),
    "paged_attn_prefill_ex": (c_int, [c_void_p, c_void_p, c_int, c_int, c_void_p, c_void_p,
                                   c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int, c_int,
                                   c_float, c_int, c_void_p, c_int, c_void_p, c_void_p, c_void_p]),
    "paged_attn_decode_noalloc": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                          c_int, c_int, c_int, c_int, c_int, c_int, c_float,
                                          c_int, c_void_p, c_int, c_int, c_void_p, c_void_p]),
    "kv_cache_append": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_void_p, c_void_p, c_int,
                                c_int, c_int, c_int, c_int, c_void_p, c_void_p]),
    "block_copy": (c_int, [ctypes.POINTER(c_void_p), ctypes.POINTER(c_void_p), c_int, c_void_p,
                           c_int, c_int, c_int, c_int, c_int, c_int, c_void_p, c_void_p]),
    "pa_decode_partition_tokens": (c_int, [c_void_p, c_int, c_int, c_int, c_int, P_int32]),
    "pa_decode_work_items": (c_int, [c_void_p, c_int, c_int, c_int, c_int, c_void_p, c_void_p,
                                     c_int32, P_int32]),
    "pa_decode_share_plan": (c_int, [c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int,
                                     c_void_p, c_void_p, c_int32, P_int32, c_void_p, c_int32,
                                     P_int32]),
    "pa_decode_share_plan_ex": (c_int, [c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int,
                                        c_void_p, c_int, c_void_p, c_int32, P_int32, c_void_p,
                                        c_int32, P_int32, c_void_p]),
    "pa_alloc_create": (c_void_p, [c_int32, c_int32, P_int32]),
    "pa_alloc_destroy": (None, [c_void_p]),
    "pa_seq_add": (c_int, [c_void_p, c_int64, c_int32]),
    "pa_seq_fork": (c_int, [c_void_p, c_int64, c_int64]),
    "pa_seq_append": (c_int, [c_void_p, c_int64, P_int64, P_int32, P_int32]),
    "pa_seq_free": (c_int, [c_void_p, c_int64]),
    "pa_seq_len": (c_int, [c_void_p, c_int64, P_int32]),
    "pa_seq_block_table": (c_int, [c_void_p, c_int64, P_int32, c_int32, P_int32]),
    "pa_seq_slots": (c_int, [c_void_p, c_int64, c_int32, c_int32, c_void_p]),
    "pa_block_refcount": (c_int, [c_void_p, c_int32, P_int32]),
    "pa_num_free_blocks": (c_int32, [c_void_p]),
    "pa_num_seqs": (c_int32, [c_void_p]),
    "pa_batch_append": (c_int, [c_void_p, c_void_p, c_int32, c_void_p, c_void_p, P_int32]),
    "pa_batch_fork": (c_int, [c_void_p, c_void_p, c_void_p, c_int32]),
    "pa_batch_free": (c_int, [c_void_p, c_void_p, c_int32]),
    "pa_batch_block_tables": (c_int, [c_void_p, c_void_p, c_int32, c_int32, c_void_p, c_void_p]),
    "pa_alloc_stats": (c_int, [c_void_p, P_int32, P_int64, P_int64, P_int64]),
    "pa_alloc_check": (c_int, [c_void_p]),
}

_LIB: Optional[ctypes.CDLL] = None


class PagedKVError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        self.name = STATUS.get(status, str(status))
        super().__init__(f"{where}: {self.name} ({_status_text(status)})")


def _status_text(status: int) -> str:
    try:
        return load_library().pa_status_string(status).decode()
    except Exception:  # pragma: no cover - library not loadable
        return "?"


def load_library() -> ctypes.CDLL:
    """Load libpagedkv.so from the package directory; raise if it was not built."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(_build.LIB_PATH):
            raise RuntimeError(f"{_build.LIB_PATH} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(_build.LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        if lib.pa_version() != ABI_VERSION:   # the option structs below match this version
            raise RuntimeError(f"{_build.LIB_PATH} is version {lib.pa_version()}, the "
                               f"binding expects {ABI_VERSION}: rebuild it")
        _LIB = lib
    return _LIB


def _check(status: int, where: str) -> None:
    if status != 0:
        raise PagedKVError(status, where)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else c_void_p(t.data_ptr())


def _stream(stream: Optional[torch.cuda.Stream]):
    s = stream if stream is not None else torch.cuda.current_stream()
    return c_void_p(s.cuda_stream)


def _need(t: torch.Tensor, name: str, dtype=None):
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


# --------------------------------------------------------------- error record
def new_error_record(device="cuda") -> torch.Tensor:
    return torch.zeros(4, dtype=torch.int32, device=device)


def pa_error_clear(record: torch.Tensor, stream=None) -> None:
    _check(load_library().pa_error_clear(_ptr(record), _stream(stream)), "pa_error_clear")


def pa_error_read(record: torch.Tensor, stream=None):
    out = (ctypes.c_int32 * 4)()
    _check(load_library().pa_error_read(_ptr(record), out, _stream(stream)), "pa_error_read")
    return list(out)


def pa_selftest_bounded_wait(record: torch.Tensor, arrive: bool, limit_ns: int,
                             stream=None) -> None:
    _check(load_library().pa_selftest_bounded_wait(_ptr(record), int(arrive), int(limit_ns),
                                                   _stream(stream)), "pa_selftest_bounded_wait")


# ----------------------------------------------------------------- decode
def paged_attn_workspace_size(num_seqs, num_heads, head_dim, block_size, max_blocks_per_seq,
                              partition_tokens=0, tails: bool = False) -> int:
    """Workspace bytes of a decode; tails=True: with tail_start (prefix records)."""
    fn = (load_library().paged_attn_workspace_size_tails if tails
          else load_library().paged_attn_workspace_size)
    return int(fn(num_seqs, num_heads, head_dim, block_size, max_blocks_per_seq,
                  partition_tokens))


def paged_attn_decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                      block_tables: torch.Tensor, seq_lens: torch.Tensor, scale: float,
                      out: Optional[torch.Tensor] = None, out_dtype=torch.float32,
                      partition_tokens: int = 0, workspace: Optional[torch.Tensor] = None,
                      error_record: Optional[torch.Tensor] = None, heads_per_cta: int = 0,
                      stages: int = 0, phases: int = 0, seq_order: Optional[torch.Tensor] = None,
                      work_items: Optional[torch.Tensor] = None,
                      shared_records: Optional[torch.Tensor] = None,
                      early_inputs: bool = False, tail_start: Optional[torch.Tensor] = None,
                      counts: Optional[torch.Tensor] = None,
                      stream=None) -> torch.Tensor:
    """q [N,H,D]; caches [B,H,bs,D]; block_tables int32 [N,MB]; seq_lens int32 [N];
    seq_order: optional int32 [N] scheduling permutation on the device; work_items:
    optional int32 list of (sequence * P + partition) on the device; shared_records:
    optional int32 [r, PA_SHARE_RECORD_WORDS] shared partitions on the device
    (share_plan builds both); early_inputs: the kernel before the call on the stream
    writes none of the read-only inputs (pa_decode_opts.early_inputs); tail_start:
    optional int32 [N] on the device, with prefix records (share_plan_prefix);
    counts: optional int32 [2] on the device, the numbers of work items and records
    to run out of the lists given (then capacities), for CUDA-graph replays with
    lists of varying length."""
    N, H, D = q.shape
    B, _, bs, _ = k_cache.shape
    MB = block_tables.shape[1]
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, n)
    _need(block_tables, "block_tables", torch.int32)
    _need(seq_lens, "seq_lens", torch.int32)
    if out is None:
        out = torch.empty((N, H, D), dtype=out_dtype, device=q.device)
    _need(out, "out")
    if workspace is None:   # (a given one is checked against the size by the call)
        need = paged_attn_workspace_size(N, H, D, bs, MB, partition_tokens,
                                         tails=tail_start is not None)
        if need:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    opts = _decode_opts(heads_per_cta, stages, phases, seq_order, work_items,
                        shared_records, early_inputs, tail_start, counts)
    st = load_library().paged_attn_decode_ex(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(seq_lens), N, H, D, bs,
        MB, B, float(scale), _DTYPE[q.dtype], _ptr(out), _DTYPE[out.dtype], partition_tokens,
        _ptr(workspace), ws_bytes, _ptr(error_record), _stream(stream), ctypes.byref(opts))
    _check(st, "paged_attn_decode")
    return out


def paged_attn_decode_append(q: torch.Tensor, new_k: torch.Tensor, new_v: torch.Tensor,
                             k_cache: torch.Tensor, v_cache: torch.Tensor,
                             block_tables: torch.Tensor, seq_lens: torch.Tensor, scale: float,
                             out: Optional[torch.Tensor] = None, out_dtype=torch.float32,
                             partition_tokens: int = 0, workspace: Optional[torch.Tensor] = None,
                             error_record: Optional[torch.Tensor] = None, heads_per_cta: int = 0,
                             stages: int = 0, phases: int = 0,
                             seq_order: Optional[torch.Tensor] = None,
                             work_items: Optional[torch.Tensor] = None,
                             shared_records: Optional[torch.Tensor] = None,
                             early_inputs: bool = False,
                             tail_start: Optional[torch.Tensor] = None,
                             counts: Optional[torch.Tensor] = None,
                             stream=None) -> torch.Tensor:
    """Append each sequence's last token (new_k/new_v [N,H,D]) into its slot and
    decode over all seq_lens[i] tokens, in one pass."""
    N, H, D = q.shape
    B, _, bs, _ = k_cache.shape
    MB = block_tables.shape[1]
    for t, n in ((q, "q"), (new_k, "new_k"), (new_v, "new_v"), (k_cache, "k_cache"),
                 (v_cache, "v_cache")):
        _need(t, n)
    _need(block_tables, "block_tables", torch.int32)
    _need(seq_lens, "seq_lens", torch.int32)
    if out is None:
        out = torch.empty((N, H, D), dtype=out_dtype, device=q.device)
    _need(out, "out")
    if workspace is None:   # (a given one is checked against the size by the call)
        need = paged_attn_workspace_size(N, H, D, bs, MB, partition_tokens,
                                         tails=tail_start is not None)
        if need:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    opts = _decode_opts(heads_per_cta, stages, phases, seq_order, work_items,
                        shared_records, early_inputs, tail_start, counts)
    st = load_library().paged_attn_decode_append(
        _ptr(q), _ptr(new_k), _ptr(new_v), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
        _ptr(seq_lens), N, H, D, bs, MB, B, float(scale), _DTYPE[q.dtype], _ptr(out),
        _DTYPE[out.dtype], partition_tokens, _ptr(workspace), ws_bytes, _ptr(error_record),
        _stream(stream), ctypes.byref(opts))
    _check(st, "paged_attn_decode_append")
    return out


def paged_attn_prefill(q: torch.Tensor, query_start: torch.Tensor, max_query_len: int,
                       k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
                       seq_lens: torch.Tensor, scale: float, out: Optional[torch.Tensor] = None,
                       out_dtype=torch.float32, error_record: Optional[torch.Tensor] = None,
                       seq_order: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Causal multi-query attention: q [total,H,D]; query_start int32 [N+1] (device);
    seq_order: optional int32 [N] dispatch order of the sequences on the device."""
    T, H, D = q.shape
    B, _, bs, _ = k_cache.shape
    N = seq_lens.shape[0]
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, n)
    for t, n in ((query_start, "query_start"), (block_tables, "block_tables"),
                 (seq_lens, "seq_lens")):
        _need(t, n, torch.int32)
    if out is None:
        out = torch.empty((T, H, D), dtype=out_dtype, device=q.device)
    _need(out, "out")
    if seq_order is not None:
        _need(seq_order, "seq_order", torch.int32)
    opts = pa_prefill_opts(None if seq_order is None else seq_order.data_ptr())
    st = load_library().paged_attn_prefill_ex(
        _ptr(q), _ptr(query_start), T, int(max_query_len), _ptr(k_cache), _ptr(v_cache),
        _ptr(block_tables), _ptr(seq_lens), N, H, D, bs, block_tables.shape[1], B, float(scale),
        _DTYPE[q.dtype], _ptr(out), _DTYPE[out.dtype], _ptr(error_record), _stream(stream),
        ctypes.byref(opts))
    _check(st, "paged_attn_prefill")
    return out


NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024


def paged_attn_decode_noalloc(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                              block_tables: torch.Tensor, seq_lens: torch.Tensor, scale: float,
                              out: torch.Tensor, partition_tokens: int = 0,
                              error_record: Optional[torch.Tensor] = None,
                              stream=None) -> torch.Tensor:
    """paged_attn_decode with its scratch taken from the library's fixed array:
    allocates nothing (``out`` must be given)."""
    N, H, D = q.shape
    B, _, bs, _ = k_cache.shape
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache"), (out, "out")):
        _need(t, n)
    _need(block_tables, "block_tables", torch.int32)
    _need(seq_lens, "seq_lens", torch.int32)
    st = load_library().paged_attn_decode_noalloc(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(seq_lens), N, H, D, bs,
        block_tables.shape[1], B, float(scale), _DTYPE[q.dtype], _ptr(out), _DTYPE[out.dtype],
        partition_tokens, _ptr(error_record), _stream(stream))
    _check(st, "paged_attn_decode_noalloc")
    return out


# ------------------------------------------------------------ cache upkeep
def kv_cache_append(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor,
                    k_cache: torch.Tensor, v_cache: torch.Tensor,
                    error_record: Optional[torch.Tensor] = None, stream=None) -> None:
    """k, v [T,H,D]; slot_mapping int64 [T]; caches [B,H,bs,D]."""
    T, H, D = k.shape
    B, _, bs, _ = k_cache.shape
    for t, n in ((k, "k"), (v, "v"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, n)
    _need(slot_mapping, "slot_mapping", torch.int64)
    st = load_library().kv_cache_append(_ptr(k), _ptr(v), _ptr(slot_mapping), T, _ptr(k_cache),
                                        _ptr(v_cache), H, D, bs, B, _DTYPE[k.dtype],
                                        _ptr(error_record), _stream(stream))
    _check(st, "kv_cache_append")


def block_copy(k_caches: Sequence[torch.Tensor], v_caches: Sequence[torch.Tensor],
               pairs: torch.Tensor, error_record: Optional[torch.Tensor] = None,
               stream=None) -> None:
    """Per-layer caches [B,H,bs,D]; pairs int64 [n,2] (src, dst) on the device."""
    n_layers = len(k_caches)
    B, H, bs, D = k_caches[0].shape
    for t in (*k_caches, *v_caches):
        _need(t, "cache")
    _need(pairs, "pairs", torch.int64)
    kp = (c_void_p * n_layers)(*[t.data_ptr() for t in k_caches])
    vp = (c_void_p * n_layers)(*[t.data_ptr() for t in v_caches])
    st = load_library().block_copy(kp, vp, n_layers, _ptr(pairs), int(pairs.shape[0]), H, D, bs,
                                   B, _DTYPE[k_caches[0].dtype], _ptr(error_record),
                                   _stream(stream))
    _check(st, "block_copy")


# --------------------------------------------------------------- allocator
class BlockAllocator:
    """Host block allocator (C++), see pa_alloc_* in include/pagedkv.h."""

    def __init__(self, num_blocks: int, block_size: int, free_order=None):
        self._lib = load_library()
        arr = None
        if free_order is not None:
            arr = (ctypes.c_int32 * num_blocks)(*[int(b) for b in free_order])
        self._h = self._lib.pa_alloc_create(num_blocks, block_size, arr)
        if not self._h:
            raise PagedKVError(1, "pa_alloc_create")
        self.num_blocks, self.block_size = num_blocks, block_size

    def close(self):
        if getattr(self, "_h", None):
            self._lib.pa_alloc_destroy(self._h)
            self._h = None

    __del__ = close

    def add(self, seq: int, num_tokens: int) -> None:
        _check(self._lib.pa_seq_add(self._h, seq, num_tokens), "pa_seq_add")

    def fork(self, parent: int, child: int) -> None:
        _check(self._lib.pa_seq_fork(self._h, parent, child), "pa_seq_fork")

    def append(self, seq: int):
        slot, src, dst = ctypes.c_int64(), ctypes.c_int32(), ctypes.c_int32()
        _check(self._lib.pa_seq_append(self._h, seq, ctypes.byref(slot), ctypes.byref(src),
                                       ctypes.byref(dst)), "pa_seq_append")
        return slot.value, (None if src.value < 0 else (src.value, dst.value))

    def free(self, seq: int) -> None:
        _check(self._lib.pa_seq_free(self._h, seq), "pa_seq_free")

    def length(self, seq: int) -> int:
        n = ctypes.c_int32()
        _check(self._lib.pa_seq_len(self._h, seq, ctypes.byref(n)), "pa_seq_len")
        return n.value

    def block_table(self, seq: int):
        n = ctypes.c_int32()
        _check(self._lib.pa_seq_block_table(self._h, seq, None, 0, ctypes.byref(n)), "table")
        buf = (ctypes.c_int32 * max(1, n.value))()
        _check(self._lib.pa_seq_block_table(self._h, seq, buf, n.value, ctypes.byref(n)), "table")
        return list(buf[: n.value])

    def slots(self, seq: int, start: int, count: int):
        import numpy as np
        out = np.empty(count, dtype=np.int64)
        _check(self._lib.pa_seq_slots(self._h, seq, start, count,
                                      out.ctypes.data), "pa_seq_slots")
        return out

    def refcount(self, block: int) -> int:
        n = ctypes.c_int32()
        _check(self._lib.pa_block_refcount(self._h, block, ctypes.byref(n)), "pa_block_refcount")
        return n.value

    def num_free(self) -> int:
        return int(self._lib.pa_num_free_blocks(self._h))

    def num_seqs(self) -> int:
        return int(self._lib.pa_num_seqs(self._h))

    def batch_append(self, seqs):
        import numpy as np
        ids = np.ascontiguousarray(seqs, dtype=np.int64)
        n = ids.shape[0]
        slots = np.empty(n, dtype=np.int64)
        pairs = np.empty((max(n, 1), 2), dtype=np.int64)
        nc = ctypes.c_int32()
        _check(self._lib.pa_batch_append(self._h, ids.ctypes.data, n,
                                         slots.ctypes.data,
                                         pairs.ctypes.data, ctypes.byref(nc)),
               "pa_batch_append")
        return slots, pairs[: nc.value].copy()

    def batch_fork(self, parents, children) -> None:
        """children[i] shares every block of parents[i]; all-or-nothing."""
        import numpy as np
        par = np.ascontiguousarray(parents, dtype=np.int64)
        chi = np.ascontiguousarray(children, dtype=np.int64)
        if par.shape != chi.shape:
            raise ValueError("parents and children differ in length")
        _check(self._lib.pa_batch_fork(self._h, par.ctypes.data,
                                       chi.ctypes.data, par.shape[0]),
               "pa_batch_fork")

    def batch_free(self, seqs) -> None:
        """End every listed sequence; all-or-nothing."""
        import numpy as np
        ids = np.ascontiguousarray(seqs, dtype=np.int64)
        _check(self._lib.pa_batch_free(self._h, ids.ctypes.data, ids.shape[0]),
               "pa_batch_free")

    def batch_block_tables(self, seqs, max_blocks: int, out=None):
        """Block tables [n, max_blocks] (-1 past each sequence's blocks) and lengths
        of the listed sequences; out: optional (tables, lengths) int32 arrays of
        those shapes to fill in place (a pinned staging buffer, say)."""
        import numpy as np
        ids = np.ascontiguousarray(seqs, dtype=np.int64)
        n = ids.shape[0]
        if out is None:
            tables = np.empty((n, max_blocks), dtype=np.int32)
            lens = np.empty(n, dtype=np.int32)
        else:
            tables = _out_buffer(out[0], "tables", (max_blocks,))
            lens = _out_buffer(out[1], "lengths")
            if tables.shape[0] != n or lens.shape[0] != n:
                raise ValueError("out must hold one row and one length per sequence")
        _check(self._lib.pa_batch_block_tables(self._h, ids.ctypes.data, n, max_blocks,
                                               tables.ctypes.data,
                                               lens.ctypes.data),
               "pa_batch_block_tables")
        return tables, lens

    def stats(self) -> dict:
        bu, tl, sl, sf = ctypes.c_int32(), ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
        _check(self._lib.pa_alloc_stats(self._h, ctypes.byref(bu), ctypes.byref(tl),
                                        ctypes.byref(sl), ctypes.byref(sf)), "pa_alloc_stats")
        return {"blocks_used": bu.value, "tokens_logical": tl.value, "slots_logical": sl.value,
                "slots_filled": sf.value}

    def check(self) -> None:
        _check(self._lib.pa_alloc_check(self._h), "pa_alloc_check")
