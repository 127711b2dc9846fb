"""CPU oracle for the paged KV-cache decode path.  TEST INFRASTRUCTURE ONLY.

This package is the plain, slow, obviously-correct statement of what the CUDA
path computes.  Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
CPU-baseline / reference arm may import it; the library never does, and it
shares no code with the library (no kernels, helpers, constants or tables).

Source: Kwon et al., "Efficient Memory Management for Large Language Model
Serving with PagedAttention", as restated on three web pages:

* phantomic12.github.io page ("method" paragraph): the KV cache is cut into
  fixed-size blocks that need not be contiguous, a per-request block table
  records which physical blocks belong to the request, and attention reads
  through that table; the same indirection lets requests share a prefix with
  copy-on-write.
* zeroshotmind.com page, sections "Paging the cache" (16-token default block,
  blocks allocated on demand, at most one partially filled tail block),
  "Block tables: logical order, physical scatter" (logical index -> physical
  block; attention walks logical order), "Sharing a prefix without copying it"
  (reference counts; copy-on-write duplicates just the one block being written)
  and "The fragmentation arithmetic" (at most 15 wasted slots per sequence at
  block size 16).

Modules:
  attention      fp64 softmax attention over a sequence reassembled through its
                 block table; per-partition partials and their log-sum-exp merge;
                 several causal query tokens per sequence (chunked prefill).
  cache_ops      slot-mapped append and whole-block copy, element by element.
  allocator_model  reference model of the block allocator (free list, refcounts,
                 fork, copy-on-write append, free) and its invariants.
  content        logical token contents of sequences under add/fork/append/free.
  fragmentation  wasted-slot arithmetic, paged versus contiguous reservation.

Parity status: every function here is pinned by tests under ``tests/`` against
closed forms, brute force or the pages' printed numbers; none is "parity
unpinned".
"""
