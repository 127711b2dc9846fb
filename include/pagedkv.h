/*
 * pagedkv.h - C ABI of libpagedkv.so: paged KV-cache decode attention, the two
 * kernels that keep the paged cache consistent, and the host block allocator.
 *
 * Method: W. Kwon et al., "Efficient Memory Management for Large Language Model
 * Serving with PagedAttention" (SOSP 2023).  Citations below name the web page
 * that restates it and the section on that page:
 *   [P1]  phantomic12.github.io, paper note, method paragraph
 *   [P3b] zeroshotmind.com, "Paging the cache"
 *   [P3c] zeroshotmind.com, "Block tables: logical order, physical scatter"
 *   [P3d] zeroshotmind.com, "Sharing a prefix without copying it"
 *   [P3e] zeroshotmind.com, "The fragmentation arithmetic"
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Memory: every buffer is owned by the caller.  Pointers marked "device" must
 *   point to memory of the current CUDA device; "host" pointers to host memory.
 *   No call allocates device memory.  The library's device image holds one
 *   fixed array of PA_NOALLOC_SCRATCH_BYTES, the scratch of
 *   paged_attn_decode_noalloc; it is resident on a GPU from the moment the
 *   library's device code is loaded there (at context creation under eager
 *   module loading, else at the first call) until the process exits, whichever
 *   entry points are used.
 * - Streams: `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *   stream).  Kernel entry points are asynchronous on that stream: they return
 *   once the work is enqueued.
 * - Return value: a pa_status.  Host-side argument checks fail synchronously
 *   with PA_ERR_INVALID_ARG or PA_ERR_UNSUPPORTED and enqueue nothing.
 *   PA_ERR_CUDA means a CUDA call or launch failed (cudaGetLastError()).
 * - Device-side checks: indices read from device memory (block-table entries,
 *   slots, copy pairs, sequence lengths) are range-checked by the kernels on
 *   every launch.  A bad index is never dereferenced: it is clamped (decode:
 *   block 0 is read instead) or the element is skipped (append, copy), and the
 *   violation is recorded in the caller's device error record if one is given.
 *   Nothing traps.  Kernels that wait on a barrier give up after about one
 *   second, record PA_ERR_TIMEOUT and return.
 * - Device error record: int32_t[PA_ERROR_RECORD_WORDS] in device memory,
 *   zeroed by the caller (pa_error_clear).  Word 0: first error code (0 = none);
 *   word 1: number of violations; word 2: index of the first violation
 *   (sequence, token or pair number); word 3: the offending value (truncated to
 *   32 bits).  May be NULL: checks still clamp/skip, nothing is recorded.
 * - Cache layout (one layer): k_cache and v_cache are each
 *   [num_blocks][num_heads][block_size][head_dim], contiguous, row-major.
 *   Slot s is row (s % block_size) of physical block (s / block_size) [P3b].
 * - dtypes: K/V/Q storage is PA_F16 or PA_BF16; outputs may also be PA_F32.
 *   All attention arithmetic is fp32.
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* 3: pa_decode_opts gained early_inputs, tail_start and counts (appended), so a
 * caller built against version 2 passes a shorter struct and must be rebuilt. */
#define PAGEDKV_VERSION 3
#define PA_ERROR_RECORD_WORDS 4
#define PA_SHARE_MAX_MEMBERS 8
#define PA_SHARE_RECORD_WORDS (2 + PA_SHARE_MAX_MEMBERS)

typedef enum pa_status {
  PA_OK = 0,
  PA_ERR_INVALID_ARG = 1,  /* bad size, pointer, alignment or combination */
  PA_ERR_UNSUPPORTED = 2,  /* well-formed but not built (head_dim, block_size, dtype) */
  PA_ERR_CUDA = 3,         /* a CUDA runtime call or kernel launch failed */
  PA_ERR_BAD_BLOCK = 4,    /* device: block number outside [0, num_blocks) */
  PA_ERR_BAD_SLOT = 5,     /* device: slot >= num_blocks * block_size */
  PA_ERR_BAD_SEQ_LEN = 6,  /* device: seq_len < 0 or > max_blocks_per_seq * block_size */
  PA_ERR_TIMEOUT = 7,      /* device: a bounded wait ran out; the kernel bailed out */
  PA_ERR_OOM = 8,          /* allocator: not enough free blocks */
  PA_ERR_NO_SEQ = 9,       /* allocator: unknown sequence id */
  PA_ERR_SEQ_EXISTS = 10,  /* allocator: sequence id already in use */
  PA_ERR_REFCOUNT = 11     /* allocator: a reference count or free list is inconsistent */
} pa_status;

typedef enum pa_dtype { PA_F16 = 0, PA_BF16 = 1, PA_F32 = 2 } pa_dtype;

/* ---------------------------------------------------------------------------
 * Library information and device error records
 * ------------------------------------------------------------------------- */

/* PAGEDKV_VERSION of the loaded library. */
int pa_version(void);

/* Static English text for a pa_status value (never NULL). */
const char* pa_status_string(int status);

/* Enqueue a zero-fill of a device error record on `stream`. */
int pa_error_clear(int32_t* error_record, void* stream);

/* Copy a device error record into host_out[PA_ERROR_RECORD_WORDS]; waits for
 * `stream` to finish first, so it reports every kernel enqueued before it. */
int pa_error_read(const int32_t* error_record, int32_t* host_out, void* stream);

/* Self-test of the bounded wait that every kernel uses on its mbarriers (no
 * counterpart in the method: a failure-detection check).  One warp waits on a
 * barrier phase that completes only when `arrive` is nonzero.  Without the
 * arrival the wait gives up after limit_ns (1 .. 10^9 ns) and records
 * PA_ERR_TIMEOUT in error_record (device, as above); the kernel then exits
 * normally and the context stays usable.  Asynchronous on `stream`. */
int pa_selftest_bounded_wait(int32_t* error_record, int arrive, unsigned long long limit_ns,
                             void* stream);

/* ---------------------------------------------------------------------------
 * Decode attention through a block table  [P1], [P3c]
 *
 * For every sequence i and head h, with L = seq_lens[i]:
 *   token t (0 <= t < L) is row (t % block_size) of physical block
 *   block_tables[i * max_blocks_per_seq + t / block_size];
 *   s_t = scale * <q[i][h], k_t>,  out[i][h] = sum_t softmax(s)_t * v_t.
 * Attention walks the logical blocks in order; where they sit in the pool does
 * not matter [P3c].  L = 0 gives an all-zero output row.
 *
 * Arguments
 *   q             device, [num_seqs][num_heads][head_dim] in `dtype`, 16-byte aligned
 *   k_cache, v_cache  device, [num_blocks][num_heads][block_size][head_dim] in `dtype`,
 *                 16-byte aligned; read only
 *   block_tables  device int32 [num_seqs][max_blocks_per_seq]; entries past
 *                 ceil(L / block_size) are never read
 *   seq_lens      device int32 [num_seqs]; each in [0, max_blocks_per_seq * block_size]
 *   head_dim      64, 128 or 256;  block_size: a multiple of 16, or 8 (a 16-token
 *                 chunk then spans two blocks, fetched separately)
 *   scale         the softmax scale, usually 1/sqrt(head_dim)
 *   out           device [num_seqs][num_heads][head_dim] in `out_dtype`, 16-byte aligned
 *   partition_tokens  split-K partition length: 0 = automatic (512); otherwise a
 *                 positive multiple of 16 (pa_decode_partition_tokens chooses one
 *                 from the host's lengths).  When max_blocks_per_seq * block_size
 *                 fits in one partition, a single pass writes `out` directly.
 *                 Otherwise a first kernel computes per-partition partials and a
 *                 second merges them by log-sum-exp.
 *   workspace     device, 16-byte aligned, at least paged_attn_workspace_size(...)
 *                 bytes; may be NULL when that size is 0.  Scratch only.
 *   error_record  device error record or NULL.
 * ------------------------------------------------------------------------- */

/* Bytes of workspace paged_attn_decode needs for these sizes (0 if none). */
size_t paged_attn_workspace_size(int num_seqs, int num_heads, int head_dim, int block_size,
                                 int max_blocks_per_seq, int partition_tokens);
/* The same with pa_decode_opts.tail_start given: max(P, 1) partial rows per
 * (sequence, head) plus one tail row each (never 0). */
size_t paged_attn_workspace_size_tails(int num_seqs, int num_heads, int head_dim,
                                       int block_size, int max_blocks_per_seq,
                                       int partition_tokens);

int paged_attn_decode(const void* q, const void* k_cache, const void* v_cache,
                      const int32_t* block_tables, const int32_t* seq_lens, int num_seqs,
                      int num_heads, int head_dim, int block_size, int max_blocks_per_seq,
                      int num_blocks, float scale, int dtype, void* out, int out_dtype,
                      int partition_tokens, void* workspace, size_t workspace_bytes,
                      int32_t* error_record, void* stream);

/* Launch tuning and phase selection for paged_attn_decode_ex.  Zero fields take
 * the automatic choice.
 *   heads_per_cta  heads handled by one thread block (must divide num_heads, <= 8)
 *   stages         shared-memory pipeline depth, 2..8
 *   phases         0 or 3: both passes; 1: partition pass only; 2: merge pass only.
 *   seq_order      NULL, or device int32 [num_seqs]: a permutation of 0..num_seqs-1
 *                  giving the order in which sequences are scheduled (results are
 *                  identical, bit for bit).  Longest first shortens the ragged tail
 *                  of the launch; the host knows the lengths when it builds the
 *                  tables.  An entry outside [0, num_seqs) is recorded as
 *                  PA_ERR_BAD_SEQ_LEN (index = position, value = entry) and skipped;
 *                  a repeated entry leaves some sequence's output unwritten.
 *   work_items     NULL, or device int32 [num_work_items]: the (sequence, partition)
 *                  pairs to run, item = i * P + p (P as below), in the order they
 *                  should be scheduled; seq_order is then ignored.  Listing only the
 *                  partitions that hold tokens (p < ceil(L_i / partition_tokens))
 *                  avoids launching blocks that would exit at once; every such
 *                  pair must appear exactly once for `out` to be complete.  An
 *                  item outside [0, num_seqs * P) is recorded as PA_ERR_BAD_SEQ_LEN
 *                  (index = position, value = item) and skipped.  At most 65535.
 *   shared_records NULL, or device int32 [num_shared][PA_SHARE_RECORD_WORDS]:
 *                  partitions that several sequences share [P3d].  Record r =
 *                  {p, m + 256 c, s_0, ..., s_{m-1}, unused...}: partition p of the m
 *                  (1..PA_SHARE_MAX_MEMBERS) member sequences s_j, whose block
 *                  tables name the same physical blocks over that partition (c = 0),
 *                  or over its first c 16-token chunks only (c > 0, a "prefix
 *                  record", with tail_start below: the rest of the partition is
 *                  each member's own work item).  One
 *                  thread block per (record, head pair) reads each K/V chunk once
 *                  for all members' queries (mma.sync, P as high + low half-
 *                  precision parts, fp32 accumulation) and writes every member's
 *                  partial for partition p, or its output row when p is its only
 *                  partition (c = 0).  Blocks are looked up in s_0's table only.
 *                  With c = 0 each member must cover the whole partition: (p + 1) *
 *                  partition_tokens <= L (<= L - 1 for paged_attn_decode_append,
 *                  whose appended token must lie past it); with c > 0, c <
 *                  partition_tokens / 16 and tail_start[s_j] = p * partition_tokens
 *                  + 16 c < L for every member.  A record that breaks
 *                  these rules is recorded as PA_ERR_BAD_SEQ_LEN (index = record,
 *                  value = the offending field) and skipped.  Requires work_items
 *                  (the pairs not covered by a record; when there are none, any
 *                  non-NULL pointer with num_work_items = 0); every pair that
 *                  holds tokens must appear exactly once across both.  At most
 *                  65535 records.
 *                  pa_decode_share_plan builds both lists.
 *   early_inputs   0, or nonzero to promise that the kernel preceding the call on
 *                  the stream writes none of the call's read-only inputs (q, new_k,
 *                  new_v, block_tables, seq_lens, seq_order, work_items,
 *                  shared_records): they were written by copies, or by kernels that
 *                  completed before that kernel began.  The call's first kernel,
 *                  which is placed while the preceding kernel runs, may then read
 *                  them (its work item, length, block-table entries and query)
 *                  before that kernel has completed; the caches, the workspace and
 *                  `out` are still touched only after it.  Results are identical.
 *   tail_start     NULL, or device int32 [num_seqs]: -1, or for a sequence whose
 *                  partition p is split by a prefix record (see shared_records),
 *                  the token t = p * partition_tokens + 16 c where its own part of
 *                  that partition begins (a multiple of 16 below L).  Its work
 *                  item (i, p) then covers tokens t .. min(L, (p + 1) *
 *                  partition_tokens) - 1 and leaves its partial in a tail row of
 *                  the workspace, which the merge adds to the sequence's others.
 *                  The workspace must then hold paged_attn_workspace_size_tails
 *                  bytes.  pa_decode_share_plan_ex builds the records and this
 *                  array together.  An entry t >= 0 that is not a multiple of 16,
 *                  falls on a partition boundary or lies at or past L is recorded
 *                  as PA_ERR_BAD_SEQ_LEN (index = sequence, value = t); an entry
 *                  with no prefix record naming it leaves that sequence's output
 *                  undefined (its first part is never computed).
 *   counts         NULL, or device int32 [2]: how many of the work_items and of
 *                  the shared_records to run, read by the kernels on the device.
 *                  num_work_items and num_shared are then capacities (the sizes
 *                  of the launches), and the entries past the counts are never
 *                  read.  A call captured once in a CUDA graph can so be replayed
 *                  with lists of other lengths written into the same buffers
 *                  (with the counts).  A count outside [0, capacity] is recorded
 *                  as PA_ERR_BAD_SEQ_LEN (index -1 for the items, -2 for the
 *                  records; value = the count), the pass that reads it computes
 *                  nothing, and `out` is then undefined.
 * With split-K, the partition pass leaves in the workspace, for partition p of
 * sequence i and head h (row = (i * num_heads + h) * P + p, P = ceil(
 * max_blocks_per_seq * block_size / partition_tokens)):
 *   float acc[row][head_dim]  at byte 0:  sum_t 2^(u_t - m) * v_t
 *   float2 ml[row] after all acc rows:   (m, l) with u_t = s_t * log2(e),
 *                                        m = max_t u_t, l = sum_t 2^(u_t - m)
 * over the tokens t of that partition.  Partitions at or past
 * ceil(L / partition_tokens) are not written.  With tail_start, max(P, 1) rows
 * per (sequence, head) and then, after the ml rows, tail rows (i * num_heads + h):
 * float acc_tail[num_seqs * num_heads][head_dim], float2 ml_tail[...]. */
typedef struct pa_decode_opts {
  int heads_per_cta;
  int stages;
  int phases;
  const int32_t* seq_order;
  const int32_t* work_items;
  int num_work_items;
  const int32_t* shared_records;
  int num_shared;
  int early_inputs;
  const int32_t* tail_start;
  const int32_t* counts;
} pa_decode_opts;

int paged_attn_decode_ex(const void* q, const void* k_cache, const void* v_cache,
                         const int32_t* block_tables, const int32_t* seq_lens, int num_seqs,
                         int num_heads, int head_dim, int block_size, int max_blocks_per_seq,
                         int num_blocks, float scale, int dtype, void* out, int out_dtype,
                         int partition_tokens, void* workspace, size_t workspace_bytes,
                         int32_t* error_record, void* stream, const pa_decode_opts* opts);

/* Fused KV append + decode  [P3c], [P3d]
 *
 * One decode step in one pass: for every sequence i with L = seq_lens[i] >= 1,
 * the token at position L - 1 is the one being appended.  Its rows new_k[i] and
 * new_v[i] are written into its slot (row (L-1) % block_size of physical block
 * block_tables[i][(L-1) / block_size], every head) and the decode attends over
 * all L tokens, taking the last one straight from new_k/new_v.  Equivalent,
 * bit for bit, to kv_cache_append at those slots followed by paged_attn_decode,
 * minus one launch and one re-read.  The block holding position L - 1 must be
 * private to sequence i (the allocator's copy-on-write guarantees it).  A
 * sequence with L = 0 appends nothing and gets a zero row.
 *   new_k, new_v  device [num_seqs][num_heads][head_dim] in `dtype`, 16-byte aligned
 *   k_cache, v_cache  written at one row per sequence and head, read elsewhere
 *   opts          as for paged_attn_decode_ex (may be NULL); the append happens
 *                 in the partition pass.
 * Other arguments as for paged_attn_decode. */
int paged_attn_decode_append(const void* q, const void* new_k, const void* new_v, void* k_cache,
                             void* v_cache, const int32_t* block_tables, const int32_t* seq_lens,
                             int num_seqs, int num_heads, int head_dim, int block_size,
                             int max_blocks_per_seq, int num_blocks, float scale, int dtype,
                             void* out, int out_dtype, int partition_tokens, void* workspace,
                             size_t workspace_bytes, int32_t* error_record, void* stream,
                             const pa_decode_opts* opts);

/* Decode schedule, host side  [P3c]
 *
 * The host holds every sequence's length (it builds the block tables), so it
 * can shape a decode launch to the batch: pick the split-K partition length and
 * list the (sequence, partition) work items, and find the partitions that
 * several sequences share.  These functions are host code only: they read host
 * arrays, write host arrays and enqueue nothing.  Results feed
 * paged_attn_workspace_size, partition_tokens and pa_decode_opts.work_items of
 * paged_attn_decode_ex / paged_attn_decode_append; the outputs of the decode are
 * the same whatever is chosen, up to fp32 rounding order across partitions.  The
 * lengths and tables are the same for every layer of a model, so one schedule
 * (and one share plan) serves all the layers of a decode step.
 *
 * pa_decode_partition_tokens: writes to *partition_tokens the longest of 512,
 * 256, 128 and 64 for which the heaviest block, min(partition, max_i L_i)
 * tokens, is at most 1/c of the average work per SM, sum_i L_i * num_heads /
 * heads_per_cta / num_sms, with c = 3.5 for 512 and 256, c = 2 for 128 and
 * c = 1 for 64; else 32.  That length is then doubled, up to 512, while the
 * longest sequence would take more than 32 partitions.  A batch with a lot of
 * work per SM keeps 512; a few short sequences get short partitions so that
 * every SM has blocks.
 *   seq_lens       host int32 [num_seqs], the lengths the decode will see (for
 *                  the fused append: including the appended token); each >= 0
 *   heads_per_cta  as in pa_decode_opts (0 = the automatic choice)
 *   num_sms        SMs of the device the decode runs on; 0 = ask the current
 *                  CUDA device (PA_ERR_CUDA if that fails)
 * Returns PA_OK, or PA_ERR_INVALID_ARG (a negative length, heads_per_cta not
 * dividing num_heads or above 8, NULL pointers) with nothing written.
 *
 * pa_decode_work_items: the work list item = i * P + p for every sequence i,
 * taken in `order`, and every partition p < max(1, ceil(L_i / partition_tokens)),
 * partitions of a sequence in increasing order; P = ceil(max_blocks_per_seq *
 * block_size / partition_tokens).  A sequence with L_i = 0 keeps one item, which
 * writes its zero output row.
 *   partition_tokens  0 = 512 (the decode's automatic length), else a positive
 *                  multiple of 16; must equal the decode call's
 *   order          host int32 [num_seqs], a permutation of 0..num_seqs-1; or NULL
 *                  for longest first (equal lengths in index order)
 *   items          host int32 [capacity], or NULL to only count
 *   num_items      out: the number of items (the decode accepts at most 65535)
 * Returns PA_OK; PA_ERR_INVALID_ARG (a length outside [0, max_blocks_per_seq *
 * block_size], `order` not a permutation, capacity below the count: *num_items
 * still holds the count, items untouched). */
int pa_decode_partition_tokens(const int32_t* seq_lens, int num_seqs, int num_heads,
                               int heads_per_cta, int num_sms, int32_t* partition_tokens);
int pa_decode_work_items(const int32_t* seq_lens, int num_seqs, int partition_tokens,
                         int max_blocks_per_seq, int block_size, const int32_t* order,
                         int32_t* items, int32_t capacity, int32_t* num_items);

/* pa_decode_share_plan: the work list and shared-partition records of a decode
 * over sequences that share blocks [P3d] (parallel samples, beam candidates).
 * For each partition p, the sequences that hold all of it ((p + 1) *
 * partition_tokens <= L_i, or <= L_i - 1 with fused_append) and whose block
 * tables name the same blocks over it are grouped, PA_SHARE_MAX_MEMBERS at most
 * per record; a group of one stays in the work list.  The work list holds every
 * other (sequence, partition) pair as in pa_decode_work_items (same order).
 * Records come partition by partition; unused member slots are -1.
 *   block_tables   host int32 [num_seqs][max_blocks_per_seq], the tables the
 *                  decode will read (entries past a sequence's blocks are not read)
 *   seq_lens, order, partition_tokens  as for pa_decode_work_items
 *   fused_append   nonzero when the plan feeds paged_attn_decode_append
 *   work_items     host int32 [items_capacity]; records: host int32
 *                  [records_capacity][PA_SHARE_RECORD_WORDS]; both NULL to count
 *   num_items, num_records  out: the counts
 * Returns PA_OK or PA_ERR_INVALID_ARG (as for pa_decode_work_items, or a
 * capacity below a count: the counts are still written, the arrays untouched).
 * Host work: per partition, a sort of the sequences that hold it by its first
 * block (blocks are shared only through forks), and an entry-by-entry comparison
 * of the tables within runs of equal first block. */
int pa_decode_share_plan(const int32_t* block_tables, const int32_t* seq_lens, int num_seqs,
                         int max_blocks_per_seq, int block_size, int partition_tokens,
                         int fused_append, const int32_t* order, int32_t* work_items,
                         int32_t items_capacity, int32_t* num_items, int32_t* records,
                         int32_t records_capacity, int32_t* num_records);

/* pa_decode_share_plan_ex: the same, and (prefixes nonzero) prefix records for
 * the partitions a group shares only in part, typically where forked samples or
 * beams diverge.  After the whole-partition records, partition by partition, the
 * sequences whose pair (i, p) is still in the work list, that no earlier prefix
 * record took, and that hold at least 17 tokens of p are grouped by the first
 * block of p; within a group, c = the largest number of leading 16-token chunks
 * of p whose blocks all members' tables name alike, and whose tokens lie below
 * L_i - 1 for every member (the last token stays in the member's own part).  A
 * group of two or more (PA_SHARE_MAX_MEMBERS at most per record, members in
 * index order) with c >= 1 becomes a record {p, m + 256 c, members}, and
 * tail_start[s] = p * partition_tokens + 16 c for each member; the pair (s, p)
 * stays in the work list for the rest.  c is also below partition_tokens / 16.
 * Every other tail_start entry is -1.
 *   tail_start     host int32 [num_seqs] (written only when prefixes is nonzero
 *                  and the arrays are given; may be NULL otherwise) */
int pa_decode_share_plan_ex(const int32_t* block_tables, const int32_t* seq_lens,
                            int num_seqs, int max_blocks_per_seq, int block_size,
                            int partition_tokens, int fused_append, const int32_t* order,
                            int prefixes, int32_t* work_items, int32_t items_capacity,
                            int32_t* num_items, int32_t* records, int32_t records_capacity,
                            int32_t* num_records, int32_t* tail_start);

/* Chunked prefill / multi-query attention through the block table  [P1], [P3c]
 *
 * Several query tokens per sequence, on the tensor cores (tcgen05).  Sequence i
 * holds L = seq_lens[i] tokens in the cache (its new tokens already appended);
 * its last Q_i = query_start[i+1] - query_start[i] tokens are queries, stored at
 * rows query_start[i] .. query_start[i+1]-1 of q.  Query j sits at position
 * p = L - Q_i + j and attends causally over tokens 0..p:
 *   out[query_start[i] + j][h] = softmax_t<=p(scale * <q, k_t>) . v
 * Arithmetic: Q.K^T in fp32 on the tensor cores; probabilities enter P.V as a
 * pair of half-precision numbers (hi + lo), so P.V keeps about 16 mantissa bits;
 * fp32 accumulation.
 *   q             device [total_queries][num_heads][head_dim] in `dtype`, 16-byte aligned
 *   query_start   device int32 [num_seqs + 1], nondecreasing, query_start[num_seqs]
 *                 <= total_queries
 *   max_query_len host: >= every Q_i; the work is num_seqs x num_heads x
 *                 ceil(max_query_len / 128) items, which must be < 2^30
 *   head_dim      64, 128 or 256;  block_size: a multiple of 16, or 8 (each 16-key
 *                 chunk is then loaded as two 8-row boxes)
 *   out           device [total_queries][num_heads][head_dim] in `out_dtype`
 * Rows of out outside every sequence's query range are not written.  A sequence
 * whose range is inconsistent (Q_i > L, range outside q, Q_i > max_query_len) is
 * recorded as PA_ERR_BAD_SEQ_LEN and skipped.  scale must be > 0.  Other
 * arguments as for paged_attn_decode; num_blocks * num_heads * block_size must
 * be < 2^31.  Launch: one block per resident slot on the current device, each
 * looping over its share of the items (it reads the device's SM count on every
 * call). */
int paged_attn_prefill(const void* q, const int32_t* query_start, int total_queries,
                       int max_query_len, const void* k_cache, const void* v_cache,
                       const int32_t* block_tables, const int32_t* seq_lens, int num_seqs,
                       int num_heads, int head_dim, int block_size, int max_blocks_per_seq,
                       int num_blocks, float scale, int dtype, void* out, int out_dtype,
                       int32_t* error_record, void* stream);

/* paged_attn_prefill with scheduling options (opts may be NULL).
 *   seq_order  NULL, or device int32 [num_seqs]: a permutation of 0..num_seqs-1
 *              giving the order in which sequences' blocks are dispatched (results
 *              are identical, bit for bit).  Longest first shortens the ragged
 *              tail.  An entry outside [0, num_seqs) is recorded as
 *              PA_ERR_BAD_SEQ_LEN (index = position, value = entry) and skipped. */
typedef struct pa_prefill_opts {
  const int32_t* seq_order;
} pa_prefill_opts;

int paged_attn_prefill_ex(const void* q, const int32_t* query_start, int total_queries,
                          int max_query_len, const void* k_cache, const void* v_cache,
                          const int32_t* block_tables, const int32_t* seq_lens, int num_seqs,
                          int num_heads, int head_dim, int block_size, int max_blocks_per_seq,
                          int num_blocks, float scale, int dtype, void* out, int out_dtype,
                          int32_t* error_record, void* stream, const pa_prefill_opts* opts);

/* Decode without allocation.  No counterpart in the paper: this is a library
 * convenience.  Some callers cannot allocate device memory - code running
 * inside another runtime whose pool owns all device memory, a serving loop that
 * must never block in cudaMalloc/cudaFree (they can synchronise the device), or
 * a deployment whose device memory budget is fixed at start-up.  This call is
 * paged_attn_decode with the workspace taken from a fixed array of
 * PA_NOALLOC_SCRATCH_BYTES compiled into the library, so it allocates nothing.
 *  - Limit: returns PA_ERR_INVALID_ARG, enqueuing nothing, when
 *    paged_attn_workspace_size(...) for these sizes exceeds PA_NOALLOC_SCRATCH_BYTES.
 *  - The array stays resident on every GPU that loads this code until exit.
 *  - Every call looks up the array's device address in the current context
 *    (cudaGetSymbolAddress, which allocates nothing), so the call stays correct
 *    after cudaDeviceReset or under another driver-API context on the device.
 *    The first call in a context may load the library's device code there:
 *    make it before any stream capture.
 *  - All calls share the array and it keeps the last call's contents (nothing
 *    in it needs clearing: every partial is written before it is read).  Calls
 *    whose kernels overlap on the GPU race on it: serialise them.
 * Other arguments, errors and results: as paged_attn_decode. */
#define PA_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
int paged_attn_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                              const int32_t* block_tables, const int32_t* seq_lens, int num_seqs,
                              int num_heads, int head_dim, int block_size, int max_blocks_per_seq,
                              int num_blocks, float scale, int dtype, void* out, int out_dtype,
                              int partition_tokens, int32_t* error_record, void* stream);

/* ---------------------------------------------------------------------------
 * KV append into slot-mapped blocks  [P3b]
 *
 * For each token t < num_tokens with slot = slot_mapping[t] >= 0, and every head h:
 *   k_cache[slot / block_size][h][slot % block_size][:] = k[t][h][:]   (bit copy)
 *   v_cache[...] likewise.
 * A negative slot marks a padding token: nothing is written.  A slot >=
 * num_blocks * block_size is recorded as PA_ERR_BAD_SLOT and skipped.  Two
 * tokens with the same slot race (one of them wins).
 *   k, v          device [num_tokens][num_heads][head_dim] in `dtype`, 16-byte aligned
 *   slot_mapping  device int64 [num_tokens]
 *   head_dim      a multiple of 8 (rows are moved in 16-byte pieces)
 * ------------------------------------------------------------------------- */
int kv_cache_append(const void* k, const void* v, const int64_t* slot_mapping, int num_tokens,
                    void* k_cache, void* v_cache, int num_heads, int head_dim, int block_size,
                    int num_blocks, int dtype, int32_t* error_record, void* stream);

/* ---------------------------------------------------------------------------
 * Copy-on-write block copy  [P3d]
 *
 * For each pair j < num_pairs, (src, dst) = (pairs[2j], pairs[2j+1]), and each
 * layer l < num_layers: block dst of k_caches[l] and of v_caches[l] becomes a bit
 * copy of block src (all heads, rows and elements).  Destinations must be
 * distinct and no destination may be a source in the same call (the allocator
 * guarantees this: a destination is always a block just taken off the free
 * list); otherwise the result is undefined.  A pair with a block outside
 * [0, num_blocks) is recorded as PA_ERR_BAD_BLOCK and skipped, except the
 * padding pair (-1, -1), which is skipped silently: a launch captured in a CUDA
 * graph with room for num_pairs copies can then replay steps that need fewer.
 *   k_caches, v_caches  HOST arrays of num_layers device pointers (1..128 layers),
 *                 each cache laid out as above, 16-byte aligned
 *   pairs         device int64 [num_pairs][2]
 * ------------------------------------------------------------------------- */
int block_copy(void* const* k_caches, void* const* v_caches, int num_layers,
               const int64_t* pairs, int num_pairs, int num_heads, int head_dim, int block_size,
               int num_blocks, int dtype, int32_t* error_record, void* stream);

/* ---------------------------------------------------------------------------
 * Host block allocator  [P1], [P3b], [P3d], [P3e]
 *
 * Host-only C++ (no device code, no CUDA calls).  Tracks, for a pool of
 * num_blocks blocks of block_size tokens: a free list, a reference count per
 * block, and per sequence (an int64 id) its block table and length.
 *  - A sequence holds exactly ceil(len / block_size) blocks, so at most
 *    block_size - 1 slots are unused, all in its last block [P3b], [P3e].
 *  - A block's reference count is the number of sequences holding it [P3d].
 *  - Appending into a partly filled last block that others also hold first
 *    moves the appender onto a fresh copy of that one block (copy-on-write):
 *    the call returns the (src, dst) pair for block_copy [P3d].
 *  - The free list is a stack.  Blocks are first handed out in `free_order`
 *    order (or 0, 1, 2, ... when NULL) and freed blocks go back on top.
 * An allocator object is not thread-safe; calls on distinct objects are
 * independent.  All pointers are host pointers.
 * ------------------------------------------------------------------------- */
typedef struct pa_allocator pa_allocator;

/* NULL on bad arguments (num_blocks or block_size <= 0, free_order not a
 * permutation of 0..num_blocks-1) or when out of host memory. */
pa_allocator* pa_alloc_create(int32_t num_blocks, int32_t block_size, const int32_t* free_order);
void pa_alloc_destroy(pa_allocator* a);

/* New sequence of num_tokens tokens: takes ceil(num_tokens / block_size) blocks. */
int pa_seq_add(pa_allocator* a, int64_t seq, int32_t num_tokens);
/* child shares every block of parent (each count + 1); child starts at parent's length. */
int pa_seq_fork(pa_allocator* a, int64_t parent, int64_t child);
/* Reserve the slot of seq's next token.  *slot = block * block_size + row.  If the
 * token goes into a shared partly filled block, *cow_src / *cow_dst receive the
 * block pair to copy before writing; otherwise both are -1.  cow_* may be NULL. */
int pa_seq_append(pa_allocator* a, int64_t seq, int64_t* slot, int32_t* cow_src,
                  int32_t* cow_dst);
/* End a sequence: every block's count - 1; blocks reaching 0 return to the free list. */
int pa_seq_free(pa_allocator* a, int64_t seq);
int pa_seq_len(const pa_allocator* a, int64_t seq, int32_t* len);
/* Copy up to `capacity` table entries into out; *num_blocks = the table's length. */
int pa_seq_block_table(const pa_allocator* a, int64_t seq, int32_t* out, int32_t capacity,
                       int32_t* num_blocks);
/* Slots of positions [start, start + count) of seq (all < its length). */
int pa_seq_slots(const pa_allocator* a, int64_t seq, int32_t start, int32_t count,
                 int64_t* slots);
int pa_block_refcount(const pa_allocator* a, int32_t block, int32_t* refcount);
int32_t pa_num_free_blocks(const pa_allocator* a);
int32_t pa_num_seqs(const pa_allocator* a);

/* One append per listed sequence, in order.  slots[n]; cow_pairs[2 * n] receives
 * the copy pairs packed at the front, *num_cow their number.  All-or-nothing:
 * if the free list cannot cover the worst case, returns PA_ERR_OOM and changes
 * nothing. */
int pa_batch_append(pa_allocator* a, const int64_t* seqs, int32_t n, int64_t* slots,
                    int64_t* cow_pairs, int32_t* num_cow);
/* n forks, children[i] sharing every block of parents[i], applied in order (a
 * child forked earlier in the call may be a later parent).  All-or-nothing: a
 * missing parent (PA_ERR_NO_SEQ) or a child that exists or repeats
 * (PA_ERR_SEQ_EXISTS) is reported before anything changes. */
int pa_batch_fork(pa_allocator* a, const int64_t* parents, const int64_t* children, int32_t n);
/* n frees (see pa_seq_free).  All-or-nothing: an id that is missing or listed
 * twice returns PA_ERR_NO_SEQ before anything changes. */
int pa_batch_free(pa_allocator* a, const int64_t* seqs, int32_t n);
/* Block tables of the listed sequences as rows of tables[n][max_blocks] (entries
 * past a table's end are -1) and their lengths. PA_ERR_INVALID_ARG if a table
 * does not fit. */
int pa_batch_block_tables(const pa_allocator* a, const int64_t* seqs, int32_t n,
                          int32_t max_blocks, int32_t* tables, int32_t* seq_lens);
/* Occupancy of the pool [P3b], [P3e].  All outputs optional (NULL to skip):
 *   blocks_used      blocks held by at least one sequence
 *   tokens_logical   sum of all sequences' lengths
 *   slots_logical    sum over sequences of ceil(len / block_size) * block_size
 *                    (what each sequence holds, counting shared blocks once per holder)
 *   slots_filled     sum over used blocks of the rows written in them (the
 *                    furthest any holder has filled that block)
 * Paged waste = 1 - tokens_logical / slots_logical without sharing, and
 * 1 - slots_filled / (blocks_used * block_size) physically. */
int pa_alloc_stats(const pa_allocator* a, int32_t* blocks_used, int64_t* tokens_logical,
                   int64_t* slots_logical, int64_t* slots_filled);
/* Verify every invariant above; PA_OK or PA_ERR_REFCOUNT. */
int pa_alloc_check(const pa_allocator* a);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
