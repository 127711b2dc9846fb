// Single-query decode attention that reads K/V through a per-sequence block
// table (PagedAttention: phantomic12.github.io note, method paragraph;
// zeroshotmind.com page, "Block tables: logical order, physical scatter").
//
// Design (sm_103a, HBM-bound: ~1 flop per byte, so no tensor cores):
//  * Work item = (head group g, partition p, sequence i).  A thread block owns
//    `G` consecutive heads of one sequence and one partition of its tokens.
//    Warps 0..G-1 are consumers (one head each); warp G is the producer.
//  * A partition is cut into 16-token chunks.  For each chunk the producer
//    looks up the physical block in the block table and issues, per head, two
//    1-D bulk copies (cp.async.bulk, the TMA engine's untiled mode) of the K and
//    V rows (16 x head_dim contiguous elements in the [B][H][bs][D] layout) into
//    a ring of `S` shared-memory stages, completing on an mbarrier.  Only the
//    rows that hold tokens are copied, so the last chunk moves no padding.
//  * Consumers compute the 16 scores with a split of each row across
//    D/8 lanes (16-byte loads), reduce them with a transpose-reduce (D/16
//    shuffles for 16 dot products), update an online softmax in the log2
//    domain, and accumulate P*V in fp32 registers.
//  * One partition (the whole sequence fits): write out = acc / l directly.
//    Several: write (m, l, acc) partials; a merge kernel combines them by
//    log-sum-exp.
//  * Fused append (paged_attn_decode_append): the sequence's last token is the
//    one being appended.  Its K/V rows come straight from new_k/new_v into the
//    stage (one extra bulk copy per head), and the consumers of the last
//    partition write them into the token's slot, so no separate append launch
//    and no re-read are needed.  The result is bit-identical to an append
//    followed by a decode.
//  * Every wait is bounded (one second), indices from device memory are range
//    checked, and nothing traps.
//
// This header holds the partition kernel's device code (included by
// paged_attn_decode.cu, which adds the merge kernel and the host side).
#pragma once

#include <cuda_runtime.h>

#include <cmath>

#include "common.cuh"
#include "decode_config.h"

namespace pagedkv {
namespace {

constexpr int kChunk = 16;           // tokens per pipeline stage and head
constexpr int kHeaderBytes = 256;    // mbarriers + abort flag at the front of shared memory
constexpr int kMaxStages = 8;
constexpr float kLog2e = 1.4426950408889634f;

struct DecodeParams {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  const int32_t* seq_lens;
  const int32_t* seq_order;  // optional scheduling permutation of the sequences
  const int32_t* work_items; // optional (sequence * P + partition) list, one per block row
  int num_seqs;
  int num_work_items;
  const void* new_k;   // fused append: [N][H][D] rows of each sequence's last token, or null
  const void* new_v;
  void* k_out;         // fused append: the caches, written at each last token's slot
  void* v_out;
  void* out;
  float* ws_acc;
  float2* ws_ml;
  int32_t* err;
  int num_heads;
  int block_size;
  int max_blocks;
  int num_blocks;
  int partition_tokens;
  int num_partitions;  // P: partitions of the longest possible sequence
  int heads_per_cta;   // G
  int stages;          // S
  int out_dtype;
  float qscale;        // scale * log2(e): scores come out in log2 units
  int wait_first;      // this pass is the call's first kernel (no shared pass before it)
  int early_inputs;    // the read-only inputs may be read before that wait
  const int32_t* tail_start;  // optional [N]: where a sequence's own part of a split partition begins
  float* ws_tail_acc;         // [N * H][D] and [N * H]: the partials of those parts
  float2* ws_tail_ml;
  const int32_t* item_count;  // optional: the work items to run (num_work_items: capacity)
};

// Reduce each of N = TPR/2 partial dot products over the TPR lanes of a row
// group while spreading the results: after the call, the lane with column
// index c holds the full sum of value (c >> 1).  N shuffles in total.
template <int TPR>
__device__ __forceinline__ float transpose_reduce(float (&v)[TPR / 2], int c) {
  constexpr int N = TPR / 2;
#pragma unroll
  for (int step = 0; (TPR >> (step + 1)) >= 2; ++step) {
    const int mask = TPR >> (step + 1);
    const int n = N >> step;
    const bool upper = (c & mask) != 0;
#pragma unroll
    for (int j = 0; j < n / 2; ++j) {
      const float send = upper ? v[j] : v[j + n / 2];
      const float keep = upper ? v[j + n / 2] : v[j];
      v[j] = keep + __shfl_xor_sync(kFullMask, send, mask);
    }
  }
  return v[0] + __shfl_xor_sync(kFullMask, v[0], 1);
}

// Waits for the grid this pass depends on programmatically (the pass over
// shared partitions, or the kernel before the call) to complete and its writes
// to be visible.  A no-op without such a prerequisite, and when it has already
// been waited for.
__device__ __forceinline__ void wait_prerequisite() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// A block's last step.  As the call's first kernel the pass waits for its
// prerequisite in every block (no block may finish before the kernel before the
// call has).  Behind the shared-partition pass, whose blocks all waited for the
// kernel before the call before this pass could start, only the first block waits
// for that pass, so that this grid (and so the merge after it) completes after
// both; the other blocks free their slots as soon as their work is done.
__device__ __forceinline__ void finish(const DecodeParams& p) {
  if (p.wait_first || (blockIdx.x | blockIdx.y | blockIdx.z) == 0) wait_prerequisite();
}

__device__ __forceinline__ int clamp_len(const DecodeParams& p, int seq, bool report) {
  int L = p.seq_lens[seq];
  const int cap = p.max_blocks * p.block_size;
  if (L < 0 || L > cap) {
    if (report) report_error(p.err, PA_ERR_BAD_SEQ_LEN, seq, L);
    L = L < 0 ? 0 : cap;
  }
  return L;
}

template <class Tag, int D>
__global__ void __launch_bounds__((kMaxHeadsPerCta + 1) * 32)
    paged_attn_partition_kernel(const DecodeParams p) {
  constexpr int TPR = D / 8;          // lanes per K/V row (16 bytes each)
  constexpr int RPI = 32 / TPR;       // rows a warp covers per load
  constexpr int TPL = kChunk / RPI;   // rows per lane per chunk (= TPR / 2)
  constexpr int ROW_BYTES = D * 2;
  constexpr int CHUNK_BYTES = kChunk * ROW_BYTES;
  static_assert(TPL * 2 == TPR, "lane split");

  extern __shared__ __align__(128) uint8_t smem[];
  // The merge after this pass is a programmatic dependent that waits for this
  // grid to complete before reading: let it be placed once every block here has
  // started.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // As the call's first kernel this pass is itself launched as a programmatic
  // dependent of whatever precedes it on the stream (the merge of the previous
  // decode call, typically), so that its blocks are resident when that kernel
  // ends.  Nothing in memory is touched before that kernel has completed and
  // its writes are visible.  Behind the shared-partition pass the wait stays at
  // the end instead (that pass waited for the predecessor before it let this
  // one start).  With early_inputs the caller promises that the predecessor
  // writes none of the read-only inputs: the work item, length, block-table
  // entries and query are then read first, and the wait comes just before the
  // caches, the workspace or `out` are touched (in the producer before its first
  // copy, in each consumer warp before its first chunk).
  const bool early = p.wait_first && p.early_inputs;
  if (p.wait_first && !early) wait_prerequisite();
  const int G = p.heads_per_cta;
  const int S = p.stages;
  const int hg = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int part = blockIdx.y, seq = blockIdx.z;
  if (p.work_items != nullptr) {
    if (p.item_count != nullptr) {  // a launch sized for the list's capacity
      const int n = __ldg(p.item_count);
      if (n < 0 || n > p.num_work_items) {
        if (threadIdx.x == 0 && hg == 0 && blockIdx.y == 0)
          report_error(p.err, PA_ERR_BAD_SEQ_LEN, -1, n);
        finish(p);
        return;
      }
      if (static_cast<int>(blockIdx.y) >= n) {
        finish(p);
        return;
      }
    }
    const int item = __ldg(p.work_items + blockIdx.y);
    if (item < 0 || item / p.num_partitions >= p.num_seqs) {
      if (threadIdx.x == 0 && hg == 0) report_error(p.err, PA_ERR_BAD_SEQ_LEN, blockIdx.y, item);
      finish(p);
      return;
    }
    seq = item / p.num_partitions;
    part = item % p.num_partitions;
  } else if (p.seq_order != nullptr) {
    seq = __ldg(p.seq_order + blockIdx.z);
    if (static_cast<unsigned>(seq) >= static_cast<unsigned>(p.num_seqs)) {
      if (threadIdx.x == 0 && hg == 0 && part == 0)
        report_error(p.err, PA_ERR_BAD_SEQ_LEN, blockIdx.z, seq);
      finish(p);
      return;
    }
  }

  const int L = clamp_len(p, seq, threadIdx.x == 0 && hg == 0 && part == 0);
  const int nparts = L > 0 ? (L + p.partition_tokens - 1) / p.partition_tokens : 1;
  if (part >= nparts) {
    finish(p);
    return;
  }
  int tok_begin = part * p.partition_tokens;
  const int tok_end = min(L, tok_begin + p.partition_tokens);
  // A partition whose first chunks a prefix record reads for several sequences:
  // this item covers the sequence's own part, from tail_start on, and leaves its
  // partial in the sequence's tail row, which the merge adds to the others.
  bool tail = false;
  if (p.tail_start != nullptr) {
    const int ts = __ldg(p.tail_start + seq);
    if (ts >= 0 && ts / p.partition_tokens == part) {
      if (ts <= tok_begin || ts >= tok_end || ts % kChunk != 0) {
        if (threadIdx.x == 0 && hg == 0) report_error(p.err, PA_ERR_BAD_SEQ_LEN, seq, ts);
        finish(p);
        return;
      }
      tok_begin = ts;
      tail = true;
    }
  }
  const int nchunks = (max(0, tok_end - tok_begin) + kChunk - 1) / kChunk;

  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + S;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 2 * kMaxStages * 8);
  uint8_t* stages = smem + kHeaderBytes;
  const size_t stage_bytes = static_cast<size_t>(G) * 2 * CHUNK_BYTES;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], G);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  int issued = 0;  // producer lane 0 only
  if (warp == G) {
    // ------------------------------------------------------------ producer
    const uint64_t policy = l2_policy_evict_first();
    const int32_t* table = p.block_tables + static_cast<size_t>(seq) * p.max_blocks;
    const char* kbase = static_cast<const char*>(p.k_cache);
    const char* vbase = static_cast<const char*>(p.v_cache);
    const int h0 = hg * G;
    // A 16-token chunk lies in one block when the block size is a multiple of
    // 16; with 8-token blocks it spans two (sub = 2), each copied on its own.
    const int sub = p.block_size >= kChunk ? 1 : 2;
    const int per_round = 32 / sub;  // chunks whose blocks one round of table reads covers
    bool stop = false;
    for (int c0 = 0; c0 < nchunks && !stop; c0 += per_round) {
      // Lane l fetches the physical block of chunk c0 + l (sub = 1), or of
      // half l % 2 of chunk c0 + l / 2 (sub = 2); entries past the sequence's
      // last token are not read.
      int blk = 0;
      {
        const int chunk = c0 + lane / sub;
        const int tok = tok_begin + chunk * kChunk + (lane % sub) * (kChunk / sub);
        if (chunk < nchunks && tok < tok_end) {
          blk = __ldg(table + tok / p.block_size);
          if (static_cast<unsigned>(blk) >= static_cast<unsigned>(p.num_blocks)) {
            report_error(p.err, PA_ERR_BAD_BLOCK, seq, blk);
            blk = 0;
          }
        }
      }
      if (early && c0 == 0) wait_prerequisite();
      const int n = min(per_round, nchunks - c0);
      for (int j = 0; j < n; ++j) {
        const int b = __shfl_sync(kFullMask, blk, j * sub);
        const int b_hi = sub == 2 ? __shfl_sync(kFullMask, blk, j * sub + 1) : 0;
        if (lane == 0) {
          const int chunk = c0 + j;
          const int s = chunk % S;
          bool ok = true;
          if (chunk >= S) ok = mbar_wait_bounded(&empty[s], ((chunk / S) - 1) & 1);
          if (!ok) {
            *abort_flag = 1;
            report_error(p.err, PA_ERR_TIMEOUT, seq, chunk);
          } else {
            const int tok = tok_begin + chunk * kChunk;
            const int rows = min(kChunk, tok_end - tok);
            // With a fused append, the chunk that ends the sequence takes its
            // last row from new_k/new_v instead of the cache.
            const bool new_here = p.new_k != nullptr && tok + rows == L;
            const int cache_rows = rows - (new_here ? 1 : 0);
            const uint32_t bytes = static_cast<uint32_t>(cache_rows) * ROW_BYTES;
            const int row0 = tok % p.block_size;
            mbar_arrive_expect_tx(&full[s], 2u * G * static_cast<uint32_t>(rows) * ROW_BYTES);
            uint8_t* dst = stages + s * stage_bytes;
            // with 8-token blocks: rows 0-7 of the chunk from block b, rows 8-15 from b_hi
            const int rows_lo = sub == 2 ? min(cache_rows, kChunk / 2) : cache_rows;
            const int rows_hi = cache_rows - rows_lo;
            const uint32_t bytes_lo = static_cast<uint32_t>(rows_lo) * ROW_BYTES;
            for (int w = 0; w < G; ++w) {
              uint8_t* kd = dst + w * 2 * CHUNK_BYTES;
              if (rows_lo > 0) {
                const size_t off =
                    ((static_cast<size_t>(b) * p.num_heads + h0 + w) * p.block_size + row0) *
                    ROW_BYTES;
                bulk_g2s(kd, kbase + off, bytes_lo, &full[s], policy);
                bulk_g2s(kd + CHUNK_BYTES, vbase + off, bytes_lo, &full[s], policy);
              }
              if (rows_hi > 0) {
                const size_t off =
                    (static_cast<size_t>(b_hi) * p.num_heads + h0 + w) * p.block_size * ROW_BYTES;
                const uint32_t bytes_hi = static_cast<uint32_t>(rows_hi) * ROW_BYTES;
                bulk_g2s(kd + bytes_lo, kbase + off, bytes_hi, &full[s], policy);
                bulk_g2s(kd + CHUNK_BYTES + bytes_lo, vbase + off, bytes_hi, &full[s], policy);
              }
              if (new_here) {
                const size_t off = (static_cast<size_t>(seq) * p.num_heads + h0 + w) * ROW_BYTES;
                bulk_g2s(kd + bytes, static_cast<const char*>(p.new_k) + off, ROW_BYTES, &full[s],
                         policy);
                bulk_g2s(kd + CHUNK_BYTES + bytes, static_cast<const char*>(p.new_v) + off,
                         ROW_BYTES, &full[s], policy);
              }
            }
            ++issued;
          }
        }
        __syncwarp();
        if (__shfl_sync(kFullMask, *abort_flag, 0)) {
          stop = true;
          break;
        }
      }
    }
  } else {
    // ------------------------------------------------------------ consumer
    const int h = hg * G + warp;
    const int r = lane / TPR;  // row group
    const int c = lane % TPR;  // 16-byte column
    float qf[8];
    {
      const uint4 qv = *reinterpret_cast<const uint4*>(
          static_cast<const char*>(p.q) + (static_cast<size_t>(seq) * p.num_heads + h) * ROW_BYTES +
          c * 16);
      to_float8(qv, qf, Tag{});
#pragma unroll
      for (int j = 0; j < 8; ++j) qf[j] *= p.qscale;
    }
    if (early) wait_prerequisite();
    float m = -INFINITY, lsum = 0.f;
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.f;
    const int my_slot = (c >> 1) * RPI + r;  // token slot whose score this lane ends up with

    for (int chunk = 0; chunk < nchunks; ++chunk) {
      const int s = chunk % S;
      const bool ok = __all_sync(kFullMask, mbar_wait_bounded(&full[s], (chunk / S) & 1));
      if (!ok) {
        if (lane == 0) {
          *abort_flag = 1;
          report_error(p.err, PA_ERR_TIMEOUT, seq, chunk);
        }
        break;
      }
      const uint8_t* ks = stages + s * stage_bytes + warp * 2 * CHUNK_BYTES;
      const uint8_t* vs = ks + CHUNK_BYTES;
      const int rows = min(kChunk, tok_end - (tok_begin + chunk * kChunk));

      // scores (log2 units) of the 16 tokens, spread one per lane pair
      float part_dot[TPL];
#pragma unroll
      for (int k = 0; k < TPL; ++k) {
        const uint4 kv = *reinterpret_cast<const uint4*>(ks + (k * RPI + r) * ROW_BYTES + c * 16);
        float kf[8];
        to_float8(kv, kf, Tag{});
        float d = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) d = fmaf(qf[j], kf[j], d);
        part_dot[k] = d;
      }
      float score = transpose_reduce<TPR>(part_dot, c);
      if (my_slot >= rows) score = -INFINITY;

      // online softmax: the chunk max raises the running max, rescale the rest
      float cmax = score;
#pragma unroll
      for (int off = 2; off < 32; off <<= 1) cmax = fmaxf(cmax, __shfl_xor_sync(kFullMask, cmax, off));
      const float m_new = fmaxf(m, cmax);
      const float alpha = exp2f(m - m_new);
      const float pr = exp2f(score - m_new);
      lsum = fmaf(lsum, alpha, pr);
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] *= alpha;

#pragma unroll
      for (int k = 0; k < TPL; ++k) {
        const int t = k * RPI + r;
        const float pk = __shfl_sync(kFullMask, pr, r * TPR + 2 * k);
        if (t < rows) {
          const uint4 vv = *reinterpret_cast<const uint4*>(vs + t * ROW_BYTES + c * 16);
          float vf[8];
          to_float8(vv, vf, Tag{});
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[j] = fmaf(pk, vf[j], acc[j]);
        }
      }
      m = m_new;
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      if (__shfl_sync(kFullMask, *abort_flag, 0)) break;
    }

    // combine the row groups, then the per-lane softmax sums (even lanes only:
    // odd lanes hold copies of their even neighbour's score)
#pragma unroll
    for (int off = TPR; off < 32; off <<= 1) {
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] += __shfl_xor_sync(kFullMask, acc[j], off);
    }
    float l = (lane & 1) ? 0.f : lsum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) l += __shfl_xor_sync(kFullMask, l, off);

    if (tail) {
      const size_t row = static_cast<size_t>(seq) * p.num_heads + h;
      if (r == 0) {
        float* dst = p.ws_tail_acc + row * D + c * 8;
        *reinterpret_cast<float4*>(dst) = make_float4(acc[0], acc[1], acc[2], acc[3]);
        *reinterpret_cast<float4*>(dst + 4) = make_float4(acc[4], acc[5], acc[6], acc[7]);
      }
      if (lane == 0) p.ws_tail_ml[row] = make_float2(m, l);
    } else if (nparts == 1) {
      const float inv = l > 0.f ? 1.f / l : 0.f;
      if (r == 0) {
        float o[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) o[j] = acc[j] * inv;
        store_out<8>(p.out, (static_cast<size_t>(seq) * p.num_heads + h) * D + c * 8, o,
                     p.out_dtype);
      }
    } else {
      const size_t row = (static_cast<size_t>(seq) * p.num_heads + h) * p.num_partitions + part;
      if (r == 0) {
        float* dst = p.ws_acc + row * D + c * 8;
        *reinterpret_cast<float4*>(dst) = make_float4(acc[0], acc[1], acc[2], acc[3]);
        *reinterpret_cast<float4*>(dst + 4) = make_float4(acc[4], acc[5], acc[6], acc[7]);
      }
      if (lane == 0) p.ws_ml[row] = make_float2(m, l);
    }

    // Fused append: the block holding the last token stores its rows into the
    // token's slot (the table entry was range-checked by the producer; a bad
    // one is skipped here).
    if (p.new_k != nullptr && L > 0 && part == nparts - 1) {
      const int pos = L - 1;
      const int blk =
          __ldg(p.block_tables + static_cast<size_t>(seq) * p.max_blocks + pos / p.block_size);
      if (static_cast<unsigned>(blk) < static_cast<unsigned>(p.num_blocks)) {
        const size_t dst =
            ((static_cast<size_t>(blk) * p.num_heads + h) * p.block_size + pos % p.block_size) *
            ROW_BYTES;
        const size_t src = (static_cast<size_t>(seq) * p.num_heads + h) * ROW_BYTES;
        for (int piece = lane; piece < 2 * TPR; piece += 32) {
          const bool is_v = piece >= TPR;
          const int x = (is_v ? piece - TPR : piece) * 16;
          const uint4 val = *reinterpret_cast<const uint4*>(
              static_cast<const char*>(is_v ? p.new_v : p.new_k) + src + x);
          *reinterpret_cast<uint4*>(static_cast<char*>(is_v ? p.v_out : p.k_out) + dst + x) = val;
        }
      }
    }
  }

  __syncthreads();
  // After a timeout, wait (bounded) for the copies still in flight so that no
  // bulk copy lands in shared memory after the block has exited.
  if (*abort_flag && warp == G && lane == 0) {
    for (int s = 0; s < S && s < issued; ++s) {
      const int last = s + ((issued - 1 - s) / S) * S;  // last chunk issued into stage s
      mbar_wait_bounded(&full[s], (last / S) & 1);
    }
  }
  finish(p);
}

}  // namespace
}  // namespace pagedkv
