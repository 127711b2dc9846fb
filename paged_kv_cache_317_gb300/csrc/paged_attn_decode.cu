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
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>

#include "common.cuh"
#include "decode_config.h"
#include "decode_shared.h"

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
  // A pass over shared partitions may follow as a programmatic dependent (it
  // reads nothing this kernel writes): let it start once every block here has.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int G = p.heads_per_cta;
  const int S = p.stages;
  const int hg = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int part = blockIdx.y, seq = blockIdx.z;
  if (p.work_items != nullptr) {
    const int item = __ldg(p.work_items + blockIdx.y);
    if (item < 0 || item / p.num_partitions >= p.num_seqs) {
      if (threadIdx.x == 0 && hg == 0) report_error(p.err, PA_ERR_BAD_SEQ_LEN, blockIdx.y, item);
      return;
    }
    seq = item / p.num_partitions;
    part = item % p.num_partitions;
  } else if (p.seq_order != nullptr) {
    seq = __ldg(p.seq_order + blockIdx.z);
    if (static_cast<unsigned>(seq) >= static_cast<unsigned>(p.num_seqs)) {
      if (threadIdx.x == 0 && hg == 0 && part == 0)
        report_error(p.err, PA_ERR_BAD_SEQ_LEN, blockIdx.z, seq);
      return;
    }
  }

  const int L = clamp_len(p, seq, threadIdx.x == 0 && hg == 0 && part == 0);
  const int nparts = L > 0 ? (L + p.partition_tokens - 1) / p.partition_tokens : 1;
  if (part >= nparts) return;
  const int tok_begin = part * p.partition_tokens;
  const int tok_end = min(L, tok_begin + p.partition_tokens);
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
    bool stop = false;
    for (int c0 = 0; c0 < nchunks && !stop; c0 += 32) {
      // Lane j fetches the physical block of chunk c0 + j.
      int blk = 0;
      if (c0 + lane < nchunks) {
        const int tok = tok_begin + (c0 + lane) * kChunk;
        blk = __ldg(table + tok / p.block_size);
        if (static_cast<unsigned>(blk) >= static_cast<unsigned>(p.num_blocks)) {
          report_error(p.err, PA_ERR_BAD_BLOCK, seq, blk);
          blk = 0;
        }
      }
      const int n = min(32, nchunks - c0);
      for (int j = 0; j < n; ++j) {
        const int b = __shfl_sync(kFullMask, blk, j);
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
            for (int w = 0; w < G; ++w) {
              uint8_t* kd = dst + w * 2 * CHUNK_BYTES;
              if (cache_rows > 0) {
                const size_t off =
                    ((static_cast<size_t>(b) * p.num_heads + h0 + w) * p.block_size + row0) *
                    ROW_BYTES;
                bulk_g2s(kd, kbase + off, bytes, &full[s], policy);
                bulk_g2s(kd + CHUNK_BYTES, vbase + off, bytes, &full[s], policy);
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

    if (nparts == 1) {
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
}

// One warp per (sequence, head): out = sum_p 2^(m_p - M) acc_p / sum_p 2^(m_p - M) l_p.
struct MergeParams {
  const int32_t* seq_lens;
  const float* ws_acc;
  const float2* ws_ml;
  void* out;
  int num_seqs, num_heads, capacity, partition_tokens, num_partitions, out_dtype;
};

template <int D>
__global__ void __launch_bounds__(256) paged_attn_merge_kernel(const MergeParams p) {
  constexpr int DPL = D / 32;  // dims per lane
  const int gw = static_cast<int>((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (gw >= p.num_seqs * p.num_heads) return;
  const int seq = gw / p.num_heads;
  int L = p.seq_lens[seq];
  L = L < 0 ? 0 : (L > p.capacity ? p.capacity : L);
  const int nparts = L > 0 ? (L + p.partition_tokens - 1) / p.partition_tokens : 1;
  if (nparts <= 1) return;  // the partition pass wrote this row directly
  const size_t row0 = static_cast<size_t>(gw) * p.num_partitions;

  float M = -INFINITY;
  for (int i = lane; i < nparts; i += 32) M = fmaxf(M, p.ws_ml[row0 + i].x);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(kFullMask, M, off));
  float o[DPL];
#pragma unroll
  for (int j = 0; j < DPL; ++j) o[j] = 0.f;
  float lt = 0.f;
  if (M != -INFINITY) {
    for (int i = lane; i < nparts; i += 32) {
      const float2 ml = p.ws_ml[row0 + i];
      lt = fmaf(exp2f(ml.x - M), ml.y, lt);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) lt += __shfl_xor_sync(kFullMask, lt, off);
    for (int i = 0; i < nparts; ++i) {
      const float w = exp2f(p.ws_ml[row0 + i].x - M);
      const float* a = p.ws_acc + (row0 + i) * D + lane * DPL;
#pragma unroll
      for (int j = 0; j < DPL; ++j) o[j] = fmaf(w, a[j], o[j]);
    }
  }
  const float inv = lt > 0.f ? 1.f / lt : 0.f;
#pragma unroll
  for (int j = 0; j < DPL; ++j) o[j] *= inv;
  store_out<DPL>(p.out, static_cast<size_t>(gw) * D + lane * DPL, o, p.out_dtype);
}

// ------------------------------------------------------------------ host side
int num_partitions_for(int capacity, int partition_tokens) {
  return capacity <= 0 ? 1 : (capacity + partition_tokens - 1) / partition_tokens;
}

size_t workspace_bytes_for(int num_seqs, int num_heads, int head_dim, int P) {
  if (P <= 1) return 0;
  const size_t rows = static_cast<size_t>(num_seqs) * num_heads * P;
  return rows * head_dim * sizeof(float) + rows * sizeof(float2);
}

int resolve_partition(int partition_tokens) {
  return partition_tokens <= 0 ? kDefaultPartition : partition_tokens;
}

// Per-instantiation, per-device record of the opt-in shared memory attribute.
template <class Tag, int D>
cudaError_t ensure_smem_attr(int device) {
  static std::atomic<uint64_t> done{0};
  const uint64_t bit = device < 64 ? (1ull << device) : 0;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  int optin = 0;
  cudaError_t e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(paged_attn_partition_kernel<Tag, D>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

template <class Tag, int D>
int launch(const DecodeParams& p, int num_seqs, int phases, size_t smem,
           const SharedParams* shared, int dtype, cudaStream_t stream) {
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return PA_ERR_CUDA;
  if (phases & 1) {
    // The per-sequence partition pass first; the pass over shared partitions
    // (if any) follows as its programmatic dependent, so its long, uniform blocks
    // start as soon as every block of the first pass has started and fill the
    // SMs that pass's ragged last wave leaves idle.  The two write disjoint
    // partials; the shared pass's blocks wait for the first pass to complete
    // before they exit, so the merge after it follows both.
    if (ensure_smem_attr<Tag, D>(device) != cudaSuccess) return PA_ERR_CUDA;
    dim3 grid(p.num_heads / p.heads_per_cta, p.num_partitions, num_seqs);
    if (p.work_items != nullptr) grid = dim3(p.num_heads / p.heads_per_cta, p.num_work_items, 1);
    dim3 block((p.heads_per_cta + 1) * 32);
    if (grid.y > 0) {
      paged_attn_partition_kernel<Tag, D><<<grid, block, smem, stream>>>(p);
      if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;
    }
    if (shared != nullptr) {
      const int st = launch_shared_partitions(*shared, dtype, D, grid.y > 0, stream);
      if (st != PA_OK) return st;
    }
  }
  if ((phases & 2) && p.num_partitions > 1) {
    MergeParams mp{p.seq_lens, p.ws_acc, p.ws_ml, p.out, num_seqs, p.num_heads,
                   p.max_blocks * p.block_size, p.partition_tokens, p.num_partitions,
                   p.out_dtype};
    const long long warps = static_cast<long long>(num_seqs) * p.num_heads;
    dim3 grid(static_cast<unsigned>((warps + 7) / 8));
    paged_attn_merge_kernel<D><<<grid, 256, 0, stream>>>(mp);
    if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;
  }
  return PA_OK;
}

}  // namespace
}  // namespace pagedkv

using namespace pagedkv;

extern "C" size_t paged_attn_workspace_size(int num_seqs, int num_heads, int head_dim,
                                            int block_size, int max_blocks_per_seq,
                                            int partition_tokens) {
  if (num_seqs <= 0 || num_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
      max_blocks_per_seq <= 0)
    return 0;
  const int pt = resolve_partition(partition_tokens);
  const long long cap = static_cast<long long>(max_blocks_per_seq) * block_size;
  if (cap > (1ll << 30)) return 0;
  const int P = num_partitions_for(static_cast<int>(cap), pt);
  return workspace_bytes_for(num_seqs, num_heads, head_dim, P);
}

namespace {
int decode_common(const void* q, const void* new_k, const void* new_v, const void* k_cache,
                  const void* v_cache, void* k_out, void* v_out, const int32_t* block_tables,
                  const int32_t* seq_lens, int num_seqs, int num_heads, int head_dim,
                  int block_size, int max_blocks_per_seq, int num_blocks, float scale, int dtype,
                  void* out, int out_dtype, int partition_tokens, void* workspace,
                  size_t workspace_bytes, int32_t* error_record, void* stream,
                  const pa_decode_opts* opts) {
  NvtxRange range(new_k ? "paged_attn_decode_append" : "paged_attn_decode");
  if (num_seqs < 0 || num_heads <= 0 || block_size <= 0 || max_blocks_per_seq <= 0 ||
      num_blocks <= 0)
    return PA_ERR_INVALID_ARG;
  if (num_seqs == 0) return PA_OK;
  if (head_dim != 64 && head_dim != 128 && head_dim != 256) return PA_ERR_UNSUPPORTED;
  if (block_size % 16 != 0) return PA_ERR_UNSUPPORTED;
  if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
  if (out_dtype != PA_F16 && out_dtype != PA_BF16 && out_dtype != PA_F32)
    return PA_ERR_UNSUPPORTED;
  if (!q || !k_cache || !v_cache || !block_tables || !seq_lens || !out) return PA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
    return PA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return PA_ERR_INVALID_ARG;
  if (partition_tokens > 0 && partition_tokens % 16 != 0) return PA_ERR_INVALID_ARG;
  const long long cap = static_cast<long long>(max_blocks_per_seq) * block_size;
  if (cap > (1ll << 30) || static_cast<long long>(num_blocks) * num_heads * block_size > (1ll << 40))
    return PA_ERR_INVALID_ARG;

  const int G = (opts && opts->heads_per_cta > 0) ? opts->heads_per_cta : auto_heads_per_cta(num_heads);
  if (G > kMaxHeadsPerCta || num_heads % G != 0) return PA_ERR_INVALID_ARG;
  const int row_bytes = head_dim * 2;
  int S = (opts && opts->stages > 0) ? opts->stages : 0;
  if (S == 0) S = 2;
  if (S < 2 || S > kMaxStages) return PA_ERR_INVALID_ARG;
  const size_t smem = kHeaderBytes + static_cast<size_t>(S) * G * 2 * kChunk * row_bytes;
  if (smem > 227 * 1024) return PA_ERR_INVALID_ARG;
  const int phases = (opts && opts->phases > 0) ? opts->phases : 3;
  if (phases > 3) return PA_ERR_INVALID_ARG;

  const int pt = resolve_partition(partition_tokens);
  const int P = num_partitions_for(static_cast<int>(cap), pt);
  if (num_seqs > 65535 || P > 65535) return PA_ERR_INVALID_ARG;
  const size_t need = workspace_bytes_for(num_seqs, num_heads, head_dim, P);
  if (need > 0 && (!workspace || workspace_bytes < need || !aligned16(workspace)))
    return PA_ERR_INVALID_ARG;

  DecodeParams p{};
  p.q = q;
  p.seq_order = opts ? opts->seq_order : nullptr;
  p.work_items = opts ? opts->work_items : nullptr;
  p.num_work_items = p.work_items ? opts->num_work_items : 0;
  if (p.work_items && (p.num_work_items < 0 || p.num_work_items > 65535))
    return PA_ERR_INVALID_ARG;
  p.num_seqs = num_seqs;
  p.new_k = new_k;
  p.new_v = new_v;
  p.k_out = k_out;
  p.v_out = v_out;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.block_tables = block_tables;
  p.seq_lens = seq_lens;
  p.out = out;
  p.ws_acc = static_cast<float*>(workspace);
  p.ws_ml = need ? reinterpret_cast<float2*>(static_cast<char*>(workspace) +
                                             static_cast<size_t>(num_seqs) * num_heads * P *
                                                 head_dim * sizeof(float))
                 : nullptr;
  p.err = error_record;
  p.num_heads = num_heads;
  p.block_size = block_size;
  p.max_blocks = max_blocks_per_seq;
  p.num_blocks = num_blocks;
  p.partition_tokens = pt;
  p.num_partitions = P;
  p.heads_per_cta = G;
  p.stages = S;
  p.out_dtype = out_dtype;
  p.qscale = scale * kLog2e;

  // Partitions that several sequences share (records built on the host); the
  // remaining (sequence, partition) pairs must then come as a work list.
  SharedParams sp{};
  const SharedParams* shared = nullptr;
  if (opts && opts->shared_records && opts->num_shared != 0) {
    if (opts->num_shared < 0 || opts->num_shared > 65535 || !p.work_items)
      return PA_ERR_INVALID_ARG;
    sp.q = q;
    sp.k_cache = k_cache;
    sp.v_cache = v_cache;
    sp.block_tables = block_tables;
    sp.seq_lens = seq_lens;
    sp.records = opts->shared_records;
    sp.num_records = opts->num_shared;
    sp.num_seqs = num_seqs;
    sp.num_heads = num_heads;
    sp.block_size = block_size;
    sp.max_blocks = max_blocks_per_seq;
    sp.num_blocks = num_blocks;
    sp.partition_tokens = pt;
    sp.num_partitions = P;
    // one head per block: twice the blocks at ~6 per SM instead of ~4 (register
    // bound), so the shared pass's equal-sized blocks leave a smaller last wave
    sp.heads_per_cta = 1;
    sp.stages = shared_kernel_smem_bytes(head_dim, sp.heads_per_cta, S) <= 227 * 1024 ? S : 2;
    sp.fused_append = new_k != nullptr ? 1 : 0;
    sp.out_dtype = out_dtype;
    sp.qscale = p.qscale;
    sp.out = out;
    sp.ws_acc = p.ws_acc;
    sp.ws_ml = p.ws_ml;
    sp.err = error_record;
    shared = &sp;
  }

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (dtype == PA_BF16) {
    switch (head_dim) {
      case 64: return launch<BF16, 64>(p, num_seqs, phases, smem, shared, dtype, st);
      case 128: return launch<BF16, 128>(p, num_seqs, phases, smem, shared, dtype, st);
      default: return launch<BF16, 256>(p, num_seqs, phases, smem, shared, dtype, st);
    }
  }
  switch (head_dim) {
    case 64: return launch<F16, 64>(p, num_seqs, phases, smem, shared, dtype, st);
    case 128: return launch<F16, 128>(p, num_seqs, phases, smem, shared, dtype, st);
    default: return launch<F16, 256>(p, num_seqs, phases, smem, shared, dtype, st);
  }
}

}  // namespace

extern "C" int paged_attn_decode_ex(const void* q, const void* k_cache, const void* v_cache,
                                    const int32_t* block_tables, const int32_t* seq_lens,
                                    int num_seqs, int num_heads, int head_dim, int block_size,
                                    int max_blocks_per_seq, int num_blocks, float scale,
                                    int dtype, void* out, int out_dtype, int partition_tokens,
                                    void* workspace, size_t workspace_bytes,
                                    int32_t* error_record, void* stream,
                                    const pa_decode_opts* opts) {
  return decode_common(q, nullptr, nullptr, k_cache, v_cache, nullptr, nullptr, block_tables,
                       seq_lens, num_seqs, num_heads, head_dim, block_size, max_blocks_per_seq,
                       num_blocks, scale, dtype, out, out_dtype, partition_tokens, workspace,
                       workspace_bytes, error_record, stream, opts);
}

extern "C" int paged_attn_decode_append(const void* q, const void* new_k, const void* new_v,
                                        void* k_cache, void* v_cache,
                                        const int32_t* block_tables, const int32_t* seq_lens,
                                        int num_seqs, int num_heads, int head_dim,
                                        int block_size, int max_blocks_per_seq, int num_blocks,
                                        float scale, int dtype, void* out, int out_dtype,
                                        int partition_tokens, void* workspace,
                                        size_t workspace_bytes, int32_t* error_record,
                                        void* stream, const pa_decode_opts* opts) {
  if (num_seqs > 0 && (!new_k || !new_v || !aligned16(new_k) || !aligned16(new_v)))
    return PA_ERR_INVALID_ARG;
  return decode_common(q, new_k, new_v, k_cache, v_cache, k_cache, v_cache, block_tables,
                       seq_lens, num_seqs, num_heads, head_dim, block_size, max_blocks_per_seq,
                       num_blocks, scale, dtype, out, out_dtype, partition_tokens, workspace,
                       workspace_bytes, error_record, stream, opts);
}

extern "C" int paged_attn_decode(const void* q, const void* k_cache, const void* v_cache,
                                 const int32_t* block_tables, const int32_t* seq_lens,
                                 int num_seqs, int num_heads, int head_dim, int block_size,
                                 int max_blocks_per_seq, int num_blocks, float scale, int dtype,
                                 void* out, int out_dtype, int partition_tokens, void* workspace,
                                 size_t workspace_bytes, int32_t* error_record, void* stream) {
  return paged_attn_decode_ex(q, k_cache, v_cache, block_tables, seq_lens, num_seqs, num_heads,
                              head_dim, block_size, max_blocks_per_seq, num_blocks, scale, dtype,
                              out, out_dtype, partition_tokens, workspace, workspace_bytes,
                              error_record, stream, nullptr);
}
