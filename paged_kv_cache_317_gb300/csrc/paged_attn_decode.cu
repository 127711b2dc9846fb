// Decode attention through a block table (PagedAttention: phantomic12.github.io
// note, method paragraph; zeroshotmind.com page, "Block tables: logical order,
// physical scatter"): the log-sum-exp merge of split-K partials and the host
// side of paged_attn_decode / _ex / _append (argument checks, launch shapes,
// the order of the partition pass, the shared-partition pass and the merge).
// The partition kernel itself is in decode_partition.cuh.
#include <cuda_runtime.h>

#include <cmath>

#include "common.cuh"
#include "decode_config.h"
#include "decode_partition.cuh"
#include "decode_shared.h"

namespace pagedkv {
namespace {

// One warp per (sequence, head): out = sum_p 2^(m_p - M) acc_p / sum_p 2^(m_p - M) l_p,
// over the sequence's partitions and, for a sequence whose partition was split by
// a prefix record, its tail row.
struct MergeParams {
  const int32_t* seq_lens;
  const float* ws_acc;
  const float2* ws_ml;
  const int32_t* tail_start;  // optional [N]
  const float* ws_tail_acc;   // [N * H][D]
  const float2* ws_tail_ml;   // [N * H]
  int32_t* err;
  void* out;
  int num_seqs, num_heads, capacity, partition_tokens, num_partitions, out_dtype;
};

template <int D>
__global__ void __launch_bounds__(256) paged_attn_merge_kernel(const MergeParams p) {
  constexpr int DPL = D / 32;  // dims per lane
  // Launched as a programmatic dependent of the partition pass (which completes
  // only after the pass over shared partitions, if any): wait until that grid
  // has completed and its writes are visible.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // The next decode call's first kernel waits for this one to complete before
  // it touches memory: let it be placed while this grid runs.  Not before the
  // wait above: blocks of later calls placed that early would sit on SM slots
  // the partition pass still needs.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int gw = static_cast<int>((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (gw >= p.num_seqs * p.num_heads) return;
  const int seq = gw / p.num_heads;
  int L = p.seq_lens[seq];
  L = L < 0 ? 0 : (L > p.capacity ? p.capacity : L);
  const int nparts = L > 0 ? (L + p.partition_tokens - 1) / p.partition_tokens : 1;
  // a tail row, when tail_start names a split inside the sequence (partition
  // pass: the tokens from it to its partition's end)
  bool tail = false;
  if (p.tail_start != nullptr) {
    const int ts = __ldg(p.tail_start + seq);
    if (ts >= 0) {
      tail = ts < L && ts % 16 == 0 && ts % p.partition_tokens != 0;
      if (!tail && lane == 0 && gw % p.num_heads == 0)
        report_error(p.err, PA_ERR_BAD_SEQ_LEN, seq, ts);
    }
  }
  if (nparts <= 1 && !tail) return;  // the partition pass wrote this row directly
  const size_t row0 = static_cast<size_t>(gw) * p.num_partitions;
  const int n = nparts + (tail ? 1 : 0);  // partials: the partitions, then the tail row
  auto ml_of = [&](int i) { return i < nparts ? p.ws_ml[row0 + i] : p.ws_tail_ml[gw]; };
  auto acc_of = [&](int i) {
    return i < nparts ? p.ws_acc + (row0 + i) * D : p.ws_tail_acc + static_cast<size_t>(gw) * D;
  };

  float o[DPL];
#pragma unroll
  for (int j = 0; j < DPL; ++j) o[j] = 0.f;
  float M = -INFINITY, lt = 0.f;
  if (n <= 32) {
    // Lane i holds partial i's (m, l): one load for all of them, weights by
    // shuffle, and the partials' rows loaded four at a time so that their
    // latencies overlap.
    const float2 ml = lane < n ? ml_of(lane) : make_float2(-INFINITY, 0.f);
    M = ml.x;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(kFullMask, M, off));
    if (M != -INFINITY) {
      const float w = lane < n ? exp2f(ml.x - M) : 0.f;
      lt = w * ml.y;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) lt += __shfl_xor_sync(kFullMask, lt, off);
      for (int i0 = 0; i0 < n; i0 += 4) {
        float a[4][DPL];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int i = min(i0 + u, n - 1);  // repeats are weighted 0 below
          const float* src = acc_of(i) + lane * DPL;
#pragma unroll
          for (int j = 0; j < DPL; ++j) a[u][j] = src[j];
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float wu = __shfl_sync(kFullMask, w, min(i0 + u, 31));
          const float wi = i0 + u < n ? wu : 0.f;
#pragma unroll
          for (int j = 0; j < DPL; ++j) o[j] = fmaf(wi, a[u][j], o[j]);
        }
      }
    }
  } else {
    for (int i = lane; i < n; i += 32) M = fmaxf(M, ml_of(i).x);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(kFullMask, M, off));
    if (M != -INFINITY) {
      for (int i = lane; i < n; i += 32) {
        const float2 ml = ml_of(i);
        lt = fmaf(exp2f(ml.x - M), ml.y, lt);
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) lt += __shfl_xor_sync(kFullMask, lt, off);
      for (int i = 0; i < n; ++i) {
        const float w = exp2f(ml_of(i).x - M);
        const float* a = acc_of(i) + lane * DPL;
#pragma unroll
        for (int j = 0; j < DPL; ++j) o[j] = fmaf(w, a[j], o[j]);
      }
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

// With tail rows: max(P, 1) partition rows per (sequence, head), then (from a
// 256-byte boundary, so that the tail partials keep the alignment of their
// 16-byte stores) one tail row each.
size_t tail_offset_for(int num_seqs, int num_heads, int head_dim, int P) {
  const size_t rows = static_cast<size_t>(num_seqs) * num_heads * (P > 1 ? P : 1);
  const size_t main = rows * head_dim * sizeof(float) + rows * sizeof(float2);
  return (main + 255) / 256 * 256;
}
size_t workspace_bytes_tails(int num_seqs, int num_heads, int head_dim, int P) {
  const size_t rows = static_cast<size_t>(num_seqs) * num_heads;
  return tail_offset_for(num_seqs, num_heads, head_dim, P) + rows * head_dim * sizeof(float) +
         rows * sizeof(float2);
}

int resolve_partition(int partition_tokens) {
  return partition_tokens <= 0 ? kDefaultPartition : partition_tokens;
}

// Opt-in shared memory above the 48 KB default.  The attribute belongs to the
// module loaded in the current context and is lost with it (cudaDeviceReset,
// another driver-API context), so it is set on every launch that needs it, to
// the device's opt-in maximum (concurrent callers then never lower it for one
// another); a launch within the default sets nothing.
template <class Tag, int D>
cudaError_t ensure_smem_attr(int device, size_t smem) {
  if (smem <= 48 * 1024) return cudaSuccess;
  int optin = 0;
  cudaError_t e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(paged_attn_partition_kernel<Tag, D>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
}

template <class Tag, int D>
int launch(const DecodeParams& p, int num_seqs, int phases, size_t smem,
           const SharedParams* shared, int dtype, cudaStream_t stream) {
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return PA_ERR_CUDA;
  if (phases & 1) {
    // The pass over shared partitions (if any) first: its blocks are long and of
    // equal length, and trigger their dependents when they start.  The
    // per-sequence partition pass follows as a programmatic dependent, so its
    // blocks (longest first, then ever shorter) fill the SMs the shared pass's
    // last wave leaves idle.  The two write disjoint partials; the first block of
    // the second pass waits for the first pass to complete before it exits, so
    // the merge after it follows both.
    if (shared != nullptr) {
      const int st = launch_shared_partitions(*shared, dtype, D, stream);
      if (st != PA_OK) return st;
    }
    if (ensure_smem_attr<Tag, D>(device, smem) != cudaSuccess) return PA_ERR_CUDA;
    dim3 grid(p.num_heads / p.heads_per_cta, p.num_partitions, num_seqs);
    if (p.work_items != nullptr) grid = dim3(p.num_heads / p.heads_per_cta, p.num_work_items, 1);
    dim3 block((p.heads_per_cta + 1) * 32);
    if (grid.y > 0) {
      // A programmatic dependent of the kernel before it: the shared-partition
      // pass, or (as the call's first kernel, which then waits for it before
      // touching memory) whatever precedes the call on the stream.
      DecodeParams q = p;
      q.wait_first = shared == nullptr ? 1 : 0;
      cudaLaunchConfig_t cfg{};
      cfg.gridDim = grid;
      cfg.blockDim = block;
      cfg.dynamicSmemBytes = smem;
      cfg.stream = stream;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[0].val.programmaticStreamSerializationAllowed = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      if (cudaLaunchKernelEx(&cfg, paged_attn_partition_kernel<Tag, D>, q) != cudaSuccess)
        return PA_ERR_CUDA;
      if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;
    }
  }
  if ((phases & 2) && (p.num_partitions > 1 || p.tail_start != nullptr)) {
    MergeParams mp{p.seq_lens, p.ws_acc, p.ws_ml, p.tail_start, p.ws_tail_acc, p.ws_tail_ml,
                   p.err, p.out, num_seqs, p.num_heads, p.max_blocks * p.block_size,
                   p.partition_tokens, p.num_partitions, p.out_dtype};
    const long long warps = static_cast<long long>(num_seqs) * p.num_heads;
    // A programmatic dependent of the pass before it: its blocks are placed while
    // that pass drains and wait (griddepcontrol.wait) for it before reading.
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>((warps + 7) / 8));
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, paged_attn_merge_kernel<D>, mp) != cudaSuccess) return PA_ERR_CUDA;
    if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;
  }
  return PA_OK;
}

}  // namespace
}  // namespace pagedkv

using namespace pagedkv;

extern "C" size_t paged_attn_workspace_size_tails(int num_seqs, int num_heads, int head_dim,
                                                  int block_size, int max_blocks_per_seq,
                                                  int partition_tokens) {
  if (num_seqs <= 0 || num_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
      max_blocks_per_seq <= 0)
    return 0;
  const int pt = resolve_partition(partition_tokens);
  const long long cap = static_cast<long long>(max_blocks_per_seq) * block_size;
  if (cap > (1ll << 30)) return 0;
  return workspace_bytes_tails(num_seqs, num_heads, head_dim,
                               num_partitions_for(static_cast<int>(cap), pt));
}

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
  if (block_size % 16 != 0 && block_size != 8) return PA_ERR_UNSUPPORTED;
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
  const int32_t* tail_start = opts ? opts->tail_start : nullptr;
  const size_t need = tail_start ? workspace_bytes_tails(num_seqs, num_heads, head_dim, P)
                                 : workspace_bytes_for(num_seqs, num_heads, head_dim, P);
  if (need > 0 && (!workspace || workspace_bytes < need || !aligned16(workspace)))
    return PA_ERR_INVALID_ARG;

  DecodeParams p{};
  p.q = q;
  p.seq_order = opts ? opts->seq_order : nullptr;
  p.early_inputs = (opts && opts->early_inputs) ? 1 : 0;
  p.item_count = opts ? opts->counts : nullptr;
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
                                             static_cast<size_t>(num_seqs) * num_heads *
                                                 (P > 1 ? P : 1) * head_dim * sizeof(float))
                 : nullptr;
  p.tail_start = tail_start;
  if (tail_start) {
    char* t = static_cast<char*>(workspace) + tail_offset_for(num_seqs, num_heads, head_dim, P);
    p.ws_tail_acc = reinterpret_cast<float*>(t);
    p.ws_tail_ml = reinterpret_cast<float2*>(
        t + static_cast<size_t>(num_seqs) * num_heads * head_dim * sizeof(float));
  }
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
    sp.tail_start = tail_start;
    sp.record_count = opts->counts ? opts->counts + 1 : nullptr;
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
    // At least a 3-deep ring: each block streams a whole partition, and one chunk
    // more in flight outweighs the fewer blocks per SM (sampling decode on
    // GB300: 306.7 -> 303.6 us; 4 stages 304.6, 6 stages 314.8)
    const int shared_stages = S > 3 ? S : 3;
    sp.stages = shared_kernel_smem_bytes(head_dim, sp.heads_per_cta, shared_stages) <= 227 * 1024
                    ? shared_stages
                    : 2;
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
