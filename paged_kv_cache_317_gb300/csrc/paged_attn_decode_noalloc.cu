// Decode attention for callers that cannot allocate device memory.
//
// paged_attn_decode needs a scratch workspace whenever a sequence may span
// more than one split-K partition, and expects the caller to allocate it.  Some
// callers can't: code that lives inside another runtime whose memory pool owns
// all device memory, a serving loop that must never block in the allocator
// (cudaMalloc / cudaFree can synchronise the whole device), or an embedded
// deployment whose device memory budget is fixed at start-up.  For them,
// paged_attn_decode_noalloc takes that scratch from a fixed array compiled into
// this library's device image, so the call allocates nothing.
//
// The array is PA_NOALLOC_SCRATCH_BYTES (32 MiB) and, once this file's device
// code is loaded on a GPU, stays resident there until the process exits.  All
// calls share the one array: calls whose kernels overlap on the GPU (different
// streams, or different host threads) race on it.
#include <cuda_runtime.h>

#include "pagedkv.h"

namespace {

static __device__ __align__(256) unsigned char g_decode_scratch[PA_NOALLOC_SCRATCH_BYTES];

// Device address of g_decode_scratch in the current context.  In host code the
// array's name is only a host-side stand-in, so the address must come from the
// runtime.  It belongs to the context the module is loaded in, not to the
// device ordinal: after cudaDeviceReset, or under another driver-API context on
// the same device, it changes.  So it is looked up on every call (a host-side
// table lookup once the module is loaded; it allocates nothing).
int scratch_address(void** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr)
    return PA_ERR_CUDA;
  *out = p;
  return PA_OK;
}

}  // namespace

extern "C" int paged_attn_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                         const int32_t* block_tables, const int32_t* seq_lens,
                                         int num_seqs, int num_heads, int head_dim,
                                         int block_size, int max_blocks_per_seq, int num_blocks,
                                         float scale, int dtype, void* out, int out_dtype,
                                         int partition_tokens, int32_t* error_record,
                                         void* stream) {
  const size_t need = paged_attn_workspace_size(num_seqs, num_heads, head_dim, block_size,
                                                max_blocks_per_seq, partition_tokens);
  if (need > PA_NOALLOC_SCRATCH_BYTES) return PA_ERR_INVALID_ARG;
  void* scratch = nullptr;
  if (need > 0) {
    const int st = scratch_address(&scratch);
    if (st != PA_OK) return st;
  }
  // The partials in the scratch are always written before they are read, so
  // nothing needs clearing between calls.
  return paged_attn_decode(q, k_cache, v_cache, block_tables, seq_lens, num_seqs, num_heads,
                           head_dim, block_size, max_blocks_per_seq, num_blocks, scale, dtype, out,
                           out_dtype, partition_tokens, scratch,
                           need > 0 ? static_cast<size_t>(PA_NOALLOC_SCRATCH_BYTES) : 0,
                           error_record, stream);
}
