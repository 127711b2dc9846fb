// KV append into slot-mapped blocks (PagedAttention, zeroshotmind.com page,
// "Paging the cache": a sequence's blocks are filled as it grows).
//
// Token t's key/value rows for every head are bit-copied to slot
// slot_mapping[t] of the [B][H][bs][D] caches.  One thread moves one 16-byte
// piece of a K row and the matching piece of the V row; consecutive threads
// take consecutive pieces, so both the reads of k/v and the writes of each
// cache row are fully coalesced.  The kernel is latency-bound at decode sizes
// (a few MB), so the grid simply covers the work once.
#include <cuda_runtime.h>

#include "common.cuh"

namespace pagedkv {
namespace {

__global__ void __launch_bounds__(256)
    kv_append_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                     const int64_t* __restrict__ slots, long long total, int pieces_per_token,
                     int pieces_per_row, int num_heads, int block_size, long long capacity,
                     uint4* __restrict__ k_cache, uint4* __restrict__ v_cache, int32_t* err) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += stride) {
    const long long t = i / pieces_per_token;
    const int rem = static_cast<int>(i - t * pieces_per_token);
    const int h = rem / pieces_per_row;
    const int x = rem - h * pieces_per_row;
    const long long slot = __ldg(slots + t);
    if (slot < 0) continue;  // padding token
    if (slot >= capacity) {
      if (rem == 0) report_error(err, PA_ERR_BAD_SLOT, t, slot);
      continue;
    }
    const long long blk = slot / block_size;
    const long long row = slot - blk * block_size;
    const long long dst = ((blk * num_heads + h) * block_size + row) * pieces_per_row + x;
    const uint4 kv = __ldg(k + i);
    const uint4 vv = __ldg(v + i);
    k_cache[dst] = kv;
    v_cache[dst] = vv;
  }
}

}  // namespace
}  // namespace pagedkv

using namespace pagedkv;

extern "C" int kv_cache_append(const void* k, const void* v, const int64_t* slot_mapping,
                               int num_tokens, void* k_cache, void* v_cache, int num_heads,
                               int head_dim, int block_size, int num_blocks, int dtype,
                               int32_t* error_record, void* stream) {
  NvtxRange range("kv_cache_append");
  if (num_tokens < 0 || num_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks <= 0)
    return PA_ERR_INVALID_ARG;
  if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
  if (head_dim % 8 != 0) return PA_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PA_OK;
  if (!k || !v || !slot_mapping || !k_cache || !v_cache) return PA_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache))
    return PA_ERR_INVALID_ARG;
  const int pieces_per_row = head_dim * 2 / 16;
  const int pieces_per_token = pieces_per_row * num_heads;
  const long long total = static_cast<long long>(num_tokens) * pieces_per_token;
  const long long capacity = static_cast<long long>(num_blocks) * block_size;
  const long long blocks_needed = (total + 255) / 256;
  const unsigned grid = static_cast<unsigned>(blocks_needed < 152 * 64 ? blocks_needed : 152 * 64);
  kv_append_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(k), static_cast<const uint4*>(v), slot_mapping, total,
      pieces_per_token, pieces_per_row, num_heads, block_size, capacity,
      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), error_record);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
