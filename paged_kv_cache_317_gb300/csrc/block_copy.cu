// Copy-on-write block copy (PagedAttention, zeroshotmind.com page, "Sharing a
// prefix without copying it": a sequence about to write into a shared block
// gets a private copy of just that block).
//
// Grid: x = 16 KB piece of a block, y = pair, z = (layer, K or V).  Each thread
// issues four independent 16-byte loads before its four stores, so a block of
// 256 threads keeps 16 KB in flight.  A block's bytes in the [B][H][bs][D]
// layout are contiguous, so every piece is one straight run.
#include <cuda_runtime.h>

#include "common.cuh"

namespace pagedkv {
namespace {

constexpr int kMaxLayers = 128;
constexpr int kThreads = 256;
constexpr int kUnroll = 4;
constexpr int kPieceVecs = kThreads * kUnroll;  // 16-byte vectors per grid-x piece

struct LayerPtrs {
  uint4* k[kMaxLayers];
  uint4* v[kMaxLayers];
};

__global__ void __launch_bounds__(kThreads)
    block_copy_kernel(const LayerPtrs layers, const int64_t* __restrict__ pairs,
                      long long block_vecs, int num_blocks, int32_t* err) {
  const int pair = blockIdx.y;
  const int layer = blockIdx.z >> 1;
  const long long src = __ldg(pairs + 2 * pair);
  const long long dst = __ldg(pairs + 2 * pair + 1);
  if (src == -1 && dst == -1) return;  // padding
  if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
    if (blockIdx.x == 0 && blockIdx.z == 0 && threadIdx.x == 0)
      report_error(err, PA_ERR_BAD_BLOCK, pair, (src < 0 || src >= num_blocks) ? src : dst);
    return;
  }
  uint4* base = (blockIdx.z & 1) ? layers.v[layer] : layers.k[layer];
  const uint4* s = base + src * block_vecs;
  uint4* d = base + dst * block_vecs;
  const long long first = static_cast<long long>(blockIdx.x) * kPieceVecs + threadIdx.x;
  uint4 r[kUnroll];
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) {
    const long long idx = first + u * kThreads;
    if (idx < block_vecs) r[u] = s[idx];
  }
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) {
    const long long idx = first + u * kThreads;
    if (idx < block_vecs) d[idx] = r[u];
  }
}

}  // namespace
}  // namespace pagedkv

using namespace pagedkv;

extern "C" int block_copy(void* const* k_caches, void* const* v_caches, int num_layers,
                          const int64_t* pairs, int num_pairs, int num_heads, int head_dim,
                          int block_size, int num_blocks, int dtype, int32_t* error_record,
                          void* stream) {
  NvtxRange range("block_copy");
  if (num_layers <= 0 || num_layers > kMaxLayers || num_pairs < 0 || num_heads <= 0 ||
      head_dim <= 0 || block_size <= 0 || num_blocks <= 0)
    return PA_ERR_INVALID_ARG;
  if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
  if (num_pairs == 0) return PA_OK;
  if (num_pairs > 65535) return PA_ERR_INVALID_ARG;
  if (!k_caches || !v_caches || !pairs) return PA_ERR_INVALID_ARG;
  const long long block_bytes = static_cast<long long>(num_heads) * block_size * head_dim * 2;
  if (block_bytes % 16 != 0) return PA_ERR_UNSUPPORTED;
  LayerPtrs lp{};
  for (int l = 0; l < num_layers; ++l) {
    if (!k_caches[l] || !v_caches[l] || !aligned16(k_caches[l]) || !aligned16(v_caches[l]))
      return PA_ERR_INVALID_ARG;
    lp.k[l] = static_cast<uint4*>(k_caches[l]);
    lp.v[l] = static_cast<uint4*>(v_caches[l]);
  }
  const long long block_vecs = block_bytes / 16;
  dim3 grid(static_cast<unsigned>((block_vecs + kPieceVecs - 1) / kPieceVecs), num_pairs,
            2 * num_layers);
  block_copy_kernel<<<grid, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      lp, pairs, block_vecs, num_blocks, error_record);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
