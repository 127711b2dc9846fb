// paged_attn_decode_noalloc before and after cudaDeviceReset, through the C ABI
// alone.  The scratch array's device address belongs to the context the
// library's device code is loaded in; a reset destroys that context and the
// next call runs in a new one.  Each round allocates its inputs, makes a split-K
// decode through paged_attn_decode_noalloc and through paged_attn_decode with a
// caller-allocated workspace, and requires the two outputs to be identical bit
// for bit (same kernels, same partitions; only the scratch differs).
// Build: nvcc -std=c++17 -I include noalloc_after_reset.cu -L<dir> -lpagedkv
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <cstring>
#include <vector>

#include "pagedkv.h"

namespace {

constexpr int kSeqs = 8, kHeads = 4, kDim = 128, kBlock = 16, kMaxBlocks = 64;
constexpr int kBlocks = kSeqs * kMaxBlocks, kPartition = 128;

#define CUDA(call)                                                       \
  do {                                                                   \
    const cudaError_t e_ = (call);                                       \
    if (e_ != cudaSuccess) {                                             \
      std::fprintf(stderr, "%s: %s\n", #call, cudaGetErrorString(e_)); \
      return 1;                                                          \
    }                                                                    \
  } while (0)
#define CHECK(call)                                                                       \
  do {                                                                                    \
    const int st_ = (call);                                                               \
    if (st_ != 0) {                                                                       \
      std::fprintf(stderr, "%s failed: %d (%s)\n", #call, st_, pa_status_string(st_));  \
      return 1;                                                                           \
    }                                                                                     \
  } while (0)

struct Lcg {
  uint32_t s;
  uint32_t next_u32() { return s = s * 1664525u + 1013904223u; }
  float next() { return static_cast<float>(next_u32() >> 8) / 8388608.0f - 1.0f; }
};

int round_trip(int round) {
  Lcg g{0x9e3779b9u + static_cast<uint32_t>(round)};
  const size_t q_elems = static_cast<size_t>(kSeqs) * kHeads * kDim;
  const size_t cache_elems = static_cast<size_t>(kBlocks) * kHeads * kBlock * kDim;
  std::vector<__half> hq(q_elems), hk(cache_elems), hv(cache_elems);
  for (auto& x : hq) x = __float2half(g.next());
  for (auto& x : hk) x = __float2half(g.next());
  for (auto& x : hv) x = __float2half(g.next());
  // lengths 1..1024 (several 128-token partitions each); blocks handed out as a
  // stride-7 walk over the pool so the tables are scattered
  std::vector<int32_t> lens(kSeqs), tables(static_cast<size_t>(kSeqs) * kMaxBlocks, -1);
  int next = 0;
  for (int i = 0; i < kSeqs; ++i) {
    lens[i] = 1 + static_cast<int>(g.next_u32() % (kMaxBlocks * kBlock));
    const int nb = (lens[i] + kBlock - 1) / kBlock;
    for (int j = 0; j < nb; ++j) tables[i * kMaxBlocks + j] = (next++ * 7) % kBlocks;
  }

  void *q, *k, *v, *out_a, *out_b, *ws = nullptr;
  int32_t *bt, *sl;
  const size_t ws_bytes = paged_attn_workspace_size(kSeqs, kHeads, kDim, kBlock, kMaxBlocks,
                                                    kPartition);
  if (ws_bytes == 0 || ws_bytes > PA_NOALLOC_SCRATCH_BYTES) {
    std::fprintf(stderr, "unexpected workspace size %zu\n", ws_bytes);
    return 1;
  }
  CUDA(cudaMalloc(&q, q_elems * 2));
  CUDA(cudaMalloc(&k, cache_elems * 2));
  CUDA(cudaMalloc(&v, cache_elems * 2));
  CUDA(cudaMalloc(&out_a, q_elems * 4));
  CUDA(cudaMalloc(&out_b, q_elems * 4));
  CUDA(cudaMalloc(&ws, ws_bytes));
  CUDA(cudaMalloc(&bt, tables.size() * 4));
  CUDA(cudaMalloc(&sl, lens.size() * 4));
  CUDA(cudaMemcpy(q, hq.data(), q_elems * 2, cudaMemcpyHostToDevice));
  CUDA(cudaMemcpy(k, hk.data(), cache_elems * 2, cudaMemcpyHostToDevice));
  CUDA(cudaMemcpy(v, hv.data(), cache_elems * 2, cudaMemcpyHostToDevice));
  CUDA(cudaMemcpy(bt, tables.data(), tables.size() * 4, cudaMemcpyHostToDevice));
  CUDA(cudaMemcpy(sl, lens.data(), lens.size() * 4, cudaMemcpyHostToDevice));
  CUDA(cudaMemset(out_a, 0xff, q_elems * 4));   // NaN patterns: unwritten rows show up
  CUDA(cudaMemset(out_b, 0xff, q_elems * 4));

  const float scale = 0.08838834764831845f;    // 1/sqrt(128)
  CHECK(paged_attn_decode_noalloc(q, k, v, bt, sl, kSeqs, kHeads, kDim, kBlock, kMaxBlocks,
                                  kBlocks, scale, PA_F16, out_a, PA_F32, kPartition, nullptr,
                                  nullptr));
  CHECK(paged_attn_decode(q, k, v, bt, sl, kSeqs, kHeads, kDim, kBlock, kMaxBlocks, kBlocks,
                          scale, PA_F16, out_b, PA_F32, kPartition, ws, ws_bytes, nullptr,
                          nullptr));
  CUDA(cudaDeviceSynchronize());
  std::vector<float> a(q_elems), b(q_elems);
  CUDA(cudaMemcpy(a.data(), out_a, q_elems * 4, cudaMemcpyDeviceToHost));
  CUDA(cudaMemcpy(b.data(), out_b, q_elems * 4, cudaMemcpyDeviceToHost));
  for (void* p : {q, k, v, out_a, out_b, ws}) CUDA(cudaFree(p));
  CUDA(cudaFree(bt));
  CUDA(cudaFree(sl));
  if (std::memcmp(a.data(), b.data(), q_elems * 4) != 0) {
    std::fprintf(stderr, "round %d: noalloc output differs from paged_attn_decode\n", round);
    return 1;
  }
  for (float x : a)
    if (!(x == x)) {
      std::fprintf(stderr, "round %d: NaN in the output\n", round);
      return 1;
    }
  std::printf("round %d: identical (%zu floats)\n", round, q_elems);
  return 0;
}

}  // namespace

int main() {
  CUDA(cudaSetDevice(0));
  if (round_trip(0) != 0) return 1;
  CUDA(cudaDeviceReset());
  if (round_trip(1) != 0) return 1;
  std::printf("ok: noalloc matches paged_attn_decode before and after cudaDeviceReset\n");
  return 0;
}
