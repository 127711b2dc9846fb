// Decode attention over partitions that several sequences share (PagedAttention:
// zeroshotmind.com page, "Sharing a prefix without copying it": parallel samples
// and beam candidates point their block tables at the same physical blocks).
//
// The plain partition kernel streams a shared block once for every sequence
// that holds it.  Here one thread block takes one shared partition of up to 16
// sequences ("members": their tables name the same physical blocks over the
// whole partition) and reads each K/V chunk once for all of their queries.
//  * Producer warp: per 16-token chunk, looks the block up in the first
//    member's table and loads the chunk's K and V rows of its G heads into a
//    ring of S shared-memory stages with 2-D TMA boxes of 16 rows x 64 columns
//    (128-byte swizzle), so that the consumers' 8x8 matrix loads (ldmatrix)
//    hit 32 different banks.  (One 1-D bulk copy per row at a padded pitch
//    does the same with 8x as many copies, and ran at 2.8 TB/s.)
//  * One consumer warp per head: the members' queries are the 16 rows of the A
//    operand of mma.sync m16n8k16 (rows past the member count are zero).  Per
//    chunk: S = Q.K^T in fp32 (2 x D/16 MMAs), the online softmax of each row in
//    log2 units, then O += P.V with P split into a high and a low half-precision
//    part (2 x 2 x D/16 MMAs), so that P keeps about 16 significant bits and the
//    result stays well inside the fp32 path's error.
//  * Each member gets the same (m, l, acc) partial the plain kernel would write
//    for that partition, so the log-sum-exp merge combines it with the member's
//    other partitions.  A member whose only partition this is gets its output
//    row directly.
// The contraction is 16 x 16 x D per chunk and head, below the smallest tcgen05
// tile, and the kernel is bound by HBM, so the warp-level MMA is enough.
// Every wait is bounded, every index read from device memory is checked, and a
// record that breaks the rules is recorded and skipped.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <type_traits>

#include "common.cuh"
#include "decode_config.h"
#include "decode_shared.h"
#include "tma.cuh"

namespace pagedkv {
namespace {

constexpr int kChunk = 16;             // tokens per pipeline stage
constexpr int kHeader = 256;           // mbarriers (2 x kMaxRing x 8 B) + abort flag
constexpr int kAlign = 1024;           // a swizzled box must start on 1024 bytes
constexpr int kMaxRing = 8;
constexpr int kMaxG = 2;               // heads per block
constexpr int kMembers = PA_SHARE_MAX_MEMBERS;
constexpr int kRecord = PA_SHARE_RECORD_WORDS;

template <int D>
struct Geo {
  static constexpr int kGroups = D / 64;                   // 64-column groups (128 B rows)
  static constexpr int kGroupBytes = kChunk * 128;         // one TMA box: 16 rows x 128 B
  static constexpr int kTileBytes = kGroups * kGroupBytes;  // one head's K (or V) chunk
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// c += a . b for one m16n8k16 tile, fp32 accumulate.
__device__ __forceinline__ void mma(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                    uint32_t b1, BF16) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                    uint32_t b1, F16) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Two probabilities (keys k, k+1 of one row) -> packed high parts RN(x) and
// packed low parts RN(x - high), the lower key in the lower 16 bits.
__device__ __forceinline__ void split2(float x0, float x1, uint32_t& hi, uint32_t& lo, BF16) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
  const float2 hf = __bfloat1622float2(h);
  const __nv_bfloat162 l = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

__device__ __forceinline__ void split2(float x0, float x1, uint32_t& hi, uint32_t& lo, F16) {
  const __half2 h = __floats2half2_rn(x0, x1);
  const float2 hf = __half22float2(h);
  const __half2 l = __floats2half2_rn(x0 - hf.x, x1 - hf.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

// This kernel may run as a programmatic dependent of the per-sequence partition
// pass (it reads nothing that pass writes, so it starts early and fills the
// SMs the pass's last wave leaves idle).  Each block waits for that pass to
// complete before it exits, so that whatever follows this kernel in the stream
// or graph (the merge) also follows the partition pass.  Without a
// prerequisite grid the wait returns at once.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ uint32_t ld_pair(const char* base, int seq, int num_heads, int h,
                                            int d, int row_bytes) {
  if (seq < 0) return 0u;
  return __ldg(reinterpret_cast<const uint32_t*>(
      base + (static_cast<size_t>(seq) * num_heads + h) * row_bytes + d * 2));
}

template <class Tag, int D>
__global__ void __launch_bounds__((kMaxG + 1) * 32)
    paged_attn_shared_kernel(const __grid_constant__ CUtensorMap tm_k,
                             const __grid_constant__ CUtensorMap tm_v, const SharedParams p) {
  using Gm = Geo<D>;
  constexpr int kRowBytes = D * 2;
  extern __shared__ __align__(128) uint8_t smem[];
  const int G = p.heads_per_cta;
  const int S = p.stages;
  const int hg = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int32_t* rec = p.records + static_cast<size_t>(blockIdx.y) * kRecord;

  // Check the record (every thread reaches the same verdict): partition in
  // range, 1..16 members, each a valid sequence whose length covers the whole
  // partition (and, with a fused append, the appended token lies past it).
  const int part = __ldg(rec);
  const int m = __ldg(rec + 1);
  const int cap = p.max_blocks * p.block_size;
  bool bad = part < 0 || part >= p.num_partitions || m < 1 || m > kMembers;
  int bad_value = part < 0 || part >= p.num_partitions ? part : m;
  if (!bad) {
    const long long need = static_cast<long long>(part + 1) * p.partition_tokens +
                           (p.fused_append ? 1 : 0);
    for (int i = 0; i < m && !bad; ++i) {
      const int s = __ldg(rec + 2 + i);
      if (s < 0 || s >= p.num_seqs) {
        bad = true;
        bad_value = s;
      } else {
        const int L = __ldg(p.seq_lens + s);
        if (L < need || L > cap) {
          bad = true;
          bad_value = s;
        }
      }
    }
  }
  if (bad) {
    if (threadIdx.x == 0 && hg == 0) report_error(p.err, PA_ERR_BAD_SEQ_LEN, blockIdx.y, bad_value);
    grid_dependency_wait();
    return;
  }
  const int first = __ldg(rec + 2);
  const int tok_begin = part * p.partition_tokens;
  const int nchunks = p.partition_tokens / kChunk;

  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kMaxRing;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 2 * kMaxRing * 8);
  const uint32_t smem_base = smem_addr(smem);
  uint8_t* ring = smem + (((smem_base + kHeader + kAlign - 1) & ~uint32_t(kAlign - 1)) - smem_base);
  const int stage_bytes = G * 2 * Gm::kTileBytes;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], G);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  int issued = 0;  // producer lane 0 only: chunks whose copies were issued
  if (warp == G) {
    // ------------------------------------------------------------ producer
    const int32_t* table = p.block_tables + static_cast<size_t>(first) * p.max_blocks;
    const int h0 = hg * G;
    bool stop = false;
    for (int c0 = 0; c0 < nchunks && !stop; c0 += 32) {
      int blk = 0;
      if (c0 + lane < nchunks) {
        const int tok = tok_begin + (c0 + lane) * kChunk;
        blk = __ldg(table + tok / p.block_size);
        if (static_cast<unsigned>(blk) >= static_cast<unsigned>(p.num_blocks)) {
          report_error(p.err, PA_ERR_BAD_BLOCK, first, blk);
          blk = 0;
        }
      }
      const int n = min(32, nchunks - c0);
      for (int j = 0; j < n; ++j) {
        const int b = __shfl_sync(kFullMask, blk, j);
        const int chunk = c0 + j;
        const int s = chunk % S;
        if (lane == 0) {
          bool ok = true;
          if (chunk >= S) ok = mbar_wait_bounded(&empty[s], ((chunk / S) - 1) & 1);
          if (!ok) {
            *abort_flag = 1;
            report_error(p.err, PA_ERR_TIMEOUT, first, chunk);
          } else {
            mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(stage_bytes));
            // the chunk's rows of (block b, head h) are rows y .. y + 15 of the
            // cache viewed as [num_blocks * H * bs][D]
            const int row0 = (tok_begin + chunk * kChunk) % p.block_size;
            uint8_t* dst = ring + s * stage_bytes;
            for (int w = 0; w < G; ++w) {
              const int y = (b * p.num_heads + h0 + w) * p.block_size + row0;
#pragma unroll
              for (int cg = 0; cg < Gm::kGroups; ++cg) {
                tma_load_2d(dst + (w * 2) * Gm::kTileBytes + cg * Gm::kGroupBytes, &tm_k, cg * 64,
                            y, &full[s]);
                tma_load_2d(dst + (w * 2 + 1) * Gm::kTileBytes + cg * Gm::kGroupBytes, &tm_v,
                            cg * 64, y, &full[s]);
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
    const int g = lane >> 2, tq = lane & 3;
    const int seq_lo = g < m ? __ldg(rec + 2 + g) : -1;          // member of row g
    const int seq_hi = g + 8 < m ? __ldg(rec + 2 + g + 8) : -1;  // member of row g + 8
    const char* qb = static_cast<const char*>(p.q);
    uint32_t qa[D / 16][4];
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const int d0 = kk * 16 + 2 * tq;
      qa[kk][0] = ld_pair(qb, seq_lo, p.num_heads, h, d0, kRowBytes);
      qa[kk][1] = ld_pair(qb, seq_hi, p.num_heads, h, d0, kRowBytes);
      qa[kk][2] = ld_pair(qb, seq_lo, p.num_heads, h, d0 + 8, kRowBytes);
      qa[kk][3] = ld_pair(qb, seq_hi, p.num_heads, h, d0 + 8, kRowBytes);
    }
    float o[D / 8][4];
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
    float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;

    // ldmatrix row addresses of this lane: lanes 8i..8i+7 name the rows of
    // matrix i.  K (B operand of S, no transpose): matrices (tokens 0-7, d+0..7),
    // (0-7, d+8..15), (8-15, d+0..7), (8-15, d+8..15).  V (B operand of P.V,
    // transposed): (tokens 0-7, d+0..7), (8-15, d+0..7), (0-7, d+8..15), (8-15, d+8..15).
    // Token t's 16-byte chunk c of a 64-column group sits at t * 128 + (c ^ (t & 7)) * 16,
    // and t & 7 is this lane's r8.
    const int mi = lane >> 3, r8 = lane & 7;
    const uint32_t k_row = static_cast<uint32_t>(((mi >> 1) * 8 + r8) * 128);
    const uint32_t v_row = static_cast<uint32_t>(((mi & 1) * 8 + r8) * 128);
    const int k_half = mi & 1, v_half = mi >> 1;
    const uint32_t ring_addr = smem_addr(ring);

    for (int chunk = 0; chunk < nchunks; ++chunk) {
      const int s = chunk % S;
      const bool ok = __all_sync(kFullMask, mbar_wait_bounded(&full[s], (chunk / S) & 1));
      if (!ok) {
        if (lane == 0) {
          *abort_flag = 1;
          report_error(p.err, PA_ERR_TIMEOUT, first, chunk);
        }
        break;
      }
      const uint32_t kt = ring_addr + s * stage_bytes + warp * 2 * Gm::kTileBytes;
      const uint32_t vt = kt + Gm::kTileBytes;

      // scores of the 16 tokens: sc[j] covers tokens 8j..8j+7
      float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        uint32_t b[4];
        const int c = ((kk & 3) << 1) | k_half;
        ldsm_x4(kt + (kk >> 2) * Gm::kGroupBytes + k_row + ((c ^ r8) << 4), b);
        mma(sc[0], qa[kk], b[0], b[1], Tag{});
        mma(sc[1], qa[kk], b[2], b[3], Tag{});
      }
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) sc[j][e] *= p.qscale;

      // online softmax of rows g (elements 0, 1) and g + 8 (elements 2, 3); a
      // row's 16 scores sit on the four lanes of a quad
      float cm_lo = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
      float cm_hi = fmaxf(fmaxf(sc[0][2], sc[0][3]), fmaxf(sc[1][2], sc[1][3]));
      cm_lo = fmaxf(cm_lo, __shfl_xor_sync(kFullMask, cm_lo, 1));
      cm_hi = fmaxf(cm_hi, __shfl_xor_sync(kFullMask, cm_hi, 1));
      cm_lo = fmaxf(cm_lo, __shfl_xor_sync(kFullMask, cm_lo, 2));
      cm_hi = fmaxf(cm_hi, __shfl_xor_sync(kFullMask, cm_hi, 2));
      const float mn_lo = fmaxf(m_lo, cm_lo), mn_hi = fmaxf(m_hi, cm_hi);
      const float a_lo = exp2f(m_lo - mn_lo), a_hi = exp2f(m_hi - mn_hi);
      float pr[2][4];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        pr[j][0] = exp2f(sc[j][0] - mn_lo);
        pr[j][1] = exp2f(sc[j][1] - mn_lo);
        pr[j][2] = exp2f(sc[j][2] - mn_hi);
        pr[j][3] = exp2f(sc[j][3] - mn_hi);
      }
      l_lo = fmaf(l_lo, a_lo, (pr[0][0] + pr[0][1]) + (pr[1][0] + pr[1][1]));
      l_hi = fmaf(l_hi, a_hi, (pr[0][2] + pr[0][3]) + (pr[1][2] + pr[1][3]));
      if (__any_sync(kFullMask, a_lo != 1.f || a_hi != 1.f)) {
#pragma unroll
        for (int nt = 0; nt < D / 8; ++nt) {
          o[nt][0] *= a_lo;
          o[nt][1] *= a_lo;
          o[nt][2] *= a_hi;
          o[nt][3] *= a_hi;
        }
      }
      m_lo = mn_lo;
      m_hi = mn_hi;

      // P as the A operand (keys 0..15 along k), in high and low parts
      uint32_t ph[4], pl[4];
      split2(pr[0][0], pr[0][1], ph[0], pl[0], Tag{});
      split2(pr[0][2], pr[0][3], ph[1], pl[1], Tag{});
      split2(pr[1][0], pr[1][1], ph[2], pl[2], Tag{});
      split2(pr[1][2], pr[1][3], ph[3], pl[3], Tag{});
#pragma unroll
      for (int dd = 0; dd < D / 16; ++dd) {
        uint32_t b[4];
        const int c = ((dd & 3) << 1) | v_half;
        ldsm_x4_trans(vt + (dd >> 2) * Gm::kGroupBytes + v_row + ((c ^ r8) << 4), b);
        mma(o[2 * dd], ph, b[0], b[1], Tag{});
        mma(o[2 * dd], pl, b[0], b[1], Tag{});
        mma(o[2 * dd + 1], ph, b[2], b[3], Tag{});
        mma(o[2 * dd + 1], pl, b[2], b[3], Tag{});
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      if (__shfl_sync(kFullMask, *abort_flag, 0)) break;
    }

    l_lo += __shfl_xor_sync(kFullMask, l_lo, 1);
    l_hi += __shfl_xor_sync(kFullMask, l_hi, 1);
    l_lo += __shfl_xor_sync(kFullMask, l_lo, 2);
    l_hi += __shfl_xor_sync(kFullMask, l_hi, 2);
    if (!*abort_flag) {
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int seq = half ? seq_hi : seq_lo;
        if (seq < 0) continue;
        const float mrow = half ? m_hi : m_lo, lrow = half ? l_hi : l_lo;
        const int L = __ldg(p.seq_lens + seq);
        const int nparts = (L + p.partition_tokens - 1) / p.partition_tokens;
        if (nparts == 1) {
          const float inv = lrow > 0.f ? 1.f / lrow : 0.f;
#pragma unroll
          for (int nt = 0; nt < D / 8; ++nt) {
            const float v2[2] = {o[nt][2 * half] * inv, o[nt][2 * half + 1] * inv};
            store_out<2>(p.out, (static_cast<size_t>(seq) * p.num_heads + h) * D + nt * 8 + 2 * tq,
                         v2, p.out_dtype);
          }
        } else {
          const size_t row =
              (static_cast<size_t>(seq) * p.num_heads + h) * p.num_partitions + part;
          float* dst = p.ws_acc + row * D + 2 * tq;
#pragma unroll
          for (int nt = 0; nt < D / 8; ++nt)
            *reinterpret_cast<float2*>(dst + nt * 8) =
                make_float2(o[nt][2 * half], o[nt][2 * half + 1]);
          if (tq == 0) p.ws_ml[row] = make_float2(mrow, lrow);
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
  grid_dependency_wait();
}

template <class Tag, int D>
cudaError_t ensure_shared_smem_attr(int device) {
  static std::atomic<uint64_t> done{0};
  const uint64_t bit = device < 64 ? (1ull << device) : 0;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  int optin = 0;
  cudaError_t e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(paged_attn_shared_kernel<Tag, D>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

template <class Tag, int D>
int launch_t(const SharedParams& p, bool programmatic, cudaStream_t stream) {
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return PA_ERR_CUDA;
  if (ensure_shared_smem_attr<Tag, D>(device) != cudaSuccess) return PA_ERR_CUDA;
  // the caches as [num_blocks * H * bs][D] row-major, boxes of 16 rows x 64 columns
  const unsigned long long rows =
      static_cast<unsigned long long>(p.num_blocks) * p.num_heads * p.block_size;
  if (rows >= (1ull << 31)) return PA_ERR_UNSUPPORTED;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), rows};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(D) * 2};
  const cuuint32_t box[2] = {64, kChunk};
  CUtensorMap tk, tv;
  const bool bf16 = std::is_same<Tag, BF16>::value;
  if (!encode_tensor_map(&tk, bf16, p.k_cache, 2, dims, strides, box) ||
      !encode_tensor_map(&tv, bf16, p.v_cache, 2, dims, strides, box))
    return PA_ERR_CUDA;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(p.num_heads / p.heads_per_cta, p.num_records);
  cfg.blockDim = dim3((p.heads_per_cta + 1) * 32);
  cfg.dynamicSmemBytes = shared_kernel_smem_bytes(D, p.heads_per_cta, p.stages);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = programmatic ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, paged_attn_shared_kernel<Tag, D>, tk, tv, p) != cudaSuccess)
    return PA_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace

size_t shared_kernel_smem_bytes(int head_dim, int heads_per_cta, int stages) {
  return kHeader + kAlign + static_cast<size_t>(stages) * heads_per_cta * 2 * kChunk * head_dim * 2;
}

int launch_shared_partitions(const SharedParams& p, int dtype, int head_dim, bool programmatic,
                             cudaStream_t stream) {
  if (p.num_records == 0) return PA_OK;
  if (p.num_records < 0 || p.num_records > 65535 || p.heads_per_cta < 1 ||
      p.heads_per_cta > kMaxG || p.num_heads % p.heads_per_cta != 0 || p.stages < 2 ||
      p.stages > kMaxRing || p.partition_tokens % kChunk != 0 || p.block_size % kChunk != 0)
    return PA_ERR_INVALID_ARG;
  if (shared_kernel_smem_bytes(head_dim, p.heads_per_cta, p.stages) > 227 * 1024)
    return PA_ERR_INVALID_ARG;
  const bool bf16 = dtype == PA_BF16;
  switch (head_dim) {
    case 64:
      return bf16 ? launch_t<BF16, 64>(p, programmatic, stream)
                  : launch_t<F16, 64>(p, programmatic, stream);
    case 128:
      return bf16 ? launch_t<BF16, 128>(p, programmatic, stream)
                  : launch_t<F16, 128>(p, programmatic, stream);
    case 256:
      return bf16 ? launch_t<BF16, 256>(p, programmatic, stream)
                  : launch_t<F16, 256>(p, programmatic, stream);
    default: return PA_ERR_UNSUPPORTED;
  }
}

}  // namespace pagedkv
