// Decode attention over partitions that several sequences share (PagedAttention:
// zeroshotmind.com page, "Sharing a prefix without copying it": parallel samples
// and beam candidates point their block tables at the same physical blocks).
//
// The plain partition kernel streams a shared block once for every sequence
// that holds it.  Here one thread block takes one shared partition of up to 8
// sequences ("members": their tables name the same physical blocks over the
// whole partition) and reads each K/V chunk once for all of their queries.
//  * Producer warp: per 16-token chunk, looks the block up in the first
//    member's table and loads the chunk's K and V rows of its G heads into a
//    ring of S shared-memory stages with 2-D TMA boxes of 16 rows x 64 columns
//    (128-byte swizzle), so that the consumers' 8x8 matrix loads (ldmatrix)
//    hit 32 different banks.  (One 1-D bulk copy per row at a padded pitch
//    does the same with 8x as many copies, and ran at 2.8 TB/s.)
//  * One consumer warp per head, on mma.sync m16n8k16 with the chunk's 16
//    tokens as the M rows and the (up to 8) members as the N columns: S^T =
//    K.Q^T in fp32 (D/16 MMAs per chunk), the online softmax of each member's
//    column in log2 units, then O^T += V^T.P^T with P split into a high and a
//    low half-precision part (2 x D/16 MMAs; an 8x8 register transpose turns
//    P's accumulator layout into the B operand), so that P keeps about 16
//    significant bits and the result stays well inside the fp32 path's error.
//    (Members as the 16 M rows instead take twice the MMAs and registers for
//    the <= 8 members that forked samples and beams have; both run at the
//    same speed on GB300, where this pass is bound by memory latency and the
//    last wave of its equal-length blocks, not by the tensor pipe.)
//  * Each member gets the same (m, l, acc) partial the plain kernel would write
//    for that partition, so the log-sum-exp merge combines it with the member's
//    other partitions.  A member whose only partition this is gets its output
//    row directly.
// The contraction is 16 x 8 x D per chunk and head, below the smallest tcgen05
// tile, and the kernel is bound by HBM, so the warp-level MMA is enough.
// Every wait is bounded, every index read from device memory is checked, and a
// record that breaks the rules is recorded and skipped.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

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

// Transpose of an 8x8 matrix of 16-bit values held one row pair per lane
// (lane 4 r + c holds elements (r, 2 c) and (r, 2 c + 1)).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// One fp32 value stored as `dtype` at element `elem` of `out`.
__device__ __forceinline__ void store_one(void* out, size_t elem, float v, int dtype) {
  if (dtype == PA_F32) {
    static_cast<float*>(out)[elem] = v;
  } else if (dtype == PA_BF16) {
    static_cast<__nv_bfloat16*>(out)[elem] = __float2bfloat16_rn(v);
  } else {
    static_cast<__half*>(out)[elem] = __float2half_rn(v);
  }
}

__device__ __forceinline__ uint32_t ld_pair(const char* base, int seq, int num_heads, int h,
                                            int d, int row_bytes) {
  if (seq < 0) return 0u;
  return __ldg(reinterpret_cast<const uint32_t*>(
      base + (static_cast<size_t>(seq) * num_heads + h) * row_bytes + d * 2));
}

template <class Tag, int D>
__global__ void __launch_bounds__((kMaxG + 1) * 32, 1)
    paged_attn_shared_kernel(const __grid_constant__ CUtensorMap tm_k,
                             const __grid_constant__ CUtensorMap tm_v, const SharedParams p) {
  using Gm = Geo<D>;
  constexpr int kRowBytes = D * 2;
  // This pass is the call's first kernel, launched as a programmatic dependent
  // of whatever precedes the call on the stream (the previous decode call's
  // merge, typically): nothing in memory is touched before that kernel has
  // completed and its writes are visible.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // The per-sequence partition pass follows as a programmatic dependent (it
  // reads nothing this pass writes): let it start once every block here has
  // (and so only after the wait above).  Its first block waits for this pass to
  // complete before it exits, so the merge after it follows both.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  extern __shared__ __align__(128) uint8_t smem[];
  const int G = p.heads_per_cta;
  const int S = p.stages;
  const int hg = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (p.record_count != nullptr) {  // a launch sized for the list's capacity
    const int n = __ldg(p.record_count);
    if (n < 0 || n > p.num_records) {
      if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0)
        report_error(p.err, PA_ERR_BAD_SEQ_LEN, -2, n);
      return;
    }
    if (static_cast<int>(blockIdx.y) >= n) return;
  }
  const int32_t* rec = p.records + static_cast<size_t>(blockIdx.y) * kRecord;

  // Check the record (every thread reaches the same conclusion): partition in
  // range, 1..8 members, each a valid sequence whose length covers the whole
  // partition (and, with a fused append, the appended token lies past it); or,
  // for a prefix record (word 1 = m + 256 c, c > 0), the first c chunks of the
  // partition, with each member's own part starting right after them
  // (tail_start) and holding at least its last token.
  const int part = __ldg(rec);
  const int mw = __ldg(rec + 1);
  const int m = mw & 255;
  const int pc = mw >> 8;  // prefix chunks; 0: the whole partition
  const int cap = p.max_blocks * p.block_size;
  bool bad = part < 0 || part >= p.num_partitions || m < 1 || m > kMembers || pc < 0 ||
             pc >= p.partition_tokens / kChunk || (pc > 0 && p.tail_start == nullptr);
  int bad_value = part < 0 || part >= p.num_partitions ? part : mw;
  const long long split = static_cast<long long>(part) * p.partition_tokens + pc * kChunk;
  if (!bad) {
    const long long need = pc > 0 ? split + 1
                                  : static_cast<long long>(part + 1) * p.partition_tokens +
                                        (p.fused_append ? 1 : 0);
    for (int i = 0; i < m && !bad; ++i) {
      const int s = __ldg(rec + 2 + i);
      if (s < 0 || s >= p.num_seqs) {
        bad = true;
        bad_value = s;
      } else {
        const int L = __ldg(p.seq_lens + s);
        if (L < need || L > cap || (pc > 0 && __ldg(p.tail_start + s) != split)) {
          bad = true;
          bad_value = s;
        }
      }
    }
  }
  if (bad) {
    if (threadIdx.x == 0 && hg == 0) report_error(p.err, PA_ERR_BAD_SEQ_LEN, blockIdx.y, bad_value);
    return;
  }
  const int first = __ldg(rec + 2);
  const int tok_begin = part * p.partition_tokens;
  const int nchunks = pc > 0 ? pc : p.partition_tokens / kChunk;

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
    if (p.block_size >= kChunk) {
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
      // 8-token blocks: rows 0-7 of a chunk come from the block of its first
      // token, rows 8-15 from the next one (8-row boxes into the same tile);
      // lane l looks up half l % 2 of chunk c0 + l / 2.  Records cover whole
      // partitions, so both halves always hold tokens.
      for (int c0 = 0; c0 < nchunks && !stop; c0 += 16) {
        int blk = 0;
        const int chunk_l = c0 + (lane >> 1);
        if (chunk_l < nchunks) {
          const int tok = tok_begin + chunk_l * kChunk + (lane & 1) * (kChunk / 2);
          blk = __ldg(table + tok / p.block_size);
          if (static_cast<unsigned>(blk) >= static_cast<unsigned>(p.num_blocks)) {
            report_error(p.err, PA_ERR_BAD_BLOCK, first, blk);
            blk = 0;
          }
        }
        const int n = min(16, nchunks - c0);
        for (int j = 0; j < n; ++j) {
          const int b = __shfl_sync(kFullMask, blk, 2 * j);
          const int b_hi = __shfl_sync(kFullMask, blk, 2 * j + 1);
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
              uint8_t* dst = ring + s * stage_bytes;
              for (int w = 0; w < G; ++w) {
                const int y = (b * p.num_heads + h0 + w) * p.block_size;
                const int y_hi = (b_hi * p.num_heads + h0 + w) * p.block_size;
#pragma unroll
                for (int cg = 0; cg < Gm::kGroups; ++cg) {
                  uint8_t* kd = dst + (w * 2) * Gm::kTileBytes + cg * Gm::kGroupBytes;
                  uint8_t* vd = dst + (w * 2 + 1) * Gm::kTileBytes + cg * Gm::kGroupBytes;
                  tma_load_2d(kd, &tm_k, cg * 64, y, &full[s]);
                  tma_load_2d(kd + Gm::kGroupBytes / 2, &tm_k, cg * 64, y_hi, &full[s]);
                  tma_load_2d(vd, &tm_v, cg * 64, y, &full[s]);
                  tma_load_2d(vd + Gm::kGroupBytes / 2, &tm_v, cg * 64, y_hi, &full[s]);
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
    }
  } else {
    // ------------------------------------------------------------ consumer
    // Per chunk, on mma.sync m16n8k16 with the chunk's 16 tokens as the M rows and
    // the (up to 8) members as the N columns: S^T = K.Q^T (K as the A operand,
    // Q^T as B), the online softmax of each member's column in log2 units, then
    // O^T += V^T.P^T (V^T as A, P^T as B, P in high + low half-precision parts).
    // Lane (g, tq), g = lane / 4, tq = lane % 4, holds the scores of tokens g and
    // g + 8 for members 2 tq and 2 tq + 1, and the output of dims 16 dd + g and
    // 16 dd + g + 8 for the same two members.
    const int h = hg * G + warp;
    const int g = lane >> 2, tq = lane & 3;
    const char* qb = static_cast<const char*>(p.q);
    const int seq_b = g < m ? __ldg(rec + 2 + g) : -1;  // member of B column g
    uint32_t qf[D / 16][2];                              // Q^T as B fragments
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      qf[kk][0] = ld_pair(qb, seq_b, p.num_heads, h, kk * 16 + 2 * tq, kRowBytes);
      qf[kk][1] = ld_pair(qb, seq_b, p.num_heads, h, kk * 16 + 8 + 2 * tq, kRowBytes);
    }
    float o[D / 16][4];
#pragma unroll
    for (int dd = 0; dd < D / 16; ++dd) o[dd][0] = o[dd][1] = o[dd][2] = o[dd][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;  // members 2 tq, 2 tq + 1

    // ldmatrix row addresses of this lane: lanes 8i..8i+7 name the rows of
    // matrix i.  K (A operand, no transpose): matrices (tokens 0-7, d+0..7),
    // (8-15, d+0..7), (0-7, d+8..15), (8-15, d+8..15).  V (A operand of V^T,
    // transposed): (tokens 0-7, d+0..7), (0-7, d+8..15), (8-15, d+0..7), (8-15, d+8..15).
    // Token t's 16-byte chunk c of a 64-column group sits at t * 128 + (c ^ (t & 7)) * 16,
    // and t & 7 is this lane's r8.
    const int mi = lane >> 3, r8 = lane & 7;
    const uint32_t k_row = static_cast<uint32_t>(((mi & 1) * 8 + r8) * 128);
    const uint32_t v_row = static_cast<uint32_t>(((mi >> 1) * 8 + r8) * 128);
    const int k_half = mi >> 1, v_half = mi & 1;
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

      float sc[4] = {0.f, 0.f, 0.f, 0.f};  // (token g, 2 tq), (g, 2 tq + 1), (g + 8, ...)
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        uint32_t a[4];
        const int c = ((kk & 3) << 1) | k_half;
        ldsm_x4(kt + (kk >> 2) * Gm::kGroupBytes + k_row + ((c ^ r8) << 4), a);
        mma(sc, a, qf[kk][0], qf[kk][1], Tag{});
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) sc[e] *= p.qscale;

      // a member's 16 scores sit on the 8 lanes of equal tq, two per lane
      float c0 = fmaxf(sc[0], sc[2]), c1 = fmaxf(sc[1], sc[3]);
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        c0 = fmaxf(c0, __shfl_xor_sync(kFullMask, c0, off));
        c1 = fmaxf(c1, __shfl_xor_sync(kFullMask, c1, off));
      }
      const float mn0 = fmaxf(m0, c0), mn1 = fmaxf(m1, c1);
      const float a0 = exp2f(m0 - mn0), a1 = exp2f(m1 - mn1);
      const float p0 = exp2f(sc[0] - mn0), p1 = exp2f(sc[1] - mn1);
      const float p2 = exp2f(sc[2] - mn0), p3 = exp2f(sc[3] - mn1);
      l0 = fmaf(l0, a0, p0 + p2);
      l1 = fmaf(l1, a1, p1 + p3);
      if (__any_sync(kFullMask, a0 != 1.f || a1 != 1.f)) {
#pragma unroll
        for (int dd = 0; dd < D / 16; ++dd) {
          o[dd][0] *= a0;
          o[dd][1] *= a1;
          o[dd][2] *= a0;
          o[dd][3] *= a1;
        }
      }
      m0 = mn0;
      m1 = mn1;

      // P^T as the B operand: the C layout holds (token, two members); an 8x8
      // transpose per half (tokens 0-7, 8-15) gives (two tokens, member)
      uint32_t hi_a, lo_a, hi_b, lo_b;
      split2(p0, p1, hi_a, lo_a, Tag{});
      split2(p2, p3, hi_b, lo_b, Tag{});
      const uint32_t bh0 = movmatrix_trans(hi_a), bh1 = movmatrix_trans(hi_b);
      const uint32_t bl0 = movmatrix_trans(lo_a), bl1 = movmatrix_trans(lo_b);
#pragma unroll
      for (int dd = 0; dd < D / 16; ++dd) {
        uint32_t a[4];
        const int c = ((dd & 3) << 1) | v_half;
        ldsm_x4_trans(vt + (dd >> 2) * Gm::kGroupBytes + v_row + ((c ^ r8) << 4), a);
        mma(o[dd], a, bh0, bh1, Tag{});
        mma(o[dd], a, bl0, bl1, Tag{});
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      if (__shfl_sync(kFullMask, *abort_flag, 0)) break;
    }

#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l0 += __shfl_xor_sync(kFullMask, l0, off);
      l1 += __shfl_xor_sync(kFullMask, l1, off);
    }
    if (!*abort_flag) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int mm = 2 * tq + e;
        if (mm >= m) continue;
        const int seq = __ldg(rec + 2 + mm);
        const float mrow = e ? m1 : m0, lrow = e ? l1 : l0;
        const int L = __ldg(p.seq_lens + seq);
        const int nparts = (L + p.partition_tokens - 1) / p.partition_tokens;
        const size_t base = (static_cast<size_t>(seq) * p.num_heads + h) * D + g;
        if (nparts == 1 && pc == 0) {
          const float inv = lrow > 0.f ? 1.f / lrow : 0.f;
#pragma unroll
          for (int dd = 0; dd < D / 16; ++dd) {
            store_one(p.out, base + dd * 16, o[dd][e] * inv, p.out_dtype);
            store_one(p.out, base + dd * 16 + 8, o[dd][2 + e] * inv, p.out_dtype);
          }
        } else {
          const size_t row =
              (static_cast<size_t>(seq) * p.num_heads + h) * p.num_partitions + part;
          float* dst = p.ws_acc + row * D + g;
#pragma unroll
          for (int dd = 0; dd < D / 16; ++dd) {
            dst[dd * 16] = o[dd][e];
            dst[dd * 16 + 8] = o[dd][2 + e];
          }
          if (g == 0) p.ws_ml[row] = make_float2(mrow, lrow);
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

// Opt-in shared memory above the 48 KB default, set on every launch that needs
// it (the attribute is lost with the context, e.g. after cudaDeviceReset).
template <class Tag, int D>
cudaError_t ensure_shared_smem_attr(int device, size_t smem) {
  if (smem <= 48 * 1024) return cudaSuccess;
  int optin = 0;
  cudaError_t e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(paged_attn_shared_kernel<Tag, D>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
}

template <class Tag, int D>
int launch_t(const SharedParams& p, cudaStream_t stream) {
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return PA_ERR_CUDA;
  const size_t smem = shared_kernel_smem_bytes(D, p.heads_per_cta, p.stages);
  if (ensure_shared_smem_attr<Tag, D>(device, smem) != cudaSuccess) return PA_ERR_CUDA;
  // the caches as [num_blocks * H * bs][D] row-major, boxes of 16 rows x 64 columns
  const unsigned long long rows =
      static_cast<unsigned long long>(p.num_blocks) * p.num_heads * p.block_size;
  if (rows >= (1ull << 31)) return PA_ERR_UNSUPPORTED;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), rows};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(D) * 2};
  // a box is one 16-token chunk, or half of one with 8-token blocks
  const cuuint32_t box[2] = {64, p.block_size >= kChunk ? 16u : 8u};
  CUtensorMap tk, tv;
  const bool bf16 = std::is_same<Tag, BF16>::value;
  if (!encode_tensor_map(&tk, bf16, p.k_cache, 2, dims, strides, box) ||
      !encode_tensor_map(&tv, bf16, p.v_cache, 2, dims, strides, box))
    return PA_ERR_CUDA;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(p.num_heads / p.heads_per_cta, p.num_records);
  cfg.blockDim = dim3((p.heads_per_cta + 1) * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
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

int launch_shared_partitions(const SharedParams& p, int dtype, int head_dim, cudaStream_t stream) {
  if (p.num_records == 0) return PA_OK;
  if (p.num_records < 0 || p.num_records > 65535 || p.heads_per_cta < 1 ||
      p.heads_per_cta > kMaxG || p.num_heads % p.heads_per_cta != 0 || p.stages < 2 ||
      p.stages > kMaxRing || p.partition_tokens % kChunk != 0 ||
      (p.block_size % kChunk != 0 && p.block_size != 8))
    return PA_ERR_INVALID_ARG;
  if (shared_kernel_smem_bytes(head_dim, p.heads_per_cta, p.stages) > 227 * 1024)
    return PA_ERR_INVALID_ARG;
  const bool bf16 = dtype == PA_BF16;
  switch (head_dim) {
    case 64:
      return bf16 ? launch_t<BF16, 64>(p, stream) : launch_t<F16, 64>(p, stream);
    case 128:
      return bf16 ? launch_t<BF16, 128>(p, stream) : launch_t<F16, 128>(p, stream);
    case 256:
      return bf16 ? launch_t<BF16, 256>(p, stream) : launch_t<F16, 256>(p, stream);
    default: return PA_ERR_UNSUPPORTED;
  }
}

}  // namespace pagedkv
