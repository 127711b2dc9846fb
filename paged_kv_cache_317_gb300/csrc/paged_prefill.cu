// Chunked prefill / multi-query attention through the block table on the
// 5th-generation tensor cores (tcgen05 + TMEM + TMA), sm_103a.
//
// Several query tokens per sequence (a prefill chunk, or draft tokens to
// verify) attend causally over the sequence's tokens, read through its block
// table (PagedAttention, zeroshotmind.com page, "Block tables: logical order,
// physical scatter").  With >1 query per head the work is a dense contraction,
// so it runs on tensor cores:
//
//  * work item = (128-query tile, head, sequence).  The kernel is persistent:
//    one block per resident slot (two per SM at head_dim <= 128).  Items are
//    numbered sequence by sequence in the given dispatch order, a sequence's
//    later (longer) query tiles first, heads innermost, and block b takes
//    items b, b + grid, b + 2 grid, ...  Key tiles are counted across a
//    block's items, so the next item's Q and first K/V tiles load while the
//    current one finishes.  7 warps: one softmax warpgroup (one query row per
//    thread = one TMEM lane; it also writes the output), a K producer (which
//    also loads Q), an MMA issuer and a V producer.  head_dim 64, 128 or 256:
//    tiles are stored as head_dim / 64 column groups of 64 elements.  At 64
//    and 128, <= 106 KB of shared memory and 256 TMEM columns, so two blocks
//    share an SM and cover each other's hand-offs; at 256, ~202 KB and 512
//    columns, one block per SM.
//  * Q tile: two 3-D TMA loads (one per 64-wide half of head_dim, 128B
//    swizzle), once every S of the block's previous item has completed.  K/V:
//    per 16-key chunk the producers follow the block table (32 entries at a
//    time) and issue 2-D TMA loads of the rows (128B swizzle) into 2-stage K
//    and V rings of 64-key tiles, each chunk's boxes by the lane holding its
//    table entry; a K tile is released when its S MMA completes, a V tile when
//    its P.V completes (the completion barriers of S/P buffer j & 1 serve for
//    both).  O is released to the next item's first P.V once the epilogue has
//    read it.
//  * S = Q K^T: 8 tcgen05.mma (M=128, N=64, K=16, fp32 accumulate) into one of
//    two 64-column TMEM buffers.  Buffer j & 1 is reused for S(j+2) only after
//    P.V(j), which reads the P stored there, has completed.
//  * Softmax: tcgen05.ld of the S row, causal/length mask only on tiles that
//    cross a row's limit, exponentials by ex2.approx against a per-row
//    reference max that moves only when the running max passes it by 2^8 (O is
//    rescaled in TMEM only then).  P is stored back over its S as two 16-bit
//    parts per key, hi = round(p) and lo = round(p - hi): a single bf16 P would
//    carry up to 2^-8 relative error per weight, more than the 2e-3 bound
//    allows on rows dominated by a few keys.
//  * O += P V: 4 + 4 tcgen05.mma (hi and lo; M=128, N=128, K=16 keys) with A
//    read from TMEM and V as an MN-major shared-memory operand, accumulating
//    in TMEM.  The commit of buffer b's P.V is also the completion signal the
//    softmax waits on before rescaling O or reading it in the epilogue.
//  * Epilogue: O / l leaves through 2 KB of shared memory per warp, so that
//    each store instruction writes whole 64-byte row segments.
//  * Every mbarrier wait is bounded (one second); on a timeout the block
//    records PA_ERR_TIMEOUT, waits (bounded) for its copies and MMAs, frees its
//    TMEM and returns.  Nothing traps.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>

#include "common.cuh"
#include "tma.cuh"

namespace pagedkv {
namespace {

constexpr int kQTile = 128;                       // query rows per block (MMA M)
constexpr int kKTile = 64;                        // keys per tile
constexpr int kThreads = 224;                     // 4 softmax, K producer, MMA, V producer
constexpr int kWarpK = 4, kWarpMma = 5, kWarpV = 6;
constexpr int kKStages = 2;                       // K ring depth (= the S buffers: a stage is freed by its S)
constexpr int kVStages = 2;                       // V ring depth (= the S/P buffers: a stage is freed by its P.V)
static_assert(kKStages == 2 && kVStages == 2,
              "K and V stage s are released through S/P buffer s's completion barriers");
constexpr int kHalfBytes = kKTile * 128;          // 64 rows x 128 B: one 64-wide column group of a K/V tile
constexpr int kQHalfBytes = kQTile * 128;         // 128 rows x 128 B: one 64-wide column group of Q
// TMEM: two S/P buffers of 64 columns (S in fp32; after the softmax, P hi in the
// first 32 columns and P lo in the next 32, two 16-bit values per column), then O.
constexpr uint32_t kTmemO = 2 * kKTile;

// Sizes that follow from head_dim D (64, 128 or 256): the tiles are stored as
// D / 64 column groups of 64 elements (128 bytes, the 128-byte swizzle atom).
template <int D>
struct Cfg {
  static constexpr int kGroups = D / 64;
  static constexpr int kQBytes = kGroups * kQHalfBytes;       // 16 / 32 / 64 KB
  static constexpr int kTileBytes = kGroups * kHalfBytes;     // one K or V tile: 8 / 16 / 32 KB
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kQBytes;
  static constexpr int kOffV = kOffK + kKStages * kTileBytes;
  static constexpr int kOffStage = kOffV + kVStages * kTileBytes;  // 4 warps x 2 KB
  static constexpr int kOffBar = kOffStage + 8192;
  // 1 KB is left for aligning the dynamic shared-memory base to 1 KB (the
  // kernel checks it); at D <= 128 two blocks still fit an SM (228 KB, less 1 KB
  // reserved per block).
  static constexpr int kAlignSlack = 1024;
  static constexpr int kSmemUsed = kOffBar + 256 + kAlignSlack;
  // Requested per block: at least 80 KB, so that no more than two blocks (two
  // 256-column TMEM allocations) ever share an SM, whatever the register count.
  static constexpr int kSmemBytes = kSmemUsed > 80 * 1024 ? kSmemUsed : 80 * 1024;
  // D = 256 needs 384 TMEM columns (allocated as 512) and ~193 KB: one block per SM.
  static constexpr int kMinBlocks = D <= 128 ? 2 : 1;
  static constexpr uint32_t kTmemCols = kTmemO + D <= 256 ? 256 : 512;
  static_assert(D == 64 || D == 128 || D == 256, "head_dim");
  static_assert(kMinBlocks == 1 || kSmemBytes <= 228 * 1024 / 2 - 1024, "two blocks per SM");
  static_assert(kSmemBytes <= 227 * 1024, "one block per SM");
};
constexpr float kLog2e = 1.4426950408889634f;
// A row's exponentials are taken against a reference max that only moves when
// the running max exceeds it by more than this (log2 units): p <= 2^8, exact in
// fp32, and O is rescaled only then.
constexpr float kRescaleThreshold = 8.0f;

struct Bars {
  uint64_t q_full, q_empty;
  uint64_t k_full[kKStages], v_full[kVStages];
  // s_free[b] completes when the P.V of buffer b's tile finishes (one phase
  // per two tiles), so it doubles as that P.V's completion signal.
  uint64_t s_full[2], s_free[2], p_full[2];
  uint64_t o_free;  // the epilogue has read O: the next tile's first P.V may overwrite it
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(Bars) <= 256, "barrier block");

struct PrefillParams {
  const int32_t* seq_order;  // optional dispatch order of the sequences
  const int32_t* query_start;
  const int32_t* seq_lens;
  const int32_t* block_tables;
  void* out;
  int32_t* err;
  int num_heads, block_size, max_blocks, num_blocks, out_dtype;
  int total_queries;  // rows of q and out
  float qscale;
};

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Shared-memory matrix descriptor (tcgen05): start, leading / stride byte
// offsets (16-byte units), descriptor version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t smem_desc_sw128(const void* p, uint32_t lbo, uint32_t sbo) {
  const uint32_t a = smem_addr(p);
  uint64_t d = static_cast<uint64_t>((a >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;
  d |= 2ull << 61;
  return d;
}

// Instruction descriptor for kind::f16: fp32 accumulator, A and B both bf16 (or
// both fp16), A K-major, B K-major or MN-major, shape M x N.
__host__ __device__ constexpr uint32_t make_idesc(int m, int n, bool bf16, bool b_mn_major) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
         ((b_mn_major ? 1u : 0u) << 16) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(m >> 4) << 24);
}

__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Same, with A read from tensor memory (M rows = lanes, K values packed two per
// 32-bit column).
__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
               : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  uint32_t r[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(v[i]);
  asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
               : "memory");
}

// Two fp32 lanes at once (sm_100+ packed f32x2 arithmetic, round to nearest:
// the same results as two scalar operations).
__device__ __forceinline__ void fma2(float& y0, float& y1, float x0, float x1, float s, float c) {
  asm("{\n\t.reg .b64 x, s, c, d;\n\tmov.b64 x, {%2, %3};\n\tmov.b64 s, {%4, %4};\n\t"
      "mov.b64 c, {%5, %5};\n\tfma.rn.f32x2 d, x, s, c;\n\tmov.b64 {%0, %1}, d;\n\t}"
      : "=f"(y0), "=f"(y1)
      : "f"(x0), "f"(x1), "f"(s), "f"(c));
}

__device__ __forceinline__ void add2(float& a0, float& a1, float x0, float x1) {
  asm("{\n\t.reg .b64 a, x, d;\n\tmov.b64 a, {%0, %1};\n\tmov.b64 x, {%2, %3};\n\t"
      "add.rn.f32x2 d, a, x;\n\tmov.b64 {%0, %1}, d;\n\t}"
      : "+f"(a0), "+f"(a1)
      : "f"(x0), "f"(x1));
}

// (y0, y1) = (a0 - b0, a1 - b1), one packed instruction, same rounding as scalar fp32.
__device__ __forceinline__ void sub2(float& y0, float& y1, float a0, float a1, float b0, float b1) {
  asm("{\n\t.reg .b64 a, b, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
      "sub.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"
      : "=f"(y0), "=f"(y1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// 2^x by the SFU's approximate base-2 exponential (PTX ex2.approx.ftz.f32;
// relative error ~2^-22, 2^-inf = +0).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Two floats -> two 16-bit values (bf16 or fp16, round to nearest even), packed.
template <bool BF16>
__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
  if constexpr (BF16) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
  } else {
    __half2 v = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
  }
}

template <bool BF16>
__device__ __forceinline__ float half_to_float(uint32_t bits16) {
  if constexpr (BF16) {
    return __uint_as_float(bits16 << 16);
  } else {
    __half h;
    *reinterpret_cast<uint16_t*>(&h) = static_cast<uint16_t>(bits16);
    return __half2float(h);
  }
}

// One work item: 128-query tile `q0 / kQTile` of sequence `seq`, head `h`.
struct Tile {
  int seq, h, q_begin, q0;
  int rows;  // valid query rows
  int pos0;  // position of the first query
  int keys;  // keys any row of the tile sees
  int T;     // 64-key tiles
  bool valid;
};

// Item `it` of the launch: dispatch position z (through seq_order), then the
// later (longer) query tiles of that sequence first, heads innermost.  Every
// thread decodes the same items from the same device values, so all roles
// agree on which items exist.
__device__ __forceinline__ Tile decode_tile(const PrefillParams& p, int it, int num_seqs,
                                            int num_qtiles, bool report) {
  Tile w;
  w.valid = false;
  const int per_seq = p.num_heads * num_qtiles;
  const int z = it / per_seq, rem = it % per_seq;
  const int qt = num_qtiles - 1 - rem / p.num_heads;
  w.h = rem % p.num_heads;
  int seq = z;
  if (p.seq_order != nullptr) {
    seq = __ldg(p.seq_order + z);
    if (static_cast<unsigned>(seq) >= static_cast<unsigned>(num_seqs)) {
      if (report && rem == 0) report_error(p.err, PA_ERR_BAD_SEQ_LEN, z, seq);
      return w;
    }
  }
  w.seq = seq;
  int L = __ldg(p.seq_lens + seq);
  w.q_begin = __ldg(p.query_start + seq);
  const int nq = __ldg(p.query_start + seq + 1) - w.q_begin;
  const int cap = p.max_blocks * p.block_size;
  // Lengths and query ranges come from device memory: a bad one is recorded and
  // the sequence is clamped or skipped, never used to address memory.
  const bool bad_len = L < 0 || L > cap;
  L = L < 0 ? 0 : (L > cap ? cap : L);
  const bool bad_q = nq < 0 || nq > L || w.q_begin < 0 || w.q_begin > p.total_queries - nq ||
                     nq > num_qtiles * kQTile;
  if (bad_len || bad_q) {
    if (report && rem == 0) report_error(p.err, PA_ERR_BAD_SEQ_LEN, seq, L);
    if (bad_q) return w;
  }
  w.q0 = qt * kQTile;
  if (w.q0 >= nq) return w;
  w.rows = min(kQTile, nq - w.q0);
  w.pos0 = L - nq + w.q0;
  w.keys = w.pos0 + w.rows;
  w.T = (w.keys + kKTile - 1) / kKTile;
  w.valid = true;
  return w;
}

// The r-th item of this block: block b takes items b, b + gridDim.x, ...
// (Dealing every other round in reverse, to even out long and short items per
// block, measured 2 % slower: the two blocks sharing an SM already even out.)
__device__ __forceinline__ int item_of(int r) {
  return r * static_cast<int>(gridDim.x) + static_cast<int>(blockIdx.x);
}

template <bool BF16, int D>
__global__ void __launch_bounds__(kThreads, Cfg<D>::kMinBlocks)
    paged_prefill_kernel(const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const PrefillParams p,
                         const int num_seqs, const int num_qtiles) {
  using C = Cfg<D>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_addr(smem_raw) & 1023u)) & 1023u;
  if (pad > C::kAlignSlack) {  // never seen: the base is 1 KB aligned in practice
    if (threadIdx.x == 0) report_error(p.err, PA_ERR_UNSUPPORTED, -1, static_cast<int>(pad));
    return;
  }
  uint8_t* smem = smem_raw + pad;
  uint8_t* Qs = smem + C::kOffQ;
  Bars* bars = reinterpret_cast<Bars*>(smem + C::kOffBar);
  volatile int* abort_flag = &bars->abort;
  auto k_tile = [&](int s) { return smem + C::kOffK + s * C::kTileBytes; };
  auto v_tile = [&](int s) { return smem + C::kOffV + s * C::kTileBytes; };
  // With 8-token blocks a 16-key chunk spans two blocks: rows 0-7 come from the
  // block of its first key, rows 8-15 from the next one (boxes of 8 rows).
  const bool half_blocks = p.block_size < 16;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, 1);
    for (int s = 0; s < kKStages; ++s) mbar_init(&bars->k_full[s], 1);
    for (int s = 0; s < kVStages; ++s) mbar_init(&bars->v_full[s], 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->s_full[b], 1);
      mbar_init(&bars->s_free[b], 1);
      mbar_init(&bars->p_full[b], kQTile);
    }
    mbar_init(&bars->o_free, kQTile);
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(&bars->tmem_base)),
                 "r"(C::kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const int n_items = num_seqs * p.num_heads * num_qtiles;

  // Key tiles are counted across the block's items: tile g of the block uses K
  // and V stage g & 1 and S/P buffer g & 1, and its barriers' phases are g >> 1.
  int kv_issued = 0;    // producers: tiles whose loads were issued (all lanes agree)
  int q_issued = 0;     // K producer: Q tiles whose loads were issued
  int mma_started = 0;  // MMA lane 0: whether any MMA was issued
  if (warp == kWarpK || warp == kWarpV) {
    // ------------------------------------------------- producers: K (+Q) and V
    const bool is_v = (warp == kWarpV);
    const CUtensorMap* map = is_v ? &tm_v : &tm_k;
    bool ok = true;
    for (int turn = 0, it = item_of(0); ok && it < n_items; it = item_of(++turn)) {
      const Tile w = decode_tile(p, it, num_seqs, num_qtiles, !is_v && lane == 0);
      if (!w.valid) continue;
      const int32_t* table = p.block_tables + static_cast<size_t>(w.seq) * p.max_blocks;
      int blk = 0, blk_hi = 0;
      for (int j = 0; j < w.T; ++j) {
        if ((j & 7) == 0) {
          // lane l looks up the physical block of 16-key chunk 4*j + l (8 tiles'
          // worth) (and, with 8-token blocks, that of its second half)
          const int key0 = (j * 4 + lane) * 16;
          blk = 0;
          blk_hi = 0;
          if (key0 < w.keys) {
            blk = __ldg(table + key0 / p.block_size);
            if (static_cast<unsigned>(blk) >= static_cast<unsigned>(p.num_blocks)) {
              if (!is_v) report_error(p.err, PA_ERR_BAD_BLOCK, w.seq, blk);
              blk = 0;
            }
          }
          if (half_blocks && key0 + 8 < w.keys) {
            blk_hi = __ldg(table + (key0 + 8) / p.block_size);
            if (static_cast<unsigned>(blk_hi) >= static_cast<unsigned>(p.num_blocks)) {
              if (!is_v) report_error(p.err, PA_ERR_BAD_BLOCK, w.seq, blk_hi);
              blk_hi = 0;
            }
          }
        }
        const int g = kv_issued, s = g & 1, use = g >> 1;
        // rows loaded: 16 per chunk holding visible keys; with 8-token blocks a
        // chunk whose second half holds none loads 8
        const int kt0 = j * kKTile;
        int rows_loaded = 16 * min(4, (w.keys - kt0 + 15) / 16);
        if (half_blocks && w.keys - kt0 < kKTile && (w.keys - kt0) % 16 != 0 &&
            (w.keys - kt0) % 16 <= 8)
          rows_loaded -= 8;
        uint64_t* full = is_v ? &bars->v_full[s] : &bars->k_full[s];
        // A K stage is free once the S that read it has completed, a V stage once
        // the P.V that read it has: with two stages of each and two S/P buffers,
        // those are s_full[s] and s_free[s].  (The next completion on either
        // barrier needs the load being waited for, so no phase can be skipped.)
        uint64_t* empty = is_v ? &bars->s_free[s] : &bars->s_full[s];
        uint8_t* dst = is_v ? v_tile(s) : k_tile(s);
        int good = 1;
        if (lane == 0) {
          if (use > 0) good = mbar_wait_bounded(empty, (use - 1) & 1);
          if (good)
            mbar_arrive_expect_tx(full, static_cast<uint32_t>(rows_loaded) * C::kGroups * 128);
        }
        good = __shfl_sync(kFullMask, good, 0);
        if (!good) {
          if (lane == 0) {
            *abort_flag = 1;
            report_error(p.err, PA_ERR_TIMEOUT, w.seq, j);
          }
          ok = false;
          break;
        }
        // Lanes 4 (j % 8) .. 4 (j % 8) + 3 hold the blocks of this tile's four
        // chunks (and, with 8-token blocks, of their second halves): each issues
        // its own chunk's boxes, so a tile's loads go out in one warp instruction
        // per column group rather than one thread's sequence of them (the
        // producers sit on the critical path).
        {
          const int c = lane - (j & 7) * 4;
          const int k0 = j * kKTile + c * 16;
          if (c >= 0 && c < 4 && k0 < w.keys) {
            const int row = (blk * p.num_heads + w.h) * p.block_size + k0 % p.block_size;
#pragma unroll
            for (int gr = 0; gr < C::kGroups; ++gr)
              tma_load_2d(dst + gr * kHalfBytes + c * 2048, map, 64 * gr, row, full);
            if (half_blocks && k0 + 8 < w.keys) {
              const int row_hi = (blk_hi * p.num_heads + w.h) * p.block_size;
#pragma unroll
              for (int gr = 0; gr < C::kGroups; ++gr)
                tma_load_2d(dst + gr * kHalfBytes + c * 2048 + 1024, map, 64 * gr, row_hi, full);
            }
          }
        }
        kv_issued = g + 1;
        if (!is_v && j == 0) {
          // This item's Q tile, once every S of the previous item has completed
          // (issued after K(0) so that tile's latency overlaps the wait).
          if (lane == 0) {
            if (q_issued > 0) good = mbar_wait_bounded(&bars->q_empty, (q_issued - 1) & 1);
            if (good) {
              mbar_arrive_expect_tx(&bars->q_full, C::kQBytes);
#pragma unroll
              for (int gr = 0; gr < C::kGroups; ++gr)
                tma_load_3d(Qs + gr * kQHalfBytes, &tm_q, 64 * gr, w.h, w.q_begin + w.q0,
                            &bars->q_full);
            }
          }
          good = __shfl_sync(kFullMask, good, 0);
          if (!good) {
            if (lane == 0) {
              *abort_flag = 1;
              report_error(p.err, PA_ERR_TIMEOUT, w.seq, -3);
            }
            ok = false;
            break;
          }
          ++q_issued;
        }
        __syncwarp();
        if (__shfl_sync(kFullMask, *abort_flag, 0)) {
          ok = false;
          break;
        }
      }
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = make_idesc(kQTile, kKTile, BF16, false);
      constexpr uint32_t idesc_o = make_idesc(kQTile, D, BF16, true);
      // descriptors of the tile bases; an offset within a tile is added to the
      // start-address field (16-byte units, no carry: shared memory < 256 KB)
      const uint64_t q_desc = smem_desc_sw128(Qs, 16, 1024);
      const uint64_t k_desc0 = smem_desc_sw128(k_tile(0), 16, 1024);
      const uint64_t v_desc0 = smem_desc_sw128(v_tile(0), kHalfBytes, 1024);
      int g = 0, items = 0;
      bool ok = true;
      for (int turn = 0, it = item_of(0); ok && it < n_items; it = item_of(++turn)) {
        const Tile w = decode_tile(p, it, num_seqs, num_qtiles, false);
        if (!w.valid) continue;
        if (!mbar_wait_bounded(&bars->q_full, items & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int g0 = g;
        // S of the block's tile gg goes to TMEM buffer gg & 1, whose previous
        // contents (P of tile gg - 2) must have been consumed by P.V(gg - 2).
        // After the item's last S, Q is released for the next item.
        auto issue_s = [&](int gg, bool last) -> bool {
          const int b = gg & 1;
          if (!mbar_wait_bounded(&bars->k_full[b], (gg >> 1) & 1)) return false;
          if (gg >= 2 && !mbar_wait_bounded(&bars->s_free[b], ((gg >> 1) - 1) & 1)) return false;
          tc_fence_after();
          const uint64_t k_desc = k_desc0 + static_cast<uint64_t>((b * C::kTileBytes) >> 4);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const int half = kk >> 2, off = (kk & 3) * 32;
            const uint64_t a = q_desc + static_cast<uint64_t>((half * kQHalfBytes + off) >> 4);
            const uint64_t bd = k_desc + static_cast<uint64_t>((half * kHalfBytes + off) >> 4);
            mma_f16(tmem + b * kKTile, a, bd, idesc_s, kk > 0);
          }
          mma_commit(&bars->s_full[b]);  // also frees K stage b (two stages)
          if (last) mma_commit(&bars->q_empty);
          mma_started = 1;
          return true;
        };
        ok = issue_s(g0, w.T == 1);
        for (int j = 0; ok && j < w.T; ++j) {
          const int gg = g0 + j, b = gg & 1;
          if (j + 1 < w.T && !issue_s(gg + 1, j + 2 == w.T)) {
            ok = false;
            break;
          }
          // the item's first P.V overwrites O: the previous item's epilogue must
          // have read it
          if (j == 0 && items > 0 && !mbar_wait_bounded(&bars->o_free, (items - 1) & 1)) {
            ok = false;
            break;
          }
          if (!mbar_wait_bounded(&bars->p_full[b], (gg >> 1) & 1) ||
              !mbar_wait_bounded(&bars->v_full[b], (gg >> 1) & 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t v_desc = v_desc0 + static_cast<uint64_t>((b * C::kTileBytes) >> 4);
          const uint32_t ph = tmem + b * kKTile, pl = ph + kKTile / 2;
#pragma unroll
          for (int kk = 0; kk < kKTile / 16; ++kk) {
            const uint64_t bd = v_desc + static_cast<uint64_t>((kk * 2048) >> 4);
            mma_f16_ts(tmem + kTmemO, ph + kk * 8, bd, idesc_o, (j > 0 || kk > 0) ? 1u : 0u);
            mma_f16_ts(tmem + kTmemO, pl + kk * 8, bd, idesc_o, 1u);
          }
          mma_commit(&bars->s_free[b]);  // also frees V stage b (two stages)
        }
        g = g0 + w.T;
        ++items;
      }
      if (!ok) {
        *abort_flag = 1;
        report_error(p.err, PA_ERR_TIMEOUT, -1, -1);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int r = threadIdx.x;  // query row = TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    int g = 0;
    bool ok = true;
    for (int turn = 0, it = item_of(0); ok && it < n_items; it = item_of(++turn)) {
      const Tile w = decode_tile(p, it, num_seqs, num_qtiles, false);
      if (!w.valid) continue;
      const bool row_valid = r < w.rows;
      const int pos = row_valid ? w.pos0 + r : -1;
      float m_ref = -INFINITY, l = 0.f;  // reference max (log2 units) and running sum
      for (int j = 0; j < w.T; ++j) {
        const int gg = g + j, b = gg & 1;
        ok = __all_sync(kFullMask, mbar_wait_bounded(&bars->s_full[b], (gg >> 1) & 1));
        if (!ok) break;
        tc_fence_after();
        float sv[kKTile];
        {
          float t[32];
          tmem_ld32(tmem + lane_base + b * kKTile, t);
#pragma unroll
          for (int c = 0; c < 32; ++c) sv[c] = t[c];
          tmem_ld32(tmem + lane_base + b * kKTile + 32, t);
#pragma unroll
          for (int c = 0; c < 32; ++c) sv[32 + c] = t[c];
        }
        // Raw scores; keys a row may not see become -inf.  Only tiles that
        // cross some row's causal limit (the diagonal and the last tile) need it.
        const int kbase = j * kKTile;
        if (!__all_sync(kFullMask, kbase + kKTile - 1 <= pos)) {
#pragma unroll
          for (int c = 0; c < kKTile; ++c) sv[c] = (kbase + c <= pos) ? sv[c] : -INFINITY;
        }
        float mx[4] = {sv[0], sv[1], sv[2], sv[3]};
#pragma unroll
        for (int c = 4; c < kKTile; c += 4) {
#pragma unroll
          for (int i = 0; i < 4; ++i) mx[i] = fmaxf(mx[i], sv[c + i]);
        }
        // scale > 0, so the max of the scaled scores is the scaled max (log2 units)
        const float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * p.qscale;
        // Move the reference only when the tile's max exceeds it by the threshold.
        float alpha = 1.f;
        if (mt > m_ref + kRescaleThreshold) {
          alpha = (m_ref == -INFINITY) ? 0.f : exp2f(m_ref - mt);
          m_ref = mt;
        }
        // No visible key yet (or an unused row): a -inf offset makes every p zero.
        const float neg_ref = (m_ref == -INFINITY) ? -INFINITY : -m_ref;
        float sum4[4] = {0.f, 0.f, 0.f, 0.f};
        // P as hi + lo halves, two 16-bit values per 32-bit TMEM column
        float hi_f[32], lo_f[32];
#pragma unroll
        for (int c = 0; c < kKTile; c += 2) {
          float x0, x1;
          fma2(x0, x1, sv[c], sv[c + 1], p.qscale, neg_ref);
          const float e0 = ex2_approx(x0);
          const float e1 = ex2_approx(x1);
          add2(sum4[c & 2], sum4[(c & 2) + 1], e0, e1);
          if constexpr (BF16) {
            // hi = the upper 16 bits of each fp32 p (a bf16 truncation), one byte
            // permute for the pair; lo = RN(p - hi), where p - hi is exact in fp32
            // and below one bf16 ulp of p, so hi + lo keeps ~16 significant bits
            const uint32_t b0 = __float_as_uint(e0), b1 = __float_as_uint(e1);
            float d0, d1;
            sub2(d0, d1, e0, e1, __uint_as_float(b0 & 0xffff0000u),
                 __uint_as_float(b1 & 0xffff0000u));
            hi_f[c / 2] = __uint_as_float(__byte_perm(b0, b1, 0x7632));
            lo_f[c / 2] = __uint_as_float(pack_half2<true>(d0, d1));
          } else {
            const uint32_t hi = pack_half2<false>(e0, e1);
            const float r0 = half_to_float<false>(hi & 0xffffu);
            const float r1 = half_to_float<false>(hi >> 16);
            hi_f[c / 2] = __uint_as_float(hi);
            lo_f[c / 2] = __uint_as_float(pack_half2<false>(e0 - r0, e1 - r1));
          }
        }
        const float rowsum = (sum4[0] + sum4[1]) + (sum4[2] + sum4[3]);
        // O must not change under a running P.V: rescaling waits for P.V(gg-1).
        if (j > 0 && __any_sync(kFullMask, alpha != 1.f)) {
          ok = __all_sync(kFullMask,
                          mbar_wait_bounded(&bars->s_free[(gg - 1) & 1], ((gg - 1) >> 1) & 1));
          if (!ok) break;
          tc_fence_after();
#pragma unroll 1
          for (int cc = 0; cc < D / 32; ++cc) {
            float o[32];
            tmem_ld32(tmem + lane_base + kTmemO + cc * 32, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= alpha;
            tmem_st32(tmem + lane_base + kTmemO + cc * 32, o);
          }
        }
        // P replaces S in this tile's buffer (S has been read into registers)
        tmem_st32(tmem + lane_base + b * kKTile, hi_f);
        tmem_st32(tmem + lane_base + b * kKTile + kKTile / 2, lo_f);
        tmem_wait_st();
        // keys past the last one any row may see: zero their V rows once the tile
        // has landed (they may hold stale or unused-slot data; 0 * NaN is NaN)
        if (j == w.T - 1 && w.keys < kbase + kKTile) {
          ok = __all_sync(kFullMask, mbar_wait_bounded(&bars->v_full[b], (gg >> 1) & 1));
          if (!ok) break;
          uint8_t* vs = v_tile(b);
          const int first = w.keys - kbase;
          constexpr int kPieces = C::kGroups * 8;  // 16-byte pieces per row
          const int n16 = (kKTile - first) * kPieces;
          for (int idx = r; idx < n16; idx += kQTile) {
            const int row = first + idx / kPieces;
            const int rest = idx % kPieces;
            *reinterpret_cast<uint4*>(vs + (rest >> 3) * kHalfBytes + row * 128 +
                                      (rest & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
          }
          fence_async_smem();
        }
        l = l * alpha + rowsum;
        tc_fence_before();
        mbar_arrive(&bars->p_full[b]);
        if (__shfl_sync(kFullMask, *abort_flag, 0)) {
          ok = false;
          break;
        }
      }
      if (!ok) break;
      // the item's last P.V (earlier ones finish first: they come from one thread
      // into the same accumulator), then the epilogue; O is then free
      const int g_last = g + w.T - 1;
      ok = __all_sync(kFullMask,
                      mbar_wait_bounded(&bars->s_free[g_last & 1], (g_last >> 1) & 1));
      if (!ok) break;
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      // Rows leave through the warp's 2 KB of the staging buffer, 64 bytes of
      // each at a time: each lane writes its row's piece, then the warp stores
      // whole 64-byte row segments (8 rows per instruction) rather than 16
      // bytes of 32 rows.  Pieces sit at an XOR of (row / 2) % 4 so that
      // neither side has bank conflicts.
      const int esz = p.out_dtype == PA_F32 ? 4 : 2;
      const size_t row_bytes = static_cast<size_t>(p.num_heads) * D * esz;
      char* out_warp = static_cast<char*>(p.out) +
                       (static_cast<size_t>(w.q_begin + w.q0 + warp * 32) * p.num_heads + w.h) *
                           D * esz;
      const int warp_rows = w.rows - warp * 32;  // this warp's valid rows (may be <= 0)
      uint8_t* stage = smem + C::kOffStage + warp * 2048;
      auto put = [&](const uint4 (&v)[4], int col_byte) {
#pragma unroll
        for (int k = 0; k < 4; ++k)
          *reinterpret_cast<uint4*>(stage + lane * 64 + ((k ^ ((lane >> 1) & 3)) << 4)) = v[k];
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int idx = lane + 32 * i, row = idx >> 2, k = idx & 3;
          if (row < warp_rows)
            *reinterpret_cast<uint4*>(out_warp + row * row_bytes + col_byte + k * 16) =
                *reinterpret_cast<const uint4*>(stage + row * 64 + ((k ^ ((row >> 1) & 3)) << 4));
        }
        __syncwarp();
      };
#pragma unroll 1
      for (int cc = 0; cc < D / 32; ++cc) {
        float o[32];
        tmem_ld32(tmem + lane_base + kTmemO + cc * 32, o);
        if (cc == D / 32 - 1) {  // O read: the next item's first P.V may overwrite it
          tc_fence_before();
          mbar_arrive(&bars->o_free);
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] *= inv;
        if (esz == 4) {
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint4 v[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float* f = o + hh * 16 + k * 4;
              v[k] = make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]),
                                __float_as_uint(f[2]), __float_as_uint(f[3]));
            }
            put(v, cc * 128 + hh * 64);
          }
        } else {
          uint4 v[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float* f = o + k * 8;
            v[k] = make_uint4(pack2(f[0], f[1], p.out_dtype), pack2(f[2], f[3], p.out_dtype),
                              pack2(f[4], f[5], p.out_dtype), pack2(f[6], f[7], p.out_dtype));
          }
          put(v, cc * 64);
        }
      }
      g += w.T;
    }
    if (!ok && lane == 0) {
      *abort_flag = 1;
      report_error(p.err, PA_ERR_TIMEOUT, -2, warp);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    // Let every copy and MMA this block started finish before its shared
    // memory and TMEM are released (bounded waits).
    if ((warp == kWarpK || warp == kWarpV) && lane == 0) {
      const bool is_v = (warp == kWarpV);
      for (int s = 0; s < 2 && s < kv_issued; ++s) {
        const int last = s + ((kv_issued - 1 - s) / 2) * 2;  // last tile issued into stage s
        mbar_wait_bounded(is_v ? &bars->v_full[s] : &bars->k_full[s], (last >> 1) & 1);
      }
      if (!is_v && q_issued > 0) mbar_wait_bounded(&bars->q_full, (q_issued - 1) & 1);
    }
    if (warp == kWarpMma && lane == 0 && mma_started) {
      mma_commit(&bars->drain);
      mbar_wait_bounded(&bars->drain, 0);
    }
    __syncthreads();
  }
  tc_fence_after();
  if (warp == kWarpMma) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(C::kTmemCols)
                 : "memory");
  }
}

// ------------------------------------------------------------------ host side
// The kernel always needs opt-in shared memory.  The attribute belongs to the
// module loaded in the current context and is lost with it (cudaDeviceReset,
// another driver-API context), so it is set on every launch.
template <bool BF16, int D>
cudaError_t ensure_prefill_smem() {
  return cudaFuncSetAttribute(paged_prefill_kernel<BF16, D>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D>::kSmemBytes);
}

template <bool BF16, int D>
int launch_prefill(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                   const PrefillParams& p, int num_seqs, int num_qtiles, cudaStream_t st) {
  if (ensure_prefill_smem<BF16, D>() != cudaSuccess) return PA_ERR_CUDA;
  // Persistent: one block per resident slot (Cfg<D>::kMinBlocks per SM), each
  // looping over its share of the (sequence, query tile, head) items.
  int device = 0, sms = 0;
  if (cudaGetDevice(&device) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
    return PA_ERR_CUDA;
  const long long items = static_cast<long long>(num_seqs) * p.num_heads * num_qtiles;
  const long long slots = static_cast<long long>(sms) * Cfg<D>::kMinBlocks;
  const unsigned grid = static_cast<unsigned>(items < slots ? items : slots);
  paged_prefill_kernel<BF16, D>
      <<<grid, kThreads, Cfg<D>::kSmemBytes, st>>>(tq, tk, tv, p, num_seqs, num_qtiles);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace
}  // namespace pagedkv

using namespace pagedkv;

extern "C" int paged_attn_prefill(const void* q, const int32_t* query_start, int total_queries,
                                  int max_query_len, const void* k_cache, const void* v_cache,
                                  const int32_t* block_tables, const int32_t* seq_lens,
                                  int num_seqs, int num_heads, int head_dim, int block_size,
                                  int max_blocks_per_seq, int num_blocks, float scale, int dtype,
                                  void* out, int out_dtype, int32_t* error_record, void* stream) {
  return paged_attn_prefill_ex(q, query_start, total_queries, max_query_len, k_cache, v_cache,
                               block_tables, seq_lens, num_seqs, num_heads, head_dim,
                               block_size, max_blocks_per_seq, num_blocks, scale, dtype, out,
                               out_dtype, error_record, stream, nullptr);
}

extern "C" int paged_attn_prefill_ex(const void* q, const int32_t* query_start,
                                     int total_queries, int max_query_len, const void* k_cache,
                                     const void* v_cache, const int32_t* block_tables,
                                     const int32_t* seq_lens, int num_seqs, int num_heads,
                                     int head_dim, int block_size, int max_blocks_per_seq,
                                     int num_blocks, float scale, int dtype, void* out,
                                     int out_dtype, int32_t* error_record, void* stream,
                                     const pa_prefill_opts* opts) {
  NvtxRange range("paged_attn_prefill");
  if (num_seqs < 0 || total_queries < 0 || max_query_len < 0 || num_heads <= 0 ||
      block_size <= 0 || max_blocks_per_seq <= 0 || num_blocks <= 0)
    return PA_ERR_INVALID_ARG;
  if (num_seqs == 0 || total_queries == 0 || max_query_len == 0) return PA_OK;
  if ((head_dim != 64 && head_dim != 128 && head_dim != 256) ||
      (block_size % 16 != 0 && block_size != 8))
    return PA_ERR_UNSUPPORTED;
  if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
  if (out_dtype != PA_F16 && out_dtype != PA_BF16 && out_dtype != PA_F32)
    return PA_ERR_UNSUPPORTED;
  if (!q || !query_start || !k_cache || !v_cache || !block_tables || !seq_lens || !out)
    return PA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
    return PA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return PA_ERR_INVALID_ARG;
  const unsigned long long cache_rows =
      static_cast<unsigned long long>(num_blocks) * num_heads * block_size;
  if (cache_rows >= (1ull << 31) || static_cast<long long>(max_blocks_per_seq) * block_size >
                                        (1ll << 30))
    return PA_ERR_INVALID_ARG;

  const int qtiles = static_cast<int>((static_cast<long long>(max_query_len) + kQTile - 1) / kQTile);
  // items are numbered in an int inside the kernel (with a grid's worth of headroom)
  if (static_cast<long long>(num_seqs) * num_heads * qtiles >= (1ll << 30))
    return PA_ERR_INVALID_ARG;

  const bool bf16 = dtype == PA_BF16;
  CUtensorMap tq, tk, tv;
  const cuuint64_t qdims[3] = {static_cast<cuuint64_t>(head_dim),
                               static_cast<cuuint64_t>(num_heads),
                               static_cast<cuuint64_t>(total_queries)};
  const cuuint64_t qstr[2] = {static_cast<cuuint64_t>(head_dim) * 2,
                              static_cast<cuuint64_t>(head_dim) * 2 * num_heads};
  const cuuint32_t qbox[3] = {64, 1, kQTile};
  const cuuint64_t cdims[2] = {static_cast<cuuint64_t>(head_dim), cache_rows};
  const cuuint64_t cstr[1] = {static_cast<cuuint64_t>(head_dim) * 2};
  // a box is one 16-key chunk, or half of one with 8-token blocks
  const cuuint32_t cbox[2] = {64, block_size >= 16 ? 16u : 8u};
  if (!encode_tensor_map(&tq, bf16, q, 3, qdims, qstr, qbox) ||
      !encode_tensor_map(&tk, bf16, k_cache, 2, cdims, cstr, cbox) ||
      !encode_tensor_map(&tv, bf16, v_cache, 2, cdims, cstr, cbox))
    return PA_ERR_CUDA;

  PrefillParams p{};
  p.seq_order = opts ? opts->seq_order : nullptr;
  p.query_start = query_start;
  p.seq_lens = seq_lens;
  p.block_tables = block_tables;
  p.out = out;
  p.err = error_record;
  p.num_heads = num_heads;
  p.block_size = block_size;
  p.max_blocks = max_blocks_per_seq;
  p.num_blocks = num_blocks;
  p.out_dtype = out_dtype;
  p.total_queries = total_queries;
  p.qscale = scale * kLog2e;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  switch ((bf16 ? 1 : 0) | (head_dim == 64 ? 0 : head_dim == 128 ? 2 : 4)) {
    case 0: return launch_prefill<false, 64>(tq, tk, tv, p, num_seqs, qtiles, st);
    case 1: return launch_prefill<true, 64>(tq, tk, tv, p, num_seqs, qtiles, st);
    case 2: return launch_prefill<false, 128>(tq, tk, tv, p, num_seqs, qtiles, st);
    case 3: return launch_prefill<true, 128>(tq, tk, tv, p, num_seqs, qtiles, st);
    case 4: return launch_prefill<false, 256>(tq, tk, tv, p, num_seqs, qtiles, st);
    default: return launch_prefill<true, 256>(tq, tk, tv, p, num_seqs, qtiles, st);
  }
}
