// A decode step driven through the C ABI alone (include/pagedkv.h and
// libpagedkv.so; no Python): host allocator, KV append, copy-on-write block
// copy, the host decode schedule (and a second plan that reads the blocks a
// fork shares with its parent once for both), paged decode attention and a
// chunked prefill over the same cache.  It checks two exact properties on both
// decodes (the first also on the prefill):
//  * a sequence forked from another and given the same next token (or the same
//    queries) gives the same bits as its parent, although its last block is a
//    private copy;
//  * a one-token sequence decodes to its value row exactly (one weight of 1);
// and that the prefill's queries that repeat the decode's match its output
// within 2e-3.
// Build: nvcc -std=c++17 -I include c_abi_step.cu -L<dir> -lpagedkv -o c_abi_step
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <vector>

#include "pagedkv.h"

namespace {

constexpr int kHeads = 4, kDim = 128, kBlock = 16, kBlocks = 64, kMaxBlocks = 8;

#define CHECK(call)                                                                 \
  do {                                                                              \
    const int st_ = (call);                                                         \
    if (st_ != 0) {                                                                 \
      std::fprintf(stderr, "%s failed: %d (%s)\n", #call, st_, pa_status_string(st_)); \
      return 1;                                                                     \
    }                                                                               \
  } while (0)
#define CUDA(call)                                                                  \
  do {                                                                              \
    const cudaError_t e_ = (call);                                                  \
    if (e_ != cudaSuccess) {                                                        \
      std::fprintf(stderr, "%s: %s\n", #call, cudaGetErrorString(e_));            \
      return 1;                                                                     \
    }                                                                               \
  } while (0)

// Deterministic values in [-1, 1) (a 32-bit linear congruential sequence).
struct Lcg {
  uint32_t s;
  float next() {
    s = s * 1664525u + 1013904223u;
    return static_cast<float>(s >> 8) / 8388608.0f - 1.0f;
  }
};

std::vector<__half> random_rows(Lcg& g, int rows) {
  std::vector<__half> v(static_cast<size_t>(rows) * kHeads * kDim);
  for (auto& x : v) x = __float2half(g.next());
  return v;
}

}  // namespace

int main() {
  std::printf("libpagedkv version %d\n", pa_version());
  if (pa_version() != PAGEDKV_VERSION) {   // the option structs differ between versions
    std::fprintf(stderr, "built against version %d\n", PAGEDKV_VERSION);
    return 1;
  }
  pa_allocator* alloc = pa_alloc_create(kBlocks, kBlock, nullptr);
  if (!alloc) return 1;

  // sequence 0: a 37-token prompt; sequence 2: one token; sequence 1 = fork of 0
  const int prompt = 37;
  CHECK(pa_seq_add(alloc, 0, prompt));
  CHECK(pa_seq_add(alloc, 2, 1));
  CHECK(pa_seq_fork(alloc, 0, 1));
  std::vector<int64_t> slots(prompt + 1);
  CHECK(pa_seq_slots(alloc, 0, 0, prompt, slots.data()));
  CHECK(pa_seq_slots(alloc, 2, 0, 1, slots.data() + prompt));

  Lcg g{12345u};
  const std::vector<__half> k0 = random_rows(g, prompt + 1), v0 = random_rows(g, prompt + 1);
  const size_t row = static_cast<size_t>(kHeads) * kDim;
  const size_t cache_elems = static_cast<size_t>(kBlocks) * kHeads * kBlock * kDim;

  __half *kc, *vc, *k, *v, *q;
  int64_t* slot_d;
  int64_t* pair_d;
  int32_t *tables_d, *lens_d, *rec;
  float* out;
  CUDA(cudaMalloc(&kc, cache_elems * sizeof(__half)));
  CUDA(cudaMalloc(&vc, cache_elems * sizeof(__half)));
  CUDA(cudaMemset(kc, 0, cache_elems * sizeof(__half)));
  CUDA(cudaMemset(vc, 0, cache_elems * sizeof(__half)));
  CUDA(cudaMalloc(&k, (prompt + 1) * row * sizeof(__half)));
  CUDA(cudaMalloc(&v, (prompt + 1) * row * sizeof(__half)));
  CUDA(cudaMalloc(&slot_d, (prompt + 1) * sizeof(int64_t)));
  CUDA(cudaMalloc(&pair_d, 2 * sizeof(int64_t)));
  CUDA(cudaMalloc(&q, 3 * row * sizeof(__half)));
  CUDA(cudaMalloc(&tables_d, 3 * kMaxBlocks * sizeof(int32_t)));
  CUDA(cudaMalloc(&lens_d, 3 * sizeof(int32_t)));
  CUDA(cudaMalloc(&out, 3 * row * sizeof(float)));
  CUDA(cudaMalloc(&rec, 4 * sizeof(int32_t)));
  CHECK(pa_error_clear(rec, nullptr));

  CUDA(cudaMemcpy(k, k0.data(), k0.size() * sizeof(__half), cudaMemcpyHostToDevice));
  CUDA(cudaMemcpy(v, v0.data(), v0.size() * sizeof(__half), cudaMemcpyHostToDevice));
  CUDA(cudaMemcpy(slot_d, slots.data(), slots.size() * sizeof(int64_t), cudaMemcpyHostToDevice));
  CHECK(kv_cache_append(k, v, slot_d, prompt + 1, kc, vc, kHeads, kDim, kBlock, kBlocks, PA_F16,
                        rec, nullptr));

  // Both holders of the shared partial block append the same new token: the
  // fork first (it gets a private copy of that block), then the parent (now the
  // sole holder, it writes in place).
  int64_t slot1, slot0;
  int32_t src, dst, src0, dst0;
  CHECK(pa_seq_append(alloc, 1, &slot1, &src, &dst));
  CHECK(pa_seq_append(alloc, 0, &slot0, &src0, &dst0));
  if (src < 0 || src0 >= 0) {
    std::fprintf(stderr, "expected exactly one copy-on-write (got %d, %d)\n", src, src0);
    return 1;
  }
  const int64_t pair[2] = {src, dst};
  CUDA(cudaMemcpy(pair_d, pair, sizeof(pair), cudaMemcpyHostToDevice));
  void* kcs[1] = {kc};
  void* vcs[1] = {vc};
  CHECK(block_copy(kcs, vcs, 1, pair_d, 1, kHeads, kDim, kBlock, kBlocks, PA_F16, rec, nullptr));
  const std::vector<__half> kn = random_rows(g, 1), vn = random_rows(g, 1);
  const int64_t new_slots[2] = {slot1, slot0};
  for (int i = 0; i < 2; ++i) {
    CUDA(cudaMemcpy(k + i * row, kn.data(), row * sizeof(__half), cudaMemcpyHostToDevice));
    CUDA(cudaMemcpy(v + i * row, vn.data(), row * sizeof(__half), cudaMemcpyHostToDevice));
  }
  CUDA(cudaMemcpy(slot_d, new_slots, sizeof(new_slots), cudaMemcpyHostToDevice));
  CHECK(kv_cache_append(k, v, slot_d, 2, kc, vc, kHeads, kDim, kBlock, kBlocks, PA_F16, rec,
                        nullptr));

  // tables and lengths of sequences 0, 1, 2
  std::vector<int32_t> tables(3 * kMaxBlocks, -1), lens(3);
  for (int s = 0; s < 3; ++s) {
    int32_t nb = 0;
    CHECK(pa_seq_block_table(alloc, s, tables.data() + s * kMaxBlocks, kMaxBlocks, &nb));
    CHECK(pa_seq_len(alloc, s, &lens[s]));
  }
  CUDA(cudaMemcpy(tables_d, tables.data(), tables.size() * 4, cudaMemcpyHostToDevice));
  CUDA(cudaMemcpy(lens_d, lens.data(), lens.size() * 4, cudaMemcpyHostToDevice));

  // the same query for sequences 0 and 1
  std::vector<__half> qh = random_rows(g, 3);
  std::memcpy(qh.data() + row, qh.data(), row * sizeof(__half));
  CUDA(cudaMemcpy(q, qh.data(), qh.size() * sizeof(__half), cudaMemcpyHostToDevice));
  // split-K partition length and (sequence, partition) work list from the host
  // lengths: a batch this small gets short partitions, so the split path runs
  int32_t pt = 0, n_items = 0;
  CHECK(pa_decode_partition_tokens(lens.data(), 3, kHeads, 0, 0, &pt));
  CHECK(pa_decode_work_items(lens.data(), 3, pt, kMaxBlocks, kBlock, nullptr, nullptr, 0,
                             &n_items));
  std::vector<int32_t> items(n_items);
  CHECK(pa_decode_work_items(lens.data(), 3, pt, kMaxBlocks, kBlock, nullptr, items.data(),
                             n_items, &n_items));
  int32_t* items_d = nullptr;
  CUDA(cudaMalloc(&items_d, items.size() * sizeof(int32_t)));
  CUDA(cudaMemcpy(items_d, items.data(), items.size() * sizeof(int32_t), cudaMemcpyHostToDevice));
  pa_decode_opts opts{};
  opts.work_items = items_d;
  opts.num_work_items = n_items;
  const size_t ws = paged_attn_workspace_size(3, kHeads, kDim, kBlock, kMaxBlocks, pt);
  void* workspace = nullptr;
  if (ws) CUDA(cudaMalloc(&workspace, ws));
  CHECK(paged_attn_decode_ex(q, kc, vc, tables_d, lens_d, 3, kHeads, kDim, kBlock, kMaxBlocks,
                             kBlocks, 1.0f / 11.3137085f, PA_F16, out, PA_F32, pt, workspace, ws,
                             rec, nullptr, &opts));
  CUDA(cudaDeviceSynchronize());
  int32_t err[4];
  CHECK(pa_error_read(rec, err, nullptr));
  if (err[0] != 0) {
    std::fprintf(stderr, "device error record: %d %d %d %d\n", err[0], err[1], err[2], err[3]);
    return 1;
  }

  std::vector<float> o(3 * row);
  CUDA(cudaMemcpy(o.data(), out, o.size() * sizeof(float), cudaMemcpyDeviceToHost));
  if (std::memcmp(o.data(), o.data() + row, row * sizeof(float)) != 0) {
    std::fprintf(stderr, "forked sequence decodes differently from its parent\n");
    return 1;
  }
  for (size_t i = 0; i < row; ++i) {
    if (o[2 * row + i] != __half2float(v0[prompt * row + i])) {
      std::fprintf(stderr, "one-token sequence: element %zu is %g, value row holds %g\n", i,
                   o[2 * row + i], __half2float(v0[prompt * row + i]));
      return 1;
    }
  }

  // The same decode with 16-token partitions, reading the two full blocks that
  // sequence 0 and its fork share once for both (pa_decode_share_plan records).
  const int pt2 = 16;
  int32_t n_items2 = 0, n_recs = 0;
  CHECK(pa_decode_share_plan(tables.data(), lens.data(), 3, kMaxBlocks, kBlock, pt2, 0, nullptr,
                             nullptr, 0, &n_items2, nullptr, 0, &n_recs));
  std::vector<int32_t> items2(n_items2), recs(static_cast<size_t>(n_recs) * PA_SHARE_RECORD_WORDS);
  CHECK(pa_decode_share_plan(tables.data(), lens.data(), 3, kMaxBlocks, kBlock, pt2, 0, nullptr,
                             items2.data(), n_items2, &n_items2, recs.data(), n_recs, &n_recs));
  if (n_recs != 2 || recs[1] != 2) {
    std::fprintf(stderr, "expected 2 shared records of 2 members, got %d\n", n_recs);
    return 1;
  }
  int32_t *items2_d = nullptr, *recs_d = nullptr;
  CUDA(cudaMalloc(&items2_d, items2.size() * sizeof(int32_t)));
  CUDA(cudaMalloc(&recs_d, recs.size() * sizeof(int32_t)));
  CUDA(cudaMemcpy(items2_d, items2.data(), items2.size() * sizeof(int32_t), cudaMemcpyHostToDevice));
  CUDA(cudaMemcpy(recs_d, recs.data(), recs.size() * sizeof(int32_t), cudaMemcpyHostToDevice));
  pa_decode_opts opts2{};
  opts2.work_items = items2_d;
  opts2.num_work_items = n_items2;
  opts2.shared_records = recs_d;
  opts2.num_shared = n_recs;
  const size_t ws2 = paged_attn_workspace_size(3, kHeads, kDim, kBlock, kMaxBlocks, pt2);
  void* workspace2 = nullptr;
  float* out2 = nullptr;
  if (ws2) CUDA(cudaMalloc(&workspace2, ws2));
  CUDA(cudaMalloc(&out2, o.size() * sizeof(float)));
  CHECK(paged_attn_decode_ex(q, kc, vc, tables_d, lens_d, 3, kHeads, kDim, kBlock, kMaxBlocks,
                             kBlocks, 1.0f / 11.3137085f, PA_F16, out2, PA_F32, pt2, workspace2,
                             ws2, rec, nullptr, &opts2));
  CUDA(cudaDeviceSynchronize());
  CHECK(pa_error_read(rec, err, nullptr));
  if (err[0] != 0) {
    std::fprintf(stderr, "device error record (shared): %d %d %d %d\n", err[0], err[1], err[2],
                 err[3]);
    return 1;
  }
  std::vector<float> o2(3 * row);
  CUDA(cudaMemcpy(o2.data(), out2, o2.size() * sizeof(float), cudaMemcpyDeviceToHost));
  if (std::memcmp(o2.data(), o2.data() + row, row * sizeof(float)) != 0) {
    std::fprintf(stderr, "shared blocks: fork decodes differently from its parent\n");
    return 1;
  }
  for (size_t i = 0; i < row; ++i) {
    if (o2[2 * row + i] != o[2 * row + i]) {
      std::fprintf(stderr, "shared blocks: one-token sequence changed at element %zu\n", i);
      return 1;
    }
  }
  float worst = 0.f;
  for (size_t i = 0; i < o.size(); ++i) worst = std::max(worst, std::fabs(o2[i] - o[i]));
  if (!(worst <= 2e-3f)) {
    std::fprintf(stderr, "shared blocks: output moved by %g from the first decode\n", worst);
    return 1;
  }

  // Prefix records with 64-token partitions (pa_decode_share_plan_ex): the first
  // two 16-token chunks of the partition, which sequence 0 and its fork share,
  // are read once for both; each reads its own tokens from tail_start on, and the
  // merge adds the two parts.  The lists' lengths are given on the device
  // (pa_decode_opts.counts), as a call replayed from a CUDA graph would.
  const int pt3 = 64;
  int32_t n_items3 = 0, n_recs3 = 0;
  std::vector<int32_t> tails(3, 0);
  CHECK(pa_decode_share_plan_ex(tables.data(), lens.data(), 3, kMaxBlocks, kBlock, pt3, 0,
                                nullptr, 1, nullptr, 0, &n_items3, nullptr, 0, &n_recs3,
                                nullptr));
  std::vector<int32_t> items3(n_items3),
      recs3(static_cast<size_t>(n_recs3) * PA_SHARE_RECORD_WORDS);
  CHECK(pa_decode_share_plan_ex(tables.data(), lens.data(), 3, kMaxBlocks, kBlock, pt3, 0,
                                nullptr, 1, items3.data(), n_items3, &n_items3, recs3.data(),
                                n_recs3, &n_recs3, tails.data()));
  if (n_recs3 != 1 || recs3[1] != 2 + 256 * 2 || tails[0] != 32 || tails[1] != 32 ||
      tails[2] != -1) {
    std::fprintf(stderr, "expected one prefix record of 2 members over 2 chunks, got %d\n",
                 n_recs3);
    return 1;
  }
  const int32_t counts3[2] = {n_items3, n_recs3};
  int32_t *items3_d = nullptr, *recs3_d = nullptr, *tails_d = nullptr, *counts3_d = nullptr;
  CUDA(cudaMalloc(&items3_d, items3.size() * sizeof(int32_t)));
  CUDA(cudaMalloc(&recs3_d, recs3.size() * sizeof(int32_t)));
  CUDA(cudaMalloc(&tails_d, tails.size() * sizeof(int32_t)));
  CUDA(cudaMalloc(&counts3_d, sizeof(counts3)));
  CUDA(cudaMemcpy(items3_d, items3.data(), items3.size() * sizeof(int32_t), cudaMemcpyHostToDevice));
  CUDA(cudaMemcpy(recs3_d, recs3.data(), recs3.size() * sizeof(int32_t), cudaMemcpyHostToDevice));
  CUDA(cudaMemcpy(tails_d, tails.data(), tails.size() * sizeof(int32_t), cudaMemcpyHostToDevice));
  CUDA(cudaMemcpy(counts3_d, counts3, sizeof(counts3), cudaMemcpyHostToDevice));
  pa_decode_opts opts3{};
  opts3.work_items = items3_d;
  opts3.num_work_items = n_items3;
  opts3.shared_records = recs3_d;
  opts3.num_shared = n_recs3;
  opts3.tail_start = tails_d;
  opts3.counts = counts3_d;
  const size_t ws3 = paged_attn_workspace_size_tails(3, kHeads, kDim, kBlock, kMaxBlocks, pt3);
  void* workspace3 = nullptr;
  float* out3 = nullptr;
  CUDA(cudaMalloc(&workspace3, ws3));
  CUDA(cudaMalloc(&out3, o.size() * sizeof(float)));
  CHECK(paged_attn_decode_ex(q, kc, vc, tables_d, lens_d, 3, kHeads, kDim, kBlock, kMaxBlocks,
                             kBlocks, 1.0f / 11.3137085f, PA_F16, out3, PA_F32, pt3, workspace3,
                             ws3, rec, nullptr, &opts3));
  CUDA(cudaDeviceSynchronize());
  CHECK(pa_error_read(rec, err, nullptr));
  if (err[0] != 0) {
    std::fprintf(stderr, "device error record (prefix records): %d %d %d %d\n", err[0], err[1],
                 err[2], err[3]);
    return 1;
  }
  std::vector<float> o3(3 * row);
  CUDA(cudaMemcpy(o3.data(), out3, o3.size() * sizeof(float), cudaMemcpyDeviceToHost));
  if (std::memcmp(o3.data(), o3.data() + row, row * sizeof(float)) != 0 ||
      std::memcmp(o3.data() + 2 * row, o.data() + 2 * row, row * sizeof(float)) != 0) {
    std::fprintf(stderr, "prefix records: fork or one-token sequence changed\n");
    return 1;
  }
  float worst3 = 0.f;
  for (size_t i = 0; i < o.size(); ++i) worst3 = std::max(worst3, std::fabs(o3[i] - o[i]));
  if (!(worst3 <= 2e-3f)) {
    std::fprintf(stderr, "prefix records: output moved by %g from the first decode\n", worst3);
    return 1;
  }

  // Chunked prefill on the tensor cores over the same cache: the last 5 tokens
  // of sequence 0 and of its fork as causal queries (the same 5 query rows for
  // both, the last one the decode's query), and sequence 2's one token with the
  // decode's query.  The fork must give its parent's bits, and the queries that
  // repeat a decode's query its output within 2e-3 (the one-token row is not
  // exact here: the tile's reference max is the product s * scale rounded once,
  // so the single weight is 2^(rounding error), not exactly 1).
  const int nq = 5, total_q = 2 * nq + 1;
  std::vector<__half> qp = random_rows(g, total_q);
  std::memcpy(qp.data() + (nq - 1) * row, qh.data(), row * sizeof(__half));
  std::memcpy(qp.data() + nq * row, qp.data(), nq * row * sizeof(__half));
  std::memcpy(qp.data() + 2 * nq * row, qh.data() + 2 * row, row * sizeof(__half));
  const int32_t qstart[4] = {0, nq, 2 * nq, total_q};
  __half* qp_d = nullptr;
  int32_t* qstart_d = nullptr;
  float* outp = nullptr;
  CUDA(cudaMalloc(&qp_d, qp.size() * sizeof(__half)));
  CUDA(cudaMalloc(&qstart_d, sizeof(qstart)));
  CUDA(cudaMalloc(&outp, static_cast<size_t>(total_q) * row * sizeof(float)));
  CUDA(cudaMemcpy(qp_d, qp.data(), qp.size() * sizeof(__half), cudaMemcpyHostToDevice));
  CUDA(cudaMemcpy(qstart_d, qstart, sizeof(qstart), cudaMemcpyHostToDevice));
  CHECK(paged_attn_prefill(qp_d, qstart_d, total_q, nq, kc, vc, tables_d, lens_d, 3, kHeads, kDim,
                           kBlock, kMaxBlocks, kBlocks, 1.0f / 11.3137085f, PA_F16, outp, PA_F32,
                           rec, nullptr));
  CUDA(cudaDeviceSynchronize());
  CHECK(pa_error_read(rec, err, nullptr));
  if (err[0] != 0) {
    std::fprintf(stderr, "device error record (prefill): %d %d %d %d\n", err[0], err[1], err[2],
                 err[3]);
    return 1;
  }
  std::vector<float> op(static_cast<size_t>(total_q) * row);
  CUDA(cudaMemcpy(op.data(), outp, op.size() * sizeof(float), cudaMemcpyDeviceToHost));
  if (std::memcmp(op.data(), op.data() + nq * row, nq * row * sizeof(float)) != 0) {
    std::fprintf(stderr, "prefill: fork differs from its parent\n");
    return 1;
  }
  float worst_p = 0.f;
  for (size_t i = 0; i < row; ++i) {
    worst_p = std::max(worst_p, std::fabs(op[(nq - 1) * row + i] - o[i]));
    worst_p = std::max(worst_p, std::fabs(op[2 * nq * row + i] - o[2 * row + i]));
  }
  if (!(worst_p <= 2e-3f)) {
    std::fprintf(stderr, "prefill: differs from the decode by %g\n", worst_p);
    return 1;
  }

  CHECK(pa_alloc_check(alloc));
  pa_alloc_destroy(alloc);
  for (void* p : {static_cast<void*>(kc), static_cast<void*>(vc), static_cast<void*>(k),
                  static_cast<void*>(v), static_cast<void*>(q), static_cast<void*>(slot_d),
                  static_cast<void*>(pair_d), static_cast<void*>(tables_d),
                  static_cast<void*>(lens_d), static_cast<void*>(out), static_cast<void*>(rec),
                  static_cast<void*>(items_d), workspace, static_cast<void*>(items2_d),
                  static_cast<void*>(recs_d), workspace2, static_cast<void*>(out2),
                  static_cast<void*>(qp_d), static_cast<void*>(qstart_d),
                  static_cast<void*>(outp), static_cast<void*>(items3_d),
                  static_cast<void*>(recs3_d), static_cast<void*>(tails_d),
                  static_cast<void*>(counts3_d), workspace3, static_cast<void*>(out3)})
    if (p) cudaFree(p);
  std::printf("ok: fork decodes like its parent (one copy-on-write), one-token sequence exact; "
              "%d-token partitions, %d work items; shared blocks read once: %d records, fork "
              "still exact, max change %.2e; prefix records: %d record over 2 chunks, fork "
              "exact, max change %.2e; prefill: fork exact, within %.2e of the decode\n",
              pt, n_items, n_recs, worst, n_recs3, worst3, worst_p);
  return 0;
}
