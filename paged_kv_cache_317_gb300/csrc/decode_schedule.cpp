// Host-side decode schedule: the split-K partition length and the list of
// (sequence, partition) work items for one decode launch, built from host
// copies of the sequence lengths (which the host holds anyway: it builds the
// block tables, PagedAttention, zeroshotmind.com page, "Block tables: logical
// order, physical scatter").  No device code and no device memory.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <numeric>
#include <vector>

#include "decode_config.h"
#include "pagedkv.h"

namespace {

// Candidate partition lengths, longest first, each with its balance constant
// c: a candidate is taken when the heaviest block (min(partition, longest
// length) tokens of heads_per_cta heads) is at most 1/c of the work an SM gets
// on average (total tokens x heads / heads_per_cta, over the SMs).  Then every
// SM holds several blocks' worth of work and the last block to start does not
// set the launch's length.  Shorter partitions add merge work and per-block
// start-up cost, so the longest one that balances is best; a 128-token block
// is cheap enough to start that it needs less balance (c = 2) than the longer
// ones (c = 3.5).  Measured on GB300 with CUDA-graph replays over 39 batches
// (1 to 512 sequences, medians of 30 to 30000 tokens, 40 heads x 128): on
// average within 1.1 % of the best of 32..512 for each batch, at worst 13 %
// (a 10 us call over 2 short sequences), where a fixed 512 is up to 2.4x slower
// on batches of 1 to 24 sequences.
struct Candidate {
  int tokens;
  long long num, den;  // c = num / den
};
constexpr Candidate kCandidates[] = {{512, 7, 2}, {256, 7, 2}, {128, 2, 1}};
constexpr int kShortest = 64;

bool valid_partition(int pt) { return pt > 0 && pt % 16 == 0; }

}  // namespace

using namespace pagedkv;

extern "C" int pa_decode_partition_tokens(const int32_t* seq_lens, int num_seqs, int num_heads,
                                          int heads_per_cta, int num_sms,
                                          int32_t* partition_tokens) {
  if (!partition_tokens || num_seqs < 0 || (num_seqs > 0 && !seq_lens) || num_heads <= 0 ||
      heads_per_cta < 0 || num_sms < 0)
    return PA_ERR_INVALID_ARG;
  const int G = heads_per_cta > 0 ? heads_per_cta : auto_heads_per_cta(num_heads);
  if (G > kMaxHeadsPerCta || num_heads % G != 0) return PA_ERR_INVALID_ARG;
  if (num_sms == 0) {
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess ||
        cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
      return PA_ERR_CUDA;
  }
  long long tokens = 0;
  int longest = 0;
  for (int i = 0; i < num_seqs; ++i) {
    if (seq_lens[i] < 0) return PA_ERR_INVALID_ARG;
    tokens += seq_lens[i];
    longest = std::max(longest, static_cast<int>(seq_lens[i]));
  }
  const long long work = tokens * (num_heads / G);
  for (const Candidate& c : kCandidates) {
    const long long heaviest = std::min(c.tokens, longest);
    if (c.num * heaviest * num_sms <= c.den * work) {
      *partition_tokens = c.tokens;
      return PA_OK;
    }
  }
  *partition_tokens = kShortest;
  return PA_OK;
}

extern "C" int pa_decode_work_items(const int32_t* seq_lens, int num_seqs, int partition_tokens,
                                    int max_blocks_per_seq, int block_size, const int32_t* order,
                                    int32_t* items, int32_t capacity, int32_t* num_items) {
  if (!num_items || num_seqs < 0 || (num_seqs > 0 && !seq_lens) || max_blocks_per_seq <= 0 ||
      block_size <= 0 || capacity < 0)
    return PA_ERR_INVALID_ARG;
  const int pt = partition_tokens == 0 ? kDefaultPartition : partition_tokens;
  if (!valid_partition(pt)) return PA_ERR_INVALID_ARG;
  const long long cap = static_cast<long long>(max_blocks_per_seq) * block_size;
  if (cap > (1ll << 30)) return PA_ERR_INVALID_ARG;
  const long long P = (cap + pt - 1) / pt;
  if (static_cast<long long>(num_seqs) * P > INT32_MAX) return PA_ERR_INVALID_ARG;

  std::vector<int32_t> seqs(static_cast<size_t>(num_seqs));
  if (order) {
    std::vector<char> seen(static_cast<size_t>(num_seqs), 0);
    for (int k = 0; k < num_seqs; ++k) {
      const int32_t i = order[k];
      if (i < 0 || i >= num_seqs || seen[i]) return PA_ERR_INVALID_ARG;
      seen[i] = 1;
      seqs[k] = i;
    }
  } else {
    // Longest first, ties in index order: long sequences start early and the
    // short ones fill the launch's tail.
    std::iota(seqs.begin(), seqs.end(), 0);
    std::stable_sort(seqs.begin(), seqs.end(),
                     [&](int32_t a, int32_t b) { return seq_lens[a] > seq_lens[b]; });
  }
  long long count = 0;
  for (int i = 0; i < num_seqs; ++i) {
    if (seq_lens[i] < 0 || seq_lens[i] > cap) return PA_ERR_INVALID_ARG;
    count += std::max<long long>(1, (seq_lens[i] + pt - 1) / pt);
  }
  if (count > INT32_MAX) return PA_ERR_INVALID_ARG;
  *num_items = static_cast<int32_t>(count);
  if (!items) return PA_OK;  // size query
  if (count > capacity) return PA_ERR_INVALID_ARG;
  int32_t* w = items;
  for (int32_t i : seqs) {
    const long long parts = std::max<long long>(1, (seq_lens[i] + pt - 1) / pt);
    for (long long p = 0; p < parts; ++p) *w++ = static_cast<int32_t>(i * P + p);
  }
  return PA_OK;
}
