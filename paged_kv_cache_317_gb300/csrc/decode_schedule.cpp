// Host-side decode schedule: the split-K partition length and the list of
// (sequence, partition) work items for one decode launch, built from host
// copies of the sequence lengths (which the host holds anyway: it builds the
// block tables, PagedAttention, zeroshotmind.com page, "Block tables: logical
// order, physical scatter").  No device code and no device memory.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
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

// Sequence indices in launch order: `order` if given (checked to be a
// permutation), else longest first with equal lengths in index order.
bool launch_order(const int32_t* seq_lens, int num_seqs, const int32_t* order,
                  std::vector<int32_t>& seqs) {
  seqs.resize(static_cast<size_t>(num_seqs));
  if (order) {
    std::vector<char> seen(static_cast<size_t>(num_seqs), 0);
    for (int k = 0; k < num_seqs; ++k) {
      const int32_t i = order[k];
      if (i < 0 || i >= num_seqs || seen[i]) return false;
      seen[i] = 1;
      seqs[k] = i;
    }
  } else {
    // Long sequences start early and the short ones fill the launch's tail.
    std::iota(seqs.begin(), seqs.end(), 0);
    std::stable_sort(seqs.begin(), seqs.end(),
                     [&](int32_t a, int32_t b) { return seq_lens[a] > seq_lens[b]; });
  }
  return true;
}

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

  std::vector<int32_t> seqs;
  if (!launch_order(seq_lens, num_seqs, order, seqs)) return PA_ERR_INVALID_ARG;
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

extern "C" int pa_decode_share_plan(const int32_t* block_tables, const int32_t* seq_lens,
                                    int num_seqs, int max_blocks_per_seq, int block_size,
                                    int partition_tokens, int fused_append, const int32_t* order,
                                    int32_t* work_items, int32_t items_capacity,
                                    int32_t* num_items, int32_t* records,
                                    int32_t records_capacity, int32_t* num_records) {
  if (!num_items || !num_records || num_seqs < 0 ||
      (num_seqs > 0 && (!seq_lens || !block_tables)) || max_blocks_per_seq <= 0 ||
      block_size <= 0 || items_capacity < 0 || records_capacity < 0)
    return PA_ERR_INVALID_ARG;
  const int pt = partition_tokens == 0 ? kDefaultPartition : partition_tokens;
  if (!valid_partition(pt)) return PA_ERR_INVALID_ARG;
  const long long cap = static_cast<long long>(max_blocks_per_seq) * block_size;
  if (cap > (1ll << 30)) return PA_ERR_INVALID_ARG;
  const long long P = (cap + pt - 1) / pt;
  if (static_cast<long long>(num_seqs) * P > INT32_MAX) return PA_ERR_INVALID_ARG;
  std::vector<int32_t> seqs;
  if (!launch_order(seq_lens, num_seqs, order, seqs)) return PA_ERR_INVALID_ARG;

  // partitions of each sequence, and how many of them (from the first) a record
  // may take: whole partitions, before the appended token if there is one
  std::vector<long long> first_part(static_cast<size_t>(num_seqs) + 1, 0);
  std::vector<int> shareable(static_cast<size_t>(num_seqs), 0);
  int most = 0;
  for (int i = 0; i < num_seqs; ++i) {
    const int L = seq_lens[i];
    if (L < 0 || L > cap) return PA_ERR_INVALID_ARG;
    first_part[i + 1] = first_part[i] + std::max(1, (L + pt - 1) / pt);
    shareable[i] = std::max(0, (L - (fused_append ? 1 : 0)) / pt);
    most = std::max(most, shareable[i]);
  }
  const long long total = first_part[num_seqs];
  std::vector<char> covered(static_cast<size_t>(total), 0);

  // Group, partition by partition, the sequences whose tables name the same
  // blocks over it.  Sequences share a physical block only through forks, so
  // candidates are sorted by the partition's first block and only runs with an
  // equal first block are compared entry by entry.
  std::vector<int32_t> recs;
  std::vector<std::pair<int32_t, int32_t>> keyed;  // (first block of the slice, sequence)
  std::vector<int32_t> run, group;
  for (int part = 0; part < most; ++part) {
    const long long b0 = static_cast<long long>(part) * pt / block_size;
    const long long b1 = (static_cast<long long>(part + 1) * pt - 1) / block_size;  // inclusive
    const size_t n = static_cast<size_t>(b1 - b0 + 1);
    keyed.clear();
    for (int i = 0; i < num_seqs; ++i)
      if (shareable[i] > part)
        keyed.emplace_back(block_tables[static_cast<size_t>(i) * max_blocks_per_seq + b0], i);
    std::sort(keyed.begin(), keyed.end());
    for (size_t a = 0; a < keyed.size();) {
      size_t e = a + 1;
      while (e < keyed.size() && keyed[e].first == keyed[a].first) ++e;
      if (e - a >= 2) {
        run.clear();
        for (size_t k = a; k < e; ++k) run.push_back(keyed[k].second);
        // split the run into groups of identical slices (members in index order)
        while (run.size() >= 2) {
          const int32_t* ref =
              block_tables + static_cast<size_t>(run[0]) * max_blocks_per_seq + b0;
          group.clear();
          size_t keep = 0;
          for (size_t k = 0; k < run.size(); ++k) {
            const int32_t* slice =
                block_tables + static_cast<size_t>(run[k]) * max_blocks_per_seq + b0;
            if (k == 0 || std::memcmp(slice, ref, n * sizeof(int32_t)) == 0)
              group.push_back(run[k]);
            else
              run[keep++] = run[k];
          }
          run.resize(keep);
          // at most PA_SHARE_MAX_MEMBERS per record; a lone leftover stays private
          for (size_t at = 0; at + 1 < group.size(); at += PA_SHARE_MAX_MEMBERS) {
            const size_t m = std::min<size_t>(PA_SHARE_MAX_MEMBERS, group.size() - at);
            recs.push_back(part);
            recs.push_back(static_cast<int32_t>(m));
            for (size_t j = 0; j < PA_SHARE_MAX_MEMBERS; ++j)
              recs.push_back(j < m ? group[at + j] : -1);
            for (size_t j = 0; j < m; ++j) covered[first_part[group[at + j]] + part] = 1;
          }
        }
      }
      a = e;
    }
  }
  const long long nrec = static_cast<long long>(recs.size()) / PA_SHARE_RECORD_WORDS;
  const long long nitems = total - std::count(covered.begin(), covered.end(), 1);
  if (nrec > INT32_MAX || nitems > INT32_MAX) return PA_ERR_INVALID_ARG;
  *num_items = static_cast<int32_t>(nitems);
  *num_records = static_cast<int32_t>(nrec);
  if (!work_items && !records) return PA_OK;  // size query
  if (!work_items || !records || nitems > items_capacity || nrec > records_capacity)
    return PA_ERR_INVALID_ARG;
  int32_t* w = work_items;
  for (int32_t i : seqs) {
    for (long long part = 0; part < first_part[i + 1] - first_part[i]; ++part)
      if (!covered[first_part[i] + part]) *w++ = static_cast<int32_t>(i * P + part);
  }
  if (!recs.empty()) std::memcpy(records, recs.data(), recs.size() * sizeof(int32_t));
  return PA_OK;
}
