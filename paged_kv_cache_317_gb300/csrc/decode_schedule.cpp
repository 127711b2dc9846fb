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
// ones (c = 3.5), a 64-token one less still (c = 1).  Measured on GB300 with
// CUDA-graph replays over 39 batches (1 to 512 sequences, medians of 30 to
// 30000 tokens, 40 heads x 128): on average within 1.1 % of the best of
// 32..512 for each batch, at worst 13 % (a 10 us call over 2 short sequences),
// where a fixed 512 is up to 2.4x slower on batches of 1 to 24 sequences.
// Calls with less work than one 64-token block per SM (a few sequences of a
// few hundred tokens and few heads) take 32: 4 sequences of 95 to 191 tokens
// with 8 heads x 64 ran in 12.9 us against 14.7 us at 64, with L2 flushed.
// Whatever balances, the longest sequence is cut into at most kMaxPieces
// partitions (the merge takes up to 32 partials in one load per lane; more go
// through a slower loop): one sequence of 1500 tokens with 8 heads ran 23.4 us
// at 32 (47 partitions) against 18.0 at 64, one of 4000 with 4 heads 36.3 us at
// 32 and 27.3 at 64 against 21.9 at 128.
constexpr int kMaxPieces = 32;
struct Candidate {
  int tokens;
  long long num, den;  // c = num / den
};
constexpr Candidate kCandidates[] = {{512, 7, 2}, {256, 7, 2}, {128, 2, 1}, {64, 1, 1}};
constexpr int kShortest = 32;

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
    // Long sequences start early and the short ones fill the launch's tail:
    // one sort of (longest first, then index) keys, all distinct.
    std::vector<uint64_t> key(static_cast<size_t>(num_seqs));
    for (int i = 0; i < num_seqs; ++i)
      key[i] = (static_cast<uint64_t>(~static_cast<uint32_t>(seq_lens[i])) << 32) |
               static_cast<uint32_t>(i);
    std::sort(key.begin(), key.end());
    for (int k = 0; k < num_seqs; ++k) seqs[k] = static_cast<int32_t>(key[k] & 0xffffffffu);
  }
  return true;
}

// How often each block id occurs among one partition's candidates, in an
// open-addressing table, so that only the candidates whose first block occurs
// more than once (the only ones a record can take) are sorted into runs.
class BlockCounts {
 public:
  void reset(size_t n) {
    size_t cap = 64;
    while (cap < 2 * n) cap <<= 1;
    if (key_.size() < cap) {
      key_.assign(cap, 0);
      count_.assign(cap, 0);
      stamp_.assign(cap, 0);
    }
    mask_ = cap - 1;
    if (++now_ == 0) {  // the generation counter wrapped: forget every stamp
      std::fill(stamp_.begin(), stamp_.end(), 0u);
      now_ = 1;
    }
  }
  void add(int32_t block) {
    const size_t h = find(block);
    if (stamp_[h] != now_) {
      stamp_[h] = now_;
      key_[h] = block;
      count_[h] = 0;
    }
    ++count_[h];
  }
  bool repeated(int32_t block) const {
    const size_t h = find(block);
    return stamp_[h] == now_ && count_[h] > 1;
  }

 private:
  size_t find(int32_t block) const {
    size_t h = (static_cast<uint32_t>(block) * 0x9E3779B1u) & mask_;
    while (stamp_[h] == now_ && key_[h] != block) h = (h + 1) & mask_;
    return h;
  }
  std::vector<int32_t> key_;
  std::vector<int32_t> count_;
  std::vector<uint32_t> stamp_;
  size_t mask_ = 0;
  uint32_t now_ = 0;
};

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
  int pt = kShortest;
  for (const Candidate& c : kCandidates) {
    const long long heaviest = std::min(c.tokens, longest);
    if (c.num * heaviest * num_sms <= c.den * work) {
      pt = c.tokens;
      break;
    }
  }
  // no shorter than needed to keep the longest sequence within kMaxPieces
  // partitions (512 at the most)
  while (pt < kCandidates[0].tokens &&
         (static_cast<long long>(longest) + pt - 1) / pt > kMaxPieces)
    pt *= 2;
  *partition_tokens = pt;
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
  return pa_decode_share_plan_ex(block_tables, seq_lens, num_seqs, max_blocks_per_seq,
                                 block_size, partition_tokens, fused_append, order, 0,
                                 work_items, items_capacity, num_items, records,
                                 records_capacity, num_records, nullptr);
}

extern "C" int pa_decode_share_plan_ex(const int32_t* block_tables, const int32_t* seq_lens,
                                       int num_seqs, int max_blocks_per_seq, int block_size,
                                       int partition_tokens, int fused_append,
                                       const int32_t* order, int prefixes, int32_t* work_items,
                                       int32_t items_capacity, int32_t* num_items,
                                       int32_t* records, int32_t records_capacity,
                                       int32_t* num_records, int32_t* tail_start) {
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
  // candidates are keyed by the partition's first block, and only the runs of
  // an equal first block are compared entry by entry, in two ways:
  //  - whole records: members whose tables agree over the whole partition;
  //  - prefix records (if asked for): of the pairs still in the work list,
  //    groups in run order that share the partition's first c whole 16-token
  //    chunks (below every member's last token); each member keeps the rest of
  //    the partition as its own item, from tail_start on.  One split per
  //    sequence (its tail row in the workspace is single).
  std::vector<int32_t> recs, prefix_recs;
  std::vector<uint64_t> keyed;  // first block of the slice (high word), sequence
  std::vector<int32_t> run, group, cand;
  std::vector<int32_t> tails(static_cast<size_t>(num_seqs), -1);
  BlockCounts counts;
  const long long max_chunks = pt / 16 - 1;  // a prefix leaves at least one chunk's start
  const bool split = prefixes && max_chunks >= 1 && max_chunks < (1ll << 22);
  long long parts_to_scan = most;
  if (split)
    for (int i = 0; i < num_seqs; ++i)
      parts_to_scan = std::max(parts_to_scan, first_part[i + 1] - first_part[i]);
  const auto row = [&](int32_t i) {
    return block_tables + static_cast<size_t>(i) * max_blocks_per_seq;
  };
  const auto key_seq = [](uint64_t k) { return static_cast<int32_t>(k & 0xffffffffu); };
  const auto key_block = [](uint64_t k) { return static_cast<uint32_t>(k >> 32); };
  for (long long part = 0; part < parts_to_scan; ++part) {
    const long long start = part * pt;
    const long long b0 = start / block_size;
    const long long b1 = (start + pt - 1) / block_size;  // inclusive
    const size_t n = static_cast<size_t>(b1 - b0 + 1);
    const auto whole_ok = [&](int32_t i) { return shareable[i] > part; };
    const auto prefix_ok = [&](int32_t i) {
      return split && tails[i] < 0 && part < first_part[i + 1] - first_part[i] &&
             seq_lens[i] - 1 - start >= 16;
    };
    cand.clear();
    for (int i = 0; i < num_seqs; ++i)
      if (whole_ok(i) || prefix_ok(i)) cand.push_back(i);
    counts.reset(cand.size());
    for (int32_t i : cand) counts.add(row(i)[b0]);
    keyed.clear();
    for (int32_t i : cand)
      if (counts.repeated(row(i)[b0]))
        keyed.push_back((static_cast<uint64_t>(static_cast<uint32_t>(row(i)[b0])) << 32) |
                        static_cast<uint32_t>(i));
    std::sort(keyed.begin(), keyed.end());
    for (size_t a = 0; a < keyed.size();) {
      size_t e = a + 1;
      while (e < keyed.size() && key_block(keyed[e]) == key_block(keyed[a])) ++e;
      // whole records: the run's members sorted by their slice of the table
      // (then by index), so that identical slices are adjacent, each group in
      // index order; one sort, whatever the number of distinct slices
      run.clear();
      for (size_t k = a; k < e; ++k)
        if (whole_ok(key_seq(keyed[k]))) run.push_back(key_seq(keyed[k]));
      const auto slice_cmp = [&](int32_t x, int32_t y) {
        return std::memcmp(row(x) + b0, row(y) + b0, n * sizeof(int32_t));
      };
      if (run.size() >= 2)
        std::sort(run.begin(), run.end(), [&](int32_t x, int32_t y) {
          const int c = slice_cmp(x, y);
          return c != 0 ? c < 0 : x < y;
        });
      for (size_t u = 0; u + 1 < run.size();) {
        size_t v = u + 1;
        while (v < run.size() && slice_cmp(run[v], run[u]) == 0) ++v;
        // at most PA_SHARE_MAX_MEMBERS per record; a lone leftover stays private
        for (size_t at = u; at + 1 < v; at += PA_SHARE_MAX_MEMBERS) {
          const size_t m = std::min<size_t>(PA_SHARE_MAX_MEMBERS, v - at);
          recs.push_back(static_cast<int32_t>(part));
          recs.push_back(static_cast<int32_t>(m));
          for (size_t j = 0; j < PA_SHARE_MAX_MEMBERS; ++j)
            recs.push_back(j < m ? run[at + j] : -1);
          for (size_t j = 0; j < m; ++j) covered[first_part[run[at + j]] + part] = 1;
        }
        u = v;
      }
      // prefix records over the run's members still in the work list
      group.clear();
      if (split)
        for (size_t k = a; k < e; ++k) {
          const int32_t i = key_seq(keyed[k]);
          if (prefix_ok(i) && !covered[first_part[i] + part]) group.push_back(i);
        }
      for (size_t at = 0; at + 1 < group.size(); at += PA_SHARE_MAX_MEMBERS) {
        const size_t m = std::min<size_t>(PA_SHARE_MAX_MEMBERS, group.size() - at);
        const int32_t* ref = row(group[at]);
        long long c = max_chunks;
        for (size_t j = 0; j < m; ++j)
          c = std::min<long long>(c, (seq_lens[group[at + j]] - 1 - start) / 16);
        // d: the first block (of those the c chunks touch) where some member's
        // table differs; a chunk is alike when it ends before block d
        long long d = (start + 16 * c - 1) / block_size + 1;
        for (size_t j = 1; j < m && d > b0; ++j)
          d = std::mismatch(ref + b0, ref + d, row(group[at + j]) + b0).first - ref;
        const long long same = std::min(c, (d * block_size - start) / 16);
        if (same < 1) continue;
        prefix_recs.push_back(static_cast<int32_t>(part));
        prefix_recs.push_back(static_cast<int32_t>(m + 256 * same));
        for (size_t j = 0; j < PA_SHARE_MAX_MEMBERS; ++j)
          prefix_recs.push_back(j < m ? group[at + j] : -1);
        for (size_t j = 0; j < m; ++j)
          tails[group[at + j]] = static_cast<int32_t>(start + 16 * same);
      }
      a = e;
    }
  }
  // whole records first: the longer ones start early in the shared pass
  recs.insert(recs.end(), prefix_recs.begin(), prefix_recs.end());
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
  if (tail_start) std::memcpy(tail_start, tails.data(), tails.size() * sizeof(int32_t));
  return PA_OK;
}
