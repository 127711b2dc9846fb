// Host block allocator for the paged KV cache (PagedAttention, zeroshotmind.com
// page: "Paging the cache" - blocks granted one at a time as a sequence grows;
// "Block tables" - a per-sequence table of physical blocks in logical order;
// "Sharing a prefix without copying it" - per-block reference counts and
// copy-on-write of the one block being written).
//
// Plain C++17, no device code.  The free list is a stack (vector back = top);
// blocks are first handed out in the caller's free_order, freed blocks go back
// on top.  Per-sequence state lives in a hash map keyed by the caller's int64 id.
#include <algorithm>
#include <cstdint>
#include <new>
#include <utility>
#include <unordered_map>
#include <vector>

#include "pagedkv.h"

struct pa_allocator {
  struct Seq {
    std::vector<int32_t> blocks;
    int32_t len = 0;
  };
  using Map = std::unordered_map<int64_t, Seq>;
  int32_t num_blocks = 0;
  int32_t block_size = 0;
  std::vector<int32_t> free_stack;
  std::vector<int32_t> refcount;
  Map seqs;
  // Map nodes of freed sequences, kept for reuse with their block vectors'
  // capacity: a loop that forks and frees about as many sequences per step (beam
  // search) then allocates no host memory in steady state.
  std::vector<Map::node_type> spare;
  static constexpr size_t kMaxSpare = size_t(1) << 16;

  // A new, empty sequence `id` (the caller checked that it does not exist).
  Seq& make(int64_t id) {
    if (!spare.empty()) {
      Map::node_type nh = std::move(spare.back());
      spare.pop_back();
      nh.key() = id;
      nh.mapped().blocks.clear();
      nh.mapped().len = 0;
      return seqs.insert(std::move(nh)).position->second;
    }
    return seqs.emplace(id, Seq{}).first->second;
  }
  // Drop a sequence whose blocks were released; its node goes to `spare`.
  void retire(Map::iterator it) {
    Map::node_type nh = seqs.extract(it);
    if (spare.size() < kMaxSpare) spare.push_back(std::move(nh));
  }

  int32_t take() {
    const int32_t b = free_stack.back();
    free_stack.pop_back();
    refcount[b] = 1;
    return b;
  }
  bool release(int32_t b) {
    if (refcount[b] <= 0) return false;
    if (--refcount[b] == 0) free_stack.push_back(b);
    return true;
  }
  int32_t blocks_for(int64_t tokens) const {
    return static_cast<int32_t>((tokens + block_size - 1) / block_size);
  }
  // Blocks one append to `s` may take: a fresh block at a block boundary, or a
  // copy when the partly filled tail is shared.
  int worst_case_take(const Seq& s) const {
    const int32_t row = s.len % block_size;
    if (row == 0) return 1;
    return refcount[s.blocks[s.len / block_size]] > 1 ? 1 : 0;
  }
  int append(Seq& s, int64_t* slot, int32_t* cow_src, int32_t* cow_dst) {
    const int32_t j = s.len / block_size;
    const int32_t row = s.len % block_size;
    int32_t src = -1, dst = -1;
    if (row == 0) {
      if (free_stack.empty()) return PA_ERR_OOM;
      s.blocks.push_back(take());
    } else {
      const int32_t b = s.blocks[j];
      if (refcount[b] > 1) {
        if (free_stack.empty()) return PA_ERR_OOM;
        const int32_t d = take();
        --refcount[b];
        s.blocks[j] = d;
        src = b;
        dst = d;
      }
    }
    ++s.len;
    if (slot) *slot = static_cast<int64_t>(s.blocks[j]) * block_size + row;
    if (cow_src) *cow_src = src;
    if (cow_dst) *cow_dst = dst;
    return PA_OK;
  }
};

extern "C" pa_allocator* pa_alloc_create(int32_t num_blocks, int32_t block_size,
                                         const int32_t* free_order) {
  if (num_blocks <= 0 || block_size <= 0) return nullptr;
  pa_allocator* a = new (std::nothrow) pa_allocator();
  if (!a) return nullptr;
  try {
    a->num_blocks = num_blocks;
    a->block_size = block_size;
    a->refcount.assign(num_blocks, 0);
    a->free_stack.resize(num_blocks);
    if (free_order) {
      std::vector<char> seen(num_blocks, 0);
      for (int32_t i = 0; i < num_blocks; ++i) {
        const int32_t b = free_order[i];
        if (b < 0 || b >= num_blocks || seen[b]) {
          delete a;
          return nullptr;
        }
        seen[b] = 1;
      }
    }
    // free_order[0] must be handed out first, so it goes on top (the back).
    for (int32_t i = 0; i < num_blocks; ++i)
      a->free_stack[num_blocks - 1 - i] = free_order ? free_order[i] : i;
  } catch (...) {
    delete a;
    return nullptr;
  }
  return a;
}

extern "C" void pa_alloc_destroy(pa_allocator* a) { delete a; }

extern "C" int pa_seq_add(pa_allocator* a, int64_t seq, int32_t num_tokens) {
  if (!a || num_tokens < 0) return PA_ERR_INVALID_ARG;
  if (a->seqs.count(seq)) return PA_ERR_SEQ_EXISTS;
  const int32_t need = a->blocks_for(num_tokens);
  if (need > static_cast<int32_t>(a->free_stack.size())) return PA_ERR_OOM;
  try {
    pa_allocator::Seq& s = a->make(seq);
    s.blocks.reserve(need);
    for (int32_t i = 0; i < need; ++i) s.blocks.push_back(a->take());
    s.len = num_tokens;
  } catch (...) {
    return PA_ERR_OOM;
  }
  return PA_OK;
}

extern "C" int pa_seq_fork(pa_allocator* a, int64_t parent, int64_t child) {
  if (!a) return PA_ERR_INVALID_ARG;
  auto it = a->seqs.find(parent);
  if (it == a->seqs.end()) return PA_ERR_NO_SEQ;
  if (a->seqs.count(child)) return PA_ERR_SEQ_EXISTS;
  try {
    const pa_allocator::Seq& p = it->second;  // element references survive rehashing
    pa_allocator::Seq& c = a->make(child);
    c.blocks = p.blocks;
    c.len = p.len;
    for (int32_t b : c.blocks) ++a->refcount[b];
  } catch (...) {
    return PA_ERR_OOM;
  }
  return PA_OK;
}

extern "C" int pa_seq_append(pa_allocator* a, int64_t seq, int64_t* slot, int32_t* cow_src,
                             int32_t* cow_dst) {
  if (!a) return PA_ERR_INVALID_ARG;
  auto it = a->seqs.find(seq);
  if (it == a->seqs.end()) return PA_ERR_NO_SEQ;
  return a->append(it->second, slot, cow_src, cow_dst);
}

extern "C" int pa_seq_free(pa_allocator* a, int64_t seq) {
  if (!a) return PA_ERR_INVALID_ARG;
  auto it = a->seqs.find(seq);
  if (it == a->seqs.end()) return PA_ERR_NO_SEQ;
  int status = PA_OK;
  for (int32_t b : it->second.blocks)
    if (!a->release(b)) status = PA_ERR_REFCOUNT;
  a->retire(it);
  return status;
}

extern "C" int pa_seq_len(const pa_allocator* a, int64_t seq, int32_t* len) {
  if (!a || !len) return PA_ERR_INVALID_ARG;
  auto it = a->seqs.find(seq);
  if (it == a->seqs.end()) return PA_ERR_NO_SEQ;
  *len = it->second.len;
  return PA_OK;
}

extern "C" int pa_seq_block_table(const pa_allocator* a, int64_t seq, int32_t* out,
                                  int32_t capacity, int32_t* num_blocks) {
  if (!a || capacity < 0 || (capacity > 0 && !out)) return PA_ERR_INVALID_ARG;
  auto it = a->seqs.find(seq);
  if (it == a->seqs.end()) return PA_ERR_NO_SEQ;
  const auto& blocks = it->second.blocks;
  const int32_t n = static_cast<int32_t>(blocks.size());
  std::copy(blocks.begin(), blocks.begin() + std::min(n, capacity), out);
  if (num_blocks) *num_blocks = n;
  return PA_OK;
}

extern "C" int pa_seq_slots(const pa_allocator* a, int64_t seq, int32_t start, int32_t count,
                            int64_t* slots) {
  if (!a || start < 0 || count < 0 || (count > 0 && !slots)) return PA_ERR_INVALID_ARG;
  auto it = a->seqs.find(seq);
  if (it == a->seqs.end()) return PA_ERR_NO_SEQ;
  const auto& s = it->second;
  if (static_cast<int64_t>(start) + count > s.len) return PA_ERR_INVALID_ARG;
  for (int32_t i = 0; i < count; ++i) {
    const int32_t pos = start + i;
    slots[i] = static_cast<int64_t>(s.blocks[pos / a->block_size]) * a->block_size +
               pos % a->block_size;
  }
  return PA_OK;
}

extern "C" int pa_block_refcount(const pa_allocator* a, int32_t block, int32_t* refcount) {
  if (!a || !refcount || block < 0 || block >= a->num_blocks) return PA_ERR_INVALID_ARG;
  *refcount = a->refcount[block];
  return PA_OK;
}

extern "C" int32_t pa_num_free_blocks(const pa_allocator* a) {
  return a ? static_cast<int32_t>(a->free_stack.size()) : -1;
}

extern "C" int32_t pa_num_seqs(const pa_allocator* a) {
  return a ? static_cast<int32_t>(a->seqs.size()) : -1;
}

extern "C" int pa_batch_append(pa_allocator* a, const int64_t* seqs, int32_t n, int64_t* slots,
                               int64_t* cow_pairs, int32_t* num_cow) {
  if (!a || n < 0 || (n > 0 && (!seqs || !slots || !cow_pairs)) || !num_cow)
    return PA_ERR_INVALID_ARG;
  // Resolve every id and bound the blocks needed before changing anything.  A
  // sequence listed twice is counted twice, which only over-estimates.
  std::vector<pa_allocator::Seq*> ptrs(n);
  long long worst = 0;
  for (int32_t i = 0; i < n; ++i) {
    auto it = a->seqs.find(seqs[i]);
    if (it == a->seqs.end()) return PA_ERR_NO_SEQ;
    ptrs[i] = &it->second;
    worst += a->worst_case_take(it->second);
  }
  // A later append of a listed sequence may open a block the first one did not
  // need; count one extra block per repeated id.
  {
    std::vector<int64_t> ids(seqs, seqs + n);
    std::sort(ids.begin(), ids.end());
    for (int32_t i = 1; i < n; ++i)
      if (ids[i] == ids[i - 1]) ++worst;
  }
  if (worst > static_cast<long long>(a->free_stack.size())) return PA_ERR_OOM;
  int32_t nc = 0;
  for (int32_t i = 0; i < n; ++i) {
    int32_t src, dst;
    const int st = a->append(*ptrs[i], &slots[i], &src, &dst);
    if (st != PA_OK) return st;  // unreachable: capacity checked above
    if (src >= 0) {
      cow_pairs[2 * nc] = src;
      cow_pairs[2 * nc + 1] = dst;
      ++nc;
    }
  }
  *num_cow = nc;
  return PA_OK;
}

extern "C" int pa_batch_fork(pa_allocator* a, const int64_t* parents, const int64_t* children,
                             int32_t n) {
  if (!a || n < 0 || (n > 0 && (!parents || !children))) return PA_ERR_INVALID_ARG;
  try {
    // Check every pair in order (a child forked earlier in the batch may be a
    // later parent) before changing anything: children new and distinct, every
    // parent an existing sequence or an earlier child.
    std::vector<std::pair<int64_t, int32_t>> kids(static_cast<size_t>(n));
    for (int32_t i = 0; i < n; ++i) kids[i] = {children[i], i};
    std::sort(kids.begin(), kids.end());
    for (int32_t i = 1; i < n; ++i)
      if (kids[i].first == kids[i - 1].first) return PA_ERR_SEQ_EXISTS;
    std::vector<const pa_allocator::Seq*> src(static_cast<size_t>(n), nullptr);
    for (int32_t i = 0; i < n; ++i) {
      if (a->seqs.count(children[i])) return PA_ERR_SEQ_EXISTS;
      auto it = a->seqs.find(parents[i]);
      if (it != a->seqs.end()) {
        src[i] = &it->second;  // element references survive rehashing
        continue;
      }
      auto k = std::lower_bound(kids.begin(), kids.end(), std::make_pair(parents[i], int32_t(0)));
      if (k == kids.end() || k->first != parents[i] || k->second >= i) return PA_ERR_NO_SEQ;
    }
    a->seqs.reserve(a->seqs.size() + static_cast<size_t>(n));
    for (int32_t i = 0; i < n; ++i) {
      const pa_allocator::Seq* p = src[i] ? src[i] : &a->seqs.find(parents[i])->second;
      pa_allocator::Seq& c = a->make(children[i]);
      c.blocks = p->blocks;
      c.len = p->len;
      for (int32_t b : c.blocks) ++a->refcount[b];
    }
  } catch (...) {
    return PA_ERR_OOM;
  }
  return PA_OK;
}

extern "C" int pa_batch_free(pa_allocator* a, const int64_t* seqs, int32_t n) {
  if (!a || n < 0 || (n > 0 && !seqs)) return PA_ERR_INVALID_ARG;
  std::vector<pa_allocator::Map::iterator> its;
  try {
    std::vector<int64_t> ids(seqs, seqs + n);
    std::sort(ids.begin(), ids.end());
    for (int32_t i = 1; i < n; ++i)
      if (ids[i] == ids[i - 1]) return PA_ERR_NO_SEQ;  // listed twice
    its.resize(static_cast<size_t>(n));
    for (int32_t i = 0; i < n; ++i) {
      its[i] = a->seqs.find(seqs[i]);
      if (its[i] == a->seqs.end()) return PA_ERR_NO_SEQ;
    }
  } catch (...) {
    return PA_ERR_OOM;
  }
  // Retiring one sequence leaves the others' iterators valid.
  int status = PA_OK;
  for (int32_t i = 0; i < n; ++i) {
    for (int32_t b : its[i]->second.blocks)
      if (!a->release(b)) status = PA_ERR_REFCOUNT;
    a->retire(its[i]);
  }
  return status;
}

extern "C" int pa_batch_block_tables(const pa_allocator* a, const int64_t* seqs, int32_t n,
                                     int32_t max_blocks, int32_t* tables, int32_t* seq_lens) {
  if (!a || n < 0 || max_blocks <= 0 || (n > 0 && (!seqs || !tables || !seq_lens)))
    return PA_ERR_INVALID_ARG;
  for (int32_t i = 0; i < n; ++i) {
    auto it = a->seqs.find(seqs[i]);
    if (it == a->seqs.end()) return PA_ERR_NO_SEQ;
    const auto& s = it->second;
    const int32_t nb = static_cast<int32_t>(s.blocks.size());
    if (nb > max_blocks) return PA_ERR_INVALID_ARG;
    int32_t* row = tables + static_cast<size_t>(i) * max_blocks;
    std::copy(s.blocks.begin(), s.blocks.end(), row);
    std::fill(row + nb, row + max_blocks, -1);
    seq_lens[i] = s.len;
  }
  return PA_OK;
}

extern "C" int pa_alloc_check(const pa_allocator* a) {
  if (!a) return PA_ERR_INVALID_ARG;
  std::vector<int32_t> holders(a->num_blocks, 0);
  for (const auto& kv : a->seqs) {
    const auto& s = kv.second;
    if (static_cast<int32_t>(s.blocks.size()) != a->blocks_for(s.len)) return PA_ERR_REFCOUNT;
    for (int32_t b : s.blocks) {
      if (b < 0 || b >= a->num_blocks) return PA_ERR_REFCOUNT;
      ++holders[b];
    }
  }
  if (holders != a->refcount) return PA_ERR_REFCOUNT;
  std::vector<char> on_free(a->num_blocks, 0);
  for (int32_t b : a->free_stack) {
    if (b < 0 || b >= a->num_blocks || on_free[b] || holders[b] != 0) return PA_ERR_REFCOUNT;
    on_free[b] = 1;
  }
  int32_t used = 0;
  for (int32_t h : holders) used += h > 0;
  if (used + static_cast<int32_t>(a->free_stack.size()) != a->num_blocks) return PA_ERR_REFCOUNT;
  return PA_OK;
}

extern "C" int pa_alloc_stats(const pa_allocator* a, int32_t* blocks_used,
                              int64_t* tokens_logical, int64_t* slots_logical,
                              int64_t* slots_filled) {
  if (!a) return PA_ERR_INVALID_ARG;
  std::vector<int32_t> fill(a->num_blocks, 0);
  int64_t tokens = 0, slots = 0;
  for (const auto& kv : a->seqs) {
    const auto& s = kv.second;
    tokens += s.len;
    slots += static_cast<int64_t>(s.blocks.size()) * a->block_size;
    for (size_t j = 0; j < s.blocks.size(); ++j) {
      const int64_t rows =
          std::min<int64_t>(a->block_size, s.len - static_cast<int64_t>(j) * a->block_size);
      fill[s.blocks[j]] = std::max<int32_t>(fill[s.blocks[j]], static_cast<int32_t>(rows));
    }
  }
  int64_t filled = 0;
  for (int32_t f : fill) filled += f;
  if (blocks_used) *blocks_used = a->num_blocks - static_cast<int32_t>(a->free_stack.size());
  if (tokens_logical) *tokens_logical = tokens;
  if (slots_logical) *slots_logical = slots;
  if (slots_filled) *slots_filled = filled;
  return PA_OK;
}
