// Host-side block manager of the paged KV pool (the scheduler-owned
// bookkeeping the review describes in §6 "KV Cache Block Tables" and §8/§9):
// fixed-size physical blocks handed out from a free list, per-sequence block
// tables that only grow, reference counts for blocks shared between
// sequences (fork for parallel sampling or a shared prompt prefix), and
// copy-on-write when a sequence appends into a shared, partially filled last
// block.  Invariant (review §8): every physical block is free, owned by
// exactly one logical block, or shared with a positive reference count.
// Waste bound (review §11): a sequence holds at most block_size - 1 unused
// slots.  Not thread-safe: one owner drives it, as the scheduler does.
#include <cstdint>
#include <new>
#include <unordered_map>
#include <unordered_set>
#include <vector>

#include "pagedattn.h"

struct pa_block_manager {
  int64_t num_blocks = 0;
  int32_t block_size = 0;
  std::vector<int32_t> free_list;  // stack of free block ids
  std::vector<int32_t> refcount;   // per physical block
  struct Seq {
    std::vector<int32_t> blocks;
    int64_t tokens = 0;
  };
  std::unordered_map<int64_t, Seq> seqs;

  int32_t take() {
    const int32_t b = free_list.back();
    free_list.pop_back();
    refcount[b] = 1;
    return b;
  }
  void release(int32_t b) {
    if (--refcount[b] == 0) free_list.push_back(b);
  }
};

namespace {
int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
}  // namespace

extern "C" {

PA_API pa_block_manager* pa_bm_create(int64_t num_blocks, int32_t block_size) {
  if (num_blocks <= 0 || num_blocks > INT32_MAX || block_size <= 0) return nullptr;
  pa_block_manager* bm = new (std::nothrow) pa_block_manager();
  if (!bm) return nullptr;
  bm->num_blocks = num_blocks;
  bm->block_size = block_size;
  bm->refcount.assign(static_cast<size_t>(num_blocks), 0);
  bm->free_list.reserve(static_cast<size_t>(num_blocks));
  for (int64_t b = num_blocks - 1; b >= 0; --b) bm->free_list.push_back(static_cast<int32_t>(b));
  return bm;
}

PA_API void pa_bm_destroy(pa_block_manager* bm) { delete bm; }

PA_API int64_t pa_bm_num_free_blocks(const pa_block_manager* bm) {
  return bm ? static_cast<int64_t>(bm->free_list.size()) : -1;
}

PA_API int32_t pa_bm_refcount(const pa_block_manager* bm, int64_t block) {
  if (!bm || block < 0 || block >= bm->num_blocks) return -1;
  return bm->refcount[static_cast<size_t>(block)];
}

PA_API int pa_bm_add_sequence(pa_block_manager* bm, int64_t seq_id, int64_t num_tokens) {
  if (!bm || num_tokens < 0) return PA_ERR_INVALID_ARG;
  if (bm->seqs.count(seq_id)) return PA_ERR_NOT_FOUND;
  const int64_t need = ceil_div(num_tokens, bm->block_size);
  if (need > static_cast<int64_t>(bm->free_list.size())) return PA_ERR_OUT_OF_BLOCKS;
  pa_block_manager::Seq s;
  s.tokens = num_tokens;
  for (int64_t i = 0; i < need; ++i) s.blocks.push_back(bm->take());
  bm->seqs.emplace(seq_id, std::move(s));
  return PA_OK;
}

PA_API int pa_bm_fork(pa_block_manager* bm, int64_t parent_id, int64_t child_id) {
  if (!bm) return PA_ERR_INVALID_ARG;
  auto it = bm->seqs.find(parent_id);
  if (it == bm->seqs.end() || bm->seqs.count(child_id)) return PA_ERR_NOT_FOUND;
  pa_block_manager::Seq child = it->second;  // shares every block: a pointer update, no data copy
  for (int32_t b : child.blocks) ++bm->refcount[b];
  bm->seqs.emplace(child_id, std::move(child));
  return PA_OK;
}

PA_API int pa_bm_append_tokens(pa_block_manager* bm, int64_t seq_id, int32_t num_new, int64_t* slots_out,
                               int64_t* cow_pair_out, int32_t* num_cow_out) {
  if (!bm || num_new < 0 || (num_new > 0 && !slots_out) || !cow_pair_out || !num_cow_out)
    return PA_ERR_INVALID_ARG;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return PA_ERR_NOT_FOUND;
  pa_block_manager::Seq& s = it->second;
  const int64_t bs = bm->block_size;
  // blocks this call needs, checked before anything changes
  const bool partial_last = s.tokens % bs != 0;
  const bool cow = num_new > 0 && partial_last && bm->refcount[s.blocks.back()] > 1;
  const int64_t fresh = ceil_div(s.tokens + num_new, bs) - static_cast<int64_t>(s.blocks.size());
  if (fresh + (cow ? 1 : 0) > static_cast<int64_t>(bm->free_list.size())) return PA_ERR_OUT_OF_BLOCKS;
  *num_cow_out = 0;
  if (cow) {
    // the shared last block keeps its other owners; this sequence continues in
    // a private copy whose rows the caller copies on the GPU (pa_copy_blocks)
    const int32_t src = s.blocks.back();
    const int32_t dst = bm->take();
    bm->release(src);
    s.blocks.back() = dst;
    cow_pair_out[0] = src;
    cow_pair_out[1] = dst;
    *num_cow_out = 1;
  }
  for (int32_t i = 0; i < num_new; ++i) {
    const int64_t pos = s.tokens;
    if (pos % bs == 0) s.blocks.push_back(bm->take());
    slots_out[i] = static_cast<int64_t>(s.blocks[static_cast<size_t>(pos / bs)]) * bs + pos % bs;
    ++s.tokens;
  }
  return PA_OK;
}

PA_API int pa_bm_free_sequence(pa_block_manager* bm, int64_t seq_id) {
  if (!bm) return PA_ERR_INVALID_ARG;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return PA_ERR_NOT_FOUND;
  for (int32_t b : it->second.blocks) bm->release(b);
  bm->seqs.erase(it);
  return PA_OK;
}

PA_API int pa_bm_block_table(const pa_block_manager* bm, int64_t seq_id, int32_t* out, int32_t capacity,
                             int32_t* num_blocks_out, int64_t* num_tokens_out) {
  if (!bm || !num_blocks_out || !num_tokens_out) return PA_ERR_INVALID_ARG;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return PA_ERR_NOT_FOUND;
  const auto& s = it->second;
  *num_blocks_out = static_cast<int32_t>(s.blocks.size());
  *num_tokens_out = s.tokens;
  if (static_cast<int64_t>(s.blocks.size()) > capacity || (!out && !s.blocks.empty())) return PA_ERR_INVALID_ARG;
  for (size_t i = 0; i < s.blocks.size(); ++i) out[i] = s.blocks[i];
  return PA_OK;
}

// Unused slots summed over sequences (each sequence at most block_size - 1).
PA_API int64_t pa_bm_tail_waste(const pa_block_manager* bm) {
  if (!bm) return -1;
  int64_t w = 0;
  for (const auto& kv : bm->seqs)
    w += static_cast<int64_t>(kv.second.blocks.size()) * bm->block_size - kv.second.tokens;
  return w;
}

// Number of violations of the block invariant (0 = consistent).
PA_API int64_t pa_bm_check(const pa_block_manager* bm) {
  if (!bm) return -1;
  int64_t bad = 0;
  std::vector<int32_t> refs(static_cast<size_t>(bm->num_blocks), 0);
  for (const auto& kv : bm->seqs) {
    const auto& s = kv.second;
    if (static_cast<int64_t>(s.blocks.size()) != ceil_div(s.tokens, bm->block_size)) ++bad;
    std::unordered_set<int32_t> seen;
    for (int32_t b : s.blocks) {
      if (b < 0 || b >= bm->num_blocks) {
        ++bad;
        continue;
      }
      if (!seen.insert(b).second) ++bad;  // two logical blocks on one physical block
      ++refs[static_cast<size_t>(b)];
    }
  }
  std::vector<char> is_free(static_cast<size_t>(bm->num_blocks), 0);
  for (int32_t b : bm->free_list) {
    if (b < 0 || b >= bm->num_blocks || is_free[static_cast<size_t>(b)]) {
      ++bad;
      continue;
    }
    is_free[static_cast<size_t>(b)] = 1;
  }
  for (int64_t b = 0; b < bm->num_blocks; ++b) {
    const int32_t rc = bm->refcount[static_cast<size_t>(b)];
    if (rc != refs[static_cast<size_t>(b)]) ++bad;                  // count matches the tables
    if ((rc == 0) != (is_free[static_cast<size_t>(b)] != 0)) ++bad;  // free exactly when unreferenced
  }
  return bad;
}

}  // extern "C"
