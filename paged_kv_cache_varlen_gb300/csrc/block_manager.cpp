// block_manager.cpp -- host-side block manager of the paged KV cache.
//
// Page 2 (su666666.com, "PagedAttention deep-dive") describes the allocator
// the attention kernels rely on: the physical block pool is carved up once at
// start-up; every sequence owns a block table mapping its logical blocks to
// physical blocks; when a sequence needs room for a token and its last block
// is full, the scheduler takes a free block and appends it to the table;
// forking a sequence copies only the table, so parent and child share the
// physical blocks; a shared block gets a private copy only when a sequence
// writes into it. The management happens on the CPU, and each step's tables
// are copied to the GPU before the kernels read them.
//
// Readings where the page is silent: the free pool is first-in first-out
// (initial order given by the caller, ascending by default; released blocks
// join the back); a shared block is copied only when the writer's next token
// falls inside it (it is partially filled) -- a full shared block is never
// written again; the copy covers the whole block (K and V), source to
// destination, and runs on the GPU (pkv_copy_blocks) before the step's KV
// write.
//
// Not thread-safe: one manager is driven by one host thread at a time.
#include <stdint.h>

#include <deque>
#include <new>
#include <unordered_map>
#include <vector>

#include "../../include/pkv.h"

struct pkv_block_manager {
  int32_t num_blocks = 0;
  int32_t block_size = 0;
  std::deque<int32_t> free_pool;
  std::vector<int32_t> refs;
  struct Seq {
    std::vector<int32_t> table;
    int64_t len = 0;
  };
  std::unordered_map<int64_t, Seq> seqs;

  // Free blocks an append of n tokens to s takes: one per new logical block,
  // plus one for copying the last block when it is partially filled and not
  // private to s.
  int64_t blocks_needed(const Seq& s, int64_t n, bool last_private) const {
    if (n <= 0) return 0;
    const int64_t bs = block_size;
    int64_t need = 0;
    if (s.len % bs != 0 && !last_private) need += 1;
    const int64_t present = (s.len + bs - 1) / bs;
    const int64_t last = (s.len + n - 1) / bs;
    need += last + 1 - present;
    return need;
  }

  bool last_is_shared(const Seq& s) const {
    return s.len % block_size != 0 && refs[s.table.back()] > 1;
  }

  // Append n tokens (room known to be available). Writes slots[0..n) and
  // appends copies to src/dst.
  void append(Seq& s, int64_t n, int32_t* slots, std::vector<int32_t>& src,
              std::vector<int32_t>& dst) {
    const int64_t bs = block_size;
    for (int64_t k = 0; k < n; ++k) {
      const int64_t pos = s.len;
      const int64_t logical = pos / bs, offset = pos % bs;
      if (offset == 0) {
        const int32_t blk = free_pool.front();
        free_pool.pop_front();
        refs[blk] = 1;
        s.table.push_back(blk);
      } else if (refs[s.table[logical]] > 1) {
        const int32_t old = s.table[logical];
        const int32_t blk = free_pool.front();
        free_pool.pop_front();
        refs[blk] = 1;
        refs[old] -= 1;
        s.table[logical] = blk;
        src.push_back(old);
        dst.push_back(blk);
      }
      if (slots) slots[k] = (int32_t)(s.table[logical] * bs + offset);
      s.len = pos + 1;
    }
  }
};

namespace {

pkv_block_manager::Seq* find(pkv_block_manager* bm, int64_t id) {
  auto it = bm->seqs.find(id);
  return it == bm->seqs.end() ? nullptr : &it->second;
}

pkv_status emit_copies(const std::vector<int32_t>& src, const std::vector<int32_t>& dst,
                       int32_t* copy_src, int32_t* copy_dst, int32_t max_copies,
                       int32_t* num_copies) {
  if (num_copies) *num_copies = (int32_t)src.size();
  for (size_t i = 0; i < src.size() && (int64_t)i < max_copies; ++i) {
    if (copy_src) copy_src[i] = src[i];
    if (copy_dst) copy_dst[i] = dst[i];
  }
  return PKV_OK;
}

}  // namespace

extern "C" {

pkv_status pkv_bm_create(int32_t num_blocks, int32_t block_size, const int32_t* free_order,
                         pkv_block_manager** out) {
  if (!out || num_blocks <= 0 || block_size <= 0) return PKV_ERR_INVALID_ARG;
  if ((int64_t)num_blocks * block_size > INT32_MAX) return PKV_ERR_UNSUPPORTED;
  pkv_block_manager* bm = new (std::nothrow) pkv_block_manager();
  if (!bm) return PKV_ERR_INVALID_ARG;
  bm->num_blocks = num_blocks;
  bm->block_size = block_size;
  bm->refs.assign(num_blocks, 0);
  if (free_order) {
    std::vector<char> seen(num_blocks, 0);
    for (int32_t i = 0; i < num_blocks; ++i) {
      const int32_t b = free_order[i];
      if (b < 0 || b >= num_blocks || seen[b]) {
        delete bm;
        return PKV_ERR_INVALID_ARG;  // not a permutation of the block ids
      }
      seen[b] = 1;
      bm->free_pool.push_back(b);
    }
  } else {
    for (int32_t b = 0; b < num_blocks; ++b) bm->free_pool.push_back(b);
  }
  *out = bm;
  return PKV_OK;
}

void pkv_bm_destroy(pkv_block_manager* bm) { delete bm; }

pkv_status pkv_bm_add_seq(pkv_block_manager* bm, int64_t seq_id) {
  if (!bm || find(bm, seq_id)) return PKV_ERR_INVALID_ARG;
  bm->seqs.emplace(seq_id, pkv_block_manager::Seq{});
  return PKV_OK;
}

pkv_status pkv_bm_fork(pkv_block_manager* bm, int64_t parent, int64_t child) {
  if (!bm) return PKV_ERR_INVALID_ARG;
  pkv_block_manager::Seq* p = find(bm, parent);
  if (!p || find(bm, child)) return PKV_ERR_INVALID_ARG;
  pkv_block_manager::Seq c = *p;  // the table is copied, the blocks are shared
  for (int32_t b : c.table) bm->refs[b] += 1;
  bm->seqs.emplace(child, std::move(c));
  return PKV_OK;
}

pkv_status pkv_bm_free_seq(pkv_block_manager* bm, int64_t seq_id) {
  if (!bm) return PKV_ERR_INVALID_ARG;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return PKV_ERR_INVALID_ARG;
  for (int32_t b : it->second.table) {
    if (--bm->refs[b] == 0) bm->free_pool.push_back(b);
  }
  bm->seqs.erase(it);
  return PKV_OK;
}

pkv_status pkv_bm_append(pkv_block_manager* bm, int64_t seq_id, int32_t num_tokens,
                         int32_t* slots, int32_t* copy_src, int32_t* copy_dst, int32_t max_copies,
                         int32_t* num_copies) {
  if (!bm || num_tokens < 0 || max_copies < 0) return PKV_ERR_INVALID_ARG;
  pkv_block_manager::Seq* s = find(bm, seq_id);
  if (!s) return PKV_ERR_INVALID_ARG;
  if (s->len + num_tokens > (int64_t)INT32_MAX) return PKV_ERR_UNSUPPORTED;
  const int64_t need = bm->blocks_needed(*s, num_tokens, !bm->last_is_shared(*s));
  if (need > (int64_t)bm->free_pool.size()) return PKV_ERR_NO_BLOCKS;
  if (num_tokens > 0 && bm->last_is_shared(*s) && (!copy_src || !copy_dst || max_copies < 1))
    return PKV_ERR_INVALID_ARG;  // the copy this append makes has nowhere to go
  if (num_tokens > 0 && !slots) return PKV_ERR_INVALID_ARG;
  std::vector<int32_t> src, dst;
  bm->append(*s, num_tokens, slots, src, dst);
  return emit_copies(src, dst, copy_src, copy_dst, max_copies, num_copies);
}

pkv_status pkv_bm_build_step(pkv_block_manager* bm, const int64_t* seq_ids, const int32_t* num_new,
                             int32_t num_seqs, int32_t max_blocks, int32_t* block_table,
                             int32_t* seq_lens, int32_t* cu_seqlens, int32_t* slot_mapping,
                             int32_t* copy_src, int32_t* copy_dst, int32_t max_copies,
                             int32_t* num_copies) {
  if (!bm || num_seqs < 0 || max_blocks <= 0 || max_copies < 0) return PKV_ERR_INVALID_ARG;
  if (num_seqs > 0 && (!seq_ids || !num_new || !block_table || !seq_lens || !cu_seqlens))
    return PKV_ERR_INVALID_ARG;
  // Dry run: the batch's block and copy needs, appends taken in order (a
  // copy made by one sequence can make a later sibling's block private).
  std::vector<pkv_block_manager::Seq*> seqs(num_seqs);
  std::unordered_map<int32_t, int32_t> ref_delta;
  int64_t need = 0, copies = 0, tokens = 0;
  for (int32_t i = 0; i < num_seqs; ++i) {
    seqs[i] = find(bm, seq_ids[i]);
    if (!seqs[i] || num_new[i] < 0) return PKV_ERR_INVALID_ARG;
    for (int32_t j = 0; j < i; ++j)
      if (seq_ids[j] == seq_ids[i]) return PKV_ERR_INVALID_ARG;  // each sequence once
    const pkv_block_manager::Seq& s = *seqs[i];
    const int64_t n = num_new[i];
    tokens += n;
    const int64_t final_len = s.len + n;
    if (final_len > (int64_t)max_blocks * bm->block_size || final_len > INT32_MAX)
      return PKV_ERR_INVALID_ARG;  // the table row cannot hold the sequence
    bool priv = true;
    if (n > 0 && s.len % bm->block_size != 0) {
      const int32_t last = s.table.back();
      const int32_t r = bm->refs[last] + ref_delta[last];
      priv = r <= 1;
      if (!priv) {
        ref_delta[last] -= 1;  // this sequence takes a private copy
        copies += 1;
      }
    }
    need += bm->blocks_needed(s, n, priv);
  }
  if (need > (int64_t)bm->free_pool.size()) return PKV_ERR_NO_BLOCKS;
  if (copies > max_copies || (copies > 0 && (!copy_src || !copy_dst))) return PKV_ERR_INVALID_ARG;
  if (tokens > 0 && !slot_mapping) return PKV_ERR_INVALID_ARG;
  // Commit: append, then describe the step.
  std::vector<int32_t> src, dst;
  int32_t t = 0;
  if (cu_seqlens) cu_seqlens[0] = 0;
  for (int32_t i = 0; i < num_seqs; ++i) {
    pkv_block_manager::Seq& s = *seqs[i];
    bm->append(s, num_new[i], slot_mapping ? slot_mapping + t : nullptr, src, dst);
    t += num_new[i];
    cu_seqlens[i + 1] = t;
    seq_lens[i] = (int32_t)s.len;
    int32_t* row = block_table + (int64_t)i * max_blocks;
    for (int32_t b = 0; b < max_blocks; ++b)
      row[b] = b < (int32_t)s.table.size() ? s.table[b] : -1;
  }
  return emit_copies(src, dst, copy_src, copy_dst, max_copies, num_copies);
}

int32_t pkv_bm_num_free(const pkv_block_manager* bm) {
  return bm ? (int32_t)bm->free_pool.size() : -1;
}

int64_t pkv_bm_seq_len(const pkv_block_manager* bm, int64_t seq_id) {
  if (!bm) return -1;
  auto it = bm->seqs.find(seq_id);
  return it == bm->seqs.end() ? -1 : it->second.len;
}

int32_t pkv_bm_refcount(const pkv_block_manager* bm, int32_t block) {
  if (!bm || block < 0 || block >= bm->num_blocks) return -1;
  return bm->refs[block];
}

pkv_status pkv_bm_block_table(const pkv_block_manager* bm, int64_t seq_id, int32_t* table,
                              int32_t capacity, int32_t* num_blocks) {
  if (!bm || capacity < 0) return PKV_ERR_INVALID_ARG;
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return PKV_ERR_INVALID_ARG;
  const std::vector<int32_t>& t = it->second.table;
  if (num_blocks) *num_blocks = (int32_t)t.size();
  if ((int64_t)t.size() > capacity) return PKV_ERR_WORKSPACE;
  for (size_t i = 0; i < t.size(); ++i) table[i] = t[i];
  return PKV_OK;
}

}  // extern "C"
