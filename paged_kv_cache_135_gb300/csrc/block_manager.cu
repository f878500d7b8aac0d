// Host block manager: the allocator of the paged cache's physical blocks.
//
// What it follows: the hotelren.com notes "Paged KV Cache + Packed Sequence"
// 2.1 (a pool of fixed-size physical blocks taken from a free list, a
// reference count per block, and per sequence the list of its physical
// blocks in logical order), 2.2 (a decode step allocates a block only when
// the token it writes opens a new one; the token's slot is
// block * block_size + position % block_size) and 5.2 (sequences that share
// a prefix share its blocks; releasing a sequence takes one reference from
// each of its blocks, and a block returns to the free list only at zero).
// Where the notes are silent: a sequence that appends into a shared, partly
// filled last block first gets a private copy of it (copy-on-write), so the
// other sequences never see its new token.
//
// Host memory only (no CUDA call).  Blocks are taken from the end of the free
// list and returned to its end.  Every operation either succeeds or changes
// nothing.
#include <stdint.h>

#include <algorithm>
#include <new>
#include <unordered_map>
#include <vector>

#include "../../include/kvc.h"

struct kvc_block_manager {
  struct Seq {
    std::vector<int32_t> blocks;  // physical blocks in logical order
    int len = 0;                  // tokens with a slot
    uint64_t mark = 0;            // the step that last listed it
  };
  int num_blocks = 0, block_size = 0, max_blocks = 0;
  std::vector<int32_t> free_list;
  std::vector<int> ref;
  std::unordered_map<int64_t, Seq> seqs;  // node-based: a Seq never moves
  // Scratch of kvc_bm_step, kept between calls so a step allocates nothing:
  // the step's sequences, and per block the holders not yet moved away.
  uint64_t epoch = 0;
  std::vector<Seq*> step_seqs;
  std::vector<int> left;
  std::vector<uint64_t> left_mark;

  int32_t take() {
    const int32_t b = free_list.back();
    free_list.pop_back();
    ref[b] = 1;
    return b;
  }
  void release(int32_t b) {
    if (--ref[b] == 0) free_list.push_back(b);
  }
  int32_t slot(const Seq& s, int pos) const {
    return s.blocks[pos / block_size] * block_size + pos % block_size;
  }
  void table_row(const Seq& s, int32_t pad, int32_t* row) const {
    const size_t nb = s.blocks.size();
    std::copy(s.blocks.begin(), s.blocks.end(), row);
    std::fill(row + nb, row + max_blocks, pad);
  }
};

namespace {

int blocks_for(int tokens, int block_size) { return (tokens + block_size - 1) / block_size; }

}  // namespace

extern "C" {

kvc_status kvc_bm_create(int num_blocks, int block_size, int max_blocks_per_seq,
                         kvc_block_manager** out) {
  if (out == nullptr) return KVC_ERR_INVALID_ARG;
  *out = nullptr;
  if (num_blocks <= 0 || block_size <= 0 || max_blocks_per_seq <= 0) return KVC_ERR_INVALID_ARG;
  if (static_cast<long long>(num_blocks) * block_size > INT32_MAX) return KVC_ERR_INVALID_ARG;
  kvc_block_manager* bm = new (std::nothrow) kvc_block_manager;
  if (bm == nullptr) return KVC_ERR_INVALID_ARG;
  try {
    bm->num_blocks = num_blocks;
    bm->block_size = block_size;
    bm->max_blocks = max_blocks_per_seq;
    bm->free_list.resize(num_blocks);
    for (int i = 0; i < num_blocks; ++i) bm->free_list[i] = i;  // popped from the end
    bm->ref.assign(num_blocks, 0);
    bm->left.assign(num_blocks, 0);
    bm->left_mark.assign(num_blocks, 0);
  } catch (...) {
    delete bm;
    return KVC_ERR_INVALID_ARG;
  }
  *out = bm;
  return KVC_OK;
}

void kvc_bm_destroy(kvc_block_manager* bm) { delete bm; }

int kvc_bm_num_free(const kvc_block_manager* bm) {
  return bm ? static_cast<int>(bm->free_list.size()) : -1;
}

int kvc_bm_ref_count(const kvc_block_manager* bm, int block) {
  if (bm == nullptr || block < 0 || block >= bm->num_blocks) return -1;
  return bm->ref[block];
}

int kvc_bm_seq_len(const kvc_block_manager* bm, int64_t seq_id) {
  if (bm == nullptr) return -1;
  const auto it = bm->seqs.find(seq_id);
  return it == bm->seqs.end() ? -1 : it->second.len;
}

kvc_status kvc_bm_add(kvc_block_manager* bm, int64_t seq_id, int num_tokens,
                      int32_t* slot_mapping) {
  if (bm == nullptr || num_tokens < 0) return KVC_ERR_INVALID_ARG;
  if (bm->seqs.count(seq_id)) return KVC_ERR_INVALID_ARG;
  const int need = blocks_for(num_tokens, bm->block_size);
  if (need > bm->max_blocks) return KVC_ERR_INVALID_ARG;
  if (need > static_cast<int>(bm->free_list.size())) return KVC_ERR_OUT_OF_BLOCKS;
  try {
    kvc_block_manager::Seq s;
    s.blocks.reserve(bm->max_blocks);
    s.len = num_tokens;
    auto& placed = bm->seqs.emplace(seq_id, std::move(s)).first->second;
    for (int i = 0; i < need; ++i) placed.blocks.push_back(bm->take());
    if (slot_mapping)
      for (int p = 0; p < num_tokens; ++p) slot_mapping[p] = bm->slot(placed, p);
  } catch (...) {
    return KVC_ERR_INVALID_ARG;  // host memory exhausted before anything was taken
  }
  return KVC_OK;
}

kvc_status kvc_bm_fork(kvc_block_manager* bm, int64_t parent, int64_t child) {
  if (bm == nullptr || parent == child) return KVC_ERR_INVALID_ARG;
  const auto it = bm->seqs.find(parent);
  if (it == bm->seqs.end() || bm->seqs.count(child)) return KVC_ERR_INVALID_ARG;
  try {
    kvc_block_manager::Seq s;
    s.blocks.reserve(bm->max_blocks);  // assign() keeps this capacity; operator= need not
    s.blocks.assign(it->second.blocks.begin(), it->second.blocks.end());
    s.len = it->second.len;
    const auto& placed = bm->seqs.emplace(child, std::move(s)).first->second;
    for (const int32_t b : placed.blocks) ++bm->ref[b];  // after the insert, which may throw
  } catch (...) {
    return KVC_ERR_INVALID_ARG;
  }
  return KVC_OK;
}

kvc_status kvc_bm_append(kvc_block_manager* bm, int64_t seq_id, int32_t* slot, int32_t* cow_src,
                         int32_t* cow_dst) {
  if (bm == nullptr || slot == nullptr) return KVC_ERR_INVALID_ARG;
  const auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return KVC_ERR_INVALID_ARG;
  kvc_block_manager::Seq& s = it->second;
  const int p = s.len;
  int32_t src = -1, dst = -1;
  if (p % bm->block_size == 0) {  // the token opens a new block
    if (static_cast<int>(s.blocks.size()) >= bm->max_blocks) return KVC_ERR_INVALID_ARG;
    if (bm->free_list.empty()) return KVC_ERR_OUT_OF_BLOCKS;
    s.blocks.push_back(bm->take());
  } else if (bm->ref[s.blocks.back()] > 1) {  // shared partly filled block: private copy
    if (bm->free_list.empty()) return KVC_ERR_OUT_OF_BLOCKS;
    src = s.blocks.back();
    dst = bm->take();
    bm->release(src);  // still held by the other sequences
    s.blocks.back() = dst;
  }
  s.len = p + 1;
  *slot = bm->slot(s, p);
  if (cow_src) *cow_src = src;
  if (cow_dst) *cow_dst = dst;
  return KVC_OK;
}

kvc_status kvc_bm_free(kvc_block_manager* bm, int64_t seq_id) {
  if (bm == nullptr) return KVC_ERR_INVALID_ARG;
  const auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return KVC_ERR_INVALID_ARG;
  for (const int32_t b : it->second.blocks) bm->release(b);
  bm->seqs.erase(it);
  return KVC_OK;
}

kvc_status kvc_bm_tables(const kvc_block_manager* bm, const int64_t* seq_ids, int n, int32_t pad,
                         int32_t* block_table, int32_t* seq_lens) {
  if (bm == nullptr || n < 0 || (n > 0 && (seq_ids == nullptr || block_table == nullptr)))
    return KVC_ERR_INVALID_ARG;
  for (int i = 0; i < n; ++i)
    if (!bm->seqs.count(seq_ids[i])) return KVC_ERR_INVALID_ARG;
  for (int i = 0; i < n; ++i) {
    const kvc_block_manager::Seq& s = bm->seqs.find(seq_ids[i])->second;
    bm->table_row(s, pad, block_table + static_cast<long long>(i) * bm->max_blocks);
    if (seq_lens) seq_lens[i] = s.len;
  }
  return KVC_OK;
}

kvc_status kvc_bm_step(kvc_block_manager* bm, const int64_t* seq_ids, int n, int32_t pad,
                       int32_t* slots, int32_t* cow_src, int32_t* cow_dst, int32_t* block_table,
                       int32_t* seq_lens) {
  if (bm == nullptr || n < 0) return KVC_ERR_INVALID_ARG;
  if (n == 0) return KVC_OK;
  if (seq_ids == nullptr || slots == nullptr || cow_src == nullptr || cow_dst == nullptr)
    return KVC_ERR_INVALID_ARG;
  // Check first, so that the step either happens for every sequence or for
  // none: ids known and distinct, room in every table, and enough free blocks
  // for the new blocks and the copies.  A shared partly filled block costs a
  // copy for each appending holder while another holder remains, so each such
  // block's remaining holders are counted (scratch stamped with this step).
  try {
    if (static_cast<int>(bm->step_seqs.size()) < n) bm->step_seqs.resize(n);
  } catch (...) {
    return KVC_ERR_INVALID_ARG;  // host memory exhausted; nothing changed
  }
  const uint64_t ep = ++bm->epoch;
  kvc_block_manager::Seq** seq = bm->step_seqs.data();
  int need = 0;
  for (int i = 0; i < n; ++i) {
    const auto it = bm->seqs.find(seq_ids[i]);
    if (it == bm->seqs.end() || it->second.mark == ep) return KVC_ERR_INVALID_ARG;
    it->second.mark = ep;
    seq[i] = &it->second;
    const int p = seq[i]->len;
    if (p % bm->block_size == 0) {
      if (static_cast<int>(seq[i]->blocks.size()) >= bm->max_blocks) return KVC_ERR_INVALID_ARG;
      // The second pass must not reallocate (it could throw half-way): make
      // sure of the capacity now, while nothing has changed yet.
      if (seq[i]->blocks.capacity() < static_cast<size_t>(bm->max_blocks)) {
        try {
          seq[i]->blocks.reserve(bm->max_blocks);
        } catch (...) {
          return KVC_ERR_OUT_OF_BLOCKS;
        }
      }
      ++need;
    } else {
      const int32_t blk = seq[i]->blocks.back();
      if (bm->left_mark[blk] != ep) {
        bm->left_mark[blk] = ep;
        bm->left[blk] = bm->ref[blk];
      }
      if (bm->left[blk] > 1) {
        ++need;
        --bm->left[blk];
      }
    }
  }
  if (need > static_cast<int>(bm->free_list.size())) return KVC_ERR_OUT_OF_BLOCKS;
  for (int i = 0; i < n; ++i) {
    kvc_block_manager::Seq& sq = *seq[i];
    const int p = sq.len;
    int32_t src = -1, dst = -1;
    if (p % bm->block_size == 0) {
      sq.blocks.push_back(bm->take());  // capacity reserved when the sequence was made
    } else if (bm->ref[sq.blocks.back()] > 1) {
      src = sq.blocks.back();
      dst = bm->take();
      bm->release(src);
      sq.blocks.back() = dst;
    }
    sq.len = p + 1;
    slots[i] = bm->slot(sq, p);
    cow_src[i] = src;
    cow_dst[i] = dst;
    if (block_table) bm->table_row(sq, pad, block_table + static_cast<long long>(i) * bm->max_blocks);
    if (seq_lens) seq_lens[i] = sq.len;
  }
  return KVC_OK;
}

}  // extern "C"
