// Host-side refcounted block allocator.
//
// Fixed-size blocks, one block table per sequence, a block taken only when
// all earlier blocks of the sequence are full ("Only 20.4% of your KV cache
// held actual tokens", section "The page table, relocated into attention");
// forked samples share blocks by reference count, the first write into a
// shared partially filled block is copy-on-write, and a block whose count
// drops to zero goes back to the pool (same page, section "The part everyone
// forgets: pages enable sharing, not just packing"; "The KV cache is a
// systems problem", section "Shared prefixes need ownership rules").
//
// The allocator only decides ids; the caller turns its answers into device
// work (pkv_block_copy for the pairs, pkv_kv_append for the slots).

#include <stdint.h>

#include <algorithm>
#include <new>
#include <unordered_map>
#include <vector>

#include "pagedkv.h"

struct pkv_allocator {
  int num_blocks = 0;
  int block_size = 0;
  std::vector<int32_t> free_list;  // LIFO: back() is handed out next
  std::vector<int32_t> refcount;
  struct Seq {
    std::vector<int32_t> table;
    int64_t length = 0;
  };
  std::unordered_map<int64_t, Seq> seqs;
  int64_t cow_copies = 0;

  int32_t take() {
    const int32_t b = free_list.back();
    free_list.pop_back();
    refcount[b] = 1;
    return b;
  }

  void release(int32_t b) {
    if (--refcount[b] == 0) free_list.push_back(b);
  }

  static int64_t blocks_for(int64_t tokens, int block_size) {
    return (tokens + block_size - 1) / block_size;
  }

  // Undo record of one append, so that a failed batch can be rolled back.
  struct Undo {
    Seq* seq;
    int32_t taken;    // block taken from the free list (-1: none)
    int32_t cow_src;  // block the sequence held before copy-on-write (-1: none)
  };

  // Reverse one append.  Undoing in reverse order restores the LIFO free
  // list exactly.
  void undo(const Undo& u) {
    u.seq->length -= 1;
    if (u.cow_src >= 0) {
      ++refcount[u.cow_src];
      u.seq->table.back() = u.cow_src;
      --cow_copies;
    } else if (u.taken >= 0) {
      u.seq->table.pop_back();
    }
    if (u.taken >= 0) {
      refcount[u.taken] = 0;
      free_list.push_back(u.taken);
    }
  }

  // One sequence's next slot; fills the copy-on-write pair (or -1, -1).
  // Leaves everything unchanged on failure.
  pkv_status_t append(int64_t seq_id, int64_t* slot, int64_t* cow_src, int64_t* cow_dst,
                      Undo* record = nullptr) {
    auto it = seqs.find(seq_id);
    if (it == seqs.end()) return PKV_ERR_UNKNOWN_SEQ;
    Seq& s = it->second;
    const int64_t pos = s.length;
    const int offset = static_cast<int>(pos % block_size);
    int64_t src = -1, dst = -1;
    int32_t taken = -1;
    if (offset == 0) {
      if (free_list.empty()) return PKV_ERR_OUT_OF_BLOCKS;
      taken = take();
      s.table.push_back(taken);
    } else {
      const int32_t last = s.table.back();
      if (refcount[last] > 1) {
        if (free_list.empty()) return PKV_ERR_OUT_OF_BLOCKS;
        const int32_t fresh = take();
        taken = fresh;
        --refcount[last];  // still > 0: other sequences keep it
        s.table.back() = fresh;
        src = last;
        dst = fresh;
        ++cow_copies;
      }
    }
    s.length = pos + 1;
    *slot = static_cast<int64_t>(s.table.back()) * block_size + offset;
    *cow_src = src;
    *cow_dst = dst;
    if (record) *record = Undo{&s, taken, static_cast<int32_t>(src)};
    return PKV_OK;
  }
};

extern "C" {

pkv_status_t pkv_alloc_create(int num_blocks, int block_size, pkv_allocator** out) {
  if (!out || num_blocks <= 0 || block_size <= 0) return PKV_ERR_INVALID_ARG;
  pkv_allocator* a = new (std::nothrow) pkv_allocator();
  if (!a) return PKV_ERR_OUT_OF_BLOCKS;
  a->num_blocks = num_blocks;
  a->block_size = block_size;
  a->refcount.assign(num_blocks, 0);
  a->free_list.resize(num_blocks);
  for (int i = 0; i < num_blocks; ++i) a->free_list[i] = num_blocks - 1 - i;
  *out = a;
  return PKV_OK;
}

void pkv_alloc_destroy(pkv_allocator* a) { delete a; }

pkv_status_t pkv_alloc_add_seq(pkv_allocator* a, int64_t seq_id, int num_tokens) {
  if (!a || num_tokens < 0) return PKV_ERR_INVALID_ARG;
  if (a->seqs.count(seq_id)) return PKV_ERR_SEQ_EXISTS;
  const int64_t need = pkv_allocator::blocks_for(num_tokens, a->block_size);
  if (need > static_cast<int64_t>(a->free_list.size())) return PKV_ERR_OUT_OF_BLOCKS;
  pkv_allocator::Seq s;
  s.table.reserve(need + 1);
  for (int64_t i = 0; i < need; ++i) s.table.push_back(a->take());
  s.length = num_tokens;
  a->seqs.emplace(seq_id, std::move(s));
  return PKV_OK;
}

pkv_status_t pkv_alloc_fork(pkv_allocator* a, int64_t parent, int64_t child) {
  if (!a) return PKV_ERR_INVALID_ARG;
  auto it = a->seqs.find(parent);
  if (it == a->seqs.end()) return PKV_ERR_UNKNOWN_SEQ;
  if (a->seqs.count(child)) return PKV_ERR_SEQ_EXISTS;
  pkv_allocator::Seq s = it->second;  // copy of the parent's table and length
  for (int32_t b : s.table) ++a->refcount[b];
  a->seqs.emplace(child, std::move(s));
  return PKV_OK;
}

pkv_status_t pkv_alloc_append_slot(pkv_allocator* a, int64_t seq_id, int64_t* slot,
                                   int64_t* cow_src, int64_t* cow_dst) {
  if (!a || !slot || !cow_src || !cow_dst) return PKV_ERR_INVALID_ARG;
  return a->append(seq_id, slot, cow_src, cow_dst);
}

pkv_status_t pkv_alloc_append_slots(pkv_allocator* a, const int64_t* seq_ids, int n,
                                    int64_t* slots, int64_t* cow_pairs, int* num_pairs) {
  if (!a || n < 0 || !num_pairs || (n > 0 && (!seq_ids || !slots || !cow_pairs)))
    return PKV_ERR_INVALID_ARG;
  // All or nothing: on failure every append of the batch is undone.
  std::vector<pkv_allocator::Undo> log(static_cast<size_t>(n));
  int pairs = 0;
  for (int i = 0; i < n; ++i) {
    int64_t src, dst;
    const pkv_status_t st = a->append(seq_ids[i], &slots[i], &src, &dst, &log[i]);
    if (st != PKV_OK) {
      for (int j = i - 1; j >= 0; --j) a->undo(log[j]);
      *num_pairs = 0;
      return st;
    }
    if (src >= 0) {
      cow_pairs[2 * pairs] = src;
      cow_pairs[2 * pairs + 1] = dst;
      ++pairs;
    }
  }
  *num_pairs = pairs;
  return PKV_OK;
}

pkv_status_t pkv_alloc_free_seq(pkv_allocator* a, int64_t seq_id) {
  if (!a) return PKV_ERR_INVALID_ARG;
  auto it = a->seqs.find(seq_id);
  if (it == a->seqs.end()) return PKV_ERR_UNKNOWN_SEQ;
  const std::vector<int32_t>& t = it->second.table;
  for (auto b = t.rbegin(); b != t.rend(); ++b) a->release(*b);
  a->seqs.erase(it);
  return PKV_OK;
}

pkv_status_t pkv_alloc_block_table(pkv_allocator* a, const int64_t* seq_ids, int n, int32_t* out,
                                   int max_blocks) {
  if (!a || n < 0 || max_blocks < 0 || (n > 0 && (!seq_ids || !out))) return PKV_ERR_INVALID_ARG;
  for (int i = 0; i < n; ++i) {  // check everything before writing anything
    auto it = a->seqs.find(seq_ids[i]);
    if (it == a->seqs.end()) return PKV_ERR_UNKNOWN_SEQ;
    if (static_cast<int64_t>(it->second.table.size()) > max_blocks) return PKV_ERR_TABLE_TOO_SMALL;
  }
  for (int i = 0; i < n; ++i) {
    const std::vector<int32_t>& t = a->seqs.find(seq_ids[i])->second.table;
    int32_t* row = out + static_cast<int64_t>(i) * max_blocks;
    std::copy(t.begin(), t.end(), row);
    std::fill(row + t.size(), row + max_blocks, -1);
  }
  return PKV_OK;
}

pkv_status_t pkv_alloc_seq_slots(pkv_allocator* a, int64_t seq_id, int start, int count,
                                 int64_t* out) {
  if (!a || start < 0 || count < 0 || (count > 0 && !out)) return PKV_ERR_INVALID_ARG;
  auto it = a->seqs.find(seq_id);
  if (it == a->seqs.end()) return PKV_ERR_UNKNOWN_SEQ;
  const pkv_allocator::Seq& s = it->second;
  if (static_cast<int64_t>(start) + count > s.length) return PKV_ERR_INVALID_ARG;
  for (int i = 0; i < count; ++i) {
    const int64_t pos = start + i;
    out[i] = static_cast<int64_t>(s.table[pos / a->block_size]) * a->block_size +
             pos % a->block_size;
  }
  return PKV_OK;
}

pkv_status_t pkv_alloc_seq_info(pkv_allocator* a, int64_t seq_id, int* num_tokens,
                                int* num_blocks) {
  if (!a) return PKV_ERR_INVALID_ARG;
  auto it = a->seqs.find(seq_id);
  if (it == a->seqs.end()) return PKV_ERR_UNKNOWN_SEQ;
  if (num_tokens) *num_tokens = static_cast<int>(it->second.length);
  if (num_blocks) *num_blocks = static_cast<int>(it->second.table.size());
  return PKV_OK;
}

pkv_status_t pkv_alloc_refcount(pkv_allocator* a, int block, int* refcount) {
  if (!a || !refcount || block < 0 || block >= a->num_blocks) return PKV_ERR_INVALID_ARG;
  *refcount = a->refcount[block];
  return PKV_OK;
}

pkv_status_t pkv_alloc_stats(pkv_allocator* a, pkv_alloc_stats_t* out) {
  if (!a || !out) return PKV_ERR_INVALID_ARG;
  pkv_alloc_stats_t st{};
  st.num_blocks = a->num_blocks;
  st.free_blocks = static_cast<int64_t>(a->free_list.size());
  for (int b = 0; b < a->num_blocks; ++b) {
    if (a->refcount[b] > 0) ++st.used_blocks;
    if (a->refcount[b] > 1) ++st.shared_blocks;
  }
  st.num_seqs = static_cast<int64_t>(a->seqs.size());
  // Distinct filled slots: a physical block is as full as its fullest owner.
  std::vector<int32_t> fill(a->num_blocks, 0);
  for (const auto& kv : a->seqs) {
    const pkv_allocator::Seq& s = kv.second;
    st.logical_tokens += s.length;
    for (size_t i = 0; i < s.table.size(); ++i) {
      const int64_t held = std::min<int64_t>(a->block_size, s.length - (int64_t)i * a->block_size);
      fill[s.table[i]] = std::max<int32_t>(fill[s.table[i]], static_cast<int32_t>(held));
    }
  }
  for (int32_t f : fill) st.filled_slots += f;
  st.cow_copies = a->cow_copies;
  *out = st;
  return PKV_OK;
}

}  // extern "C"
