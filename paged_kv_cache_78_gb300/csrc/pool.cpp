// Host block pool: block tables, slot mappings and copy-on-write pairs.
//
// The bookkeeping the pages describe for the KV block manager
// (studying-code.tistory.com/16, sections "vLLM의 메모리 관리", "물리적 블록
// 할당", "요청 완료 후 메모리 관리" and "생성 단계에서의 Copy-on-Write";
// tech.blogsailing.com/?p=100, section 3; itan.pw "vLLMにおけるKVCacheマネージャー
// の詳細解説", section "ブロック割当のロジック"):
//   * a prompt of n tokens takes ceil(n / block_size) blocks;
//   * a block is filled left to right and a new one is taken only when the
//     last is full, so a sequence wastes at most one partly filled block;
//   * fork shares blocks by reference count;
//   * a write into a shared block (count > 1) moves the writer to a fresh
//     block and reports (src, dst) for the block copy; the last holder writes
//     in place;
//   * freeing drops counts, last block first, and blocks at 0 join the tail
//     of the FIFO free list.
// Every mutating call either completes or leaves the pool unchanged.
#include <cstdint>
#include <cstring>
#include <deque>
#include <new>
#include <unordered_map>
#include <vector>

#include "pa.h"

namespace {

struct Seq {
  std::vector<int32_t> blocks;  // logical block i -> physical block
  int64_t len = 0;              // tokens written
};

// One reversible step of append_token, kept for rollback.
struct AppendUndo {
  int64_t seq;
  int kind;          // 0: filled an existing private block, 1: new block, 2: copy-on-write
  int32_t old_block; // kind 2: the shared block the sequence left
  int32_t new_block; // kind 1 and 2: the block taken from the free list
};

}  // namespace

struct pa_pool {
  int32_t num_blocks = 0;
  int32_t block_size = 0;
  std::vector<int32_t> ref;
  std::deque<int32_t> free_list;
  std::unordered_map<int64_t, Seq> seqs;
  int64_t next_id = 0;

  Seq* find(int64_t id) {
    auto it = seqs.find(id);
    return it == seqs.end() ? nullptr : &it->second;
  }
  const Seq* find(int64_t id) const {
    auto it = seqs.find(id);
    return it == seqs.end() ? nullptr : &it->second;
  }

  int32_t take_free() {
    int32_t b = free_list.front();
    free_list.pop_front();
    ref[b] = 1;
    return b;
  }

  // Reserve the next token's slot of `s` (id `id`).  Returns PA_OK or
  // PA_ERR_OUT_OF_BLOCKS with nothing changed.
  pa_status append(int64_t id, Seq& s, int64_t* slot, int64_t pair[2], AppendUndo* undo) {
    const int64_t pos = s.len;
    const int64_t logical = pos / block_size;
    const int64_t offset = pos % block_size;
    pair[0] = pair[1] = -1;
    int32_t b;
    if (logical == (int64_t)s.blocks.size()) {
      if (free_list.empty()) return PA_ERR_OUT_OF_BLOCKS;
      b = take_free();
      s.blocks.push_back(b);
      *undo = {id, 1, -1, b};
    } else {
      b = s.blocks[(size_t)logical];
      if (ref[b] > 1) {
        if (free_list.empty()) return PA_ERR_OUT_OF_BLOCKS;
        int32_t nb = take_free();
        ref[b] -= 1;
        s.blocks[(size_t)logical] = nb;
        pair[0] = b;
        pair[1] = nb;
        *undo = {id, 2, b, nb};
        b = nb;
      } else {
        *undo = {id, 0, -1, -1};
      }
    }
    s.len = pos + 1;
    *slot = (int64_t)b * block_size + offset;
    return PA_OK;
  }

  void rollback(const AppendUndo& u) {
    Seq& s = seqs[u.seq];
    s.len -= 1;
    if (u.kind == 1) {
      s.blocks.pop_back();
      ref[u.new_block] = 0;
      free_list.push_front(u.new_block);
    } else if (u.kind == 2) {
      const int64_t logical = s.len / block_size;
      s.blocks[(size_t)logical] = u.old_block;
      ref[u.old_block] += 1;
      ref[u.new_block] = 0;
      free_list.push_front(u.new_block);
    }
  }
};

extern "C" {

pa_status pa_pool_create(int32_t num_blocks, int32_t block_size, const int32_t* free_order,
                         pa_pool** out) {
  if (!out || num_blocks < 0 || block_size <= 0) return PA_ERR_INVALID_ARG;
  *out = nullptr;
  pa_pool* p = new (std::nothrow) pa_pool();
  if (!p) return PA_ERR_INVALID_ARG;
  p->num_blocks = num_blocks;
  p->block_size = block_size;
  p->ref.assign((size_t)num_blocks, 0);
  if (free_order) {
    std::vector<char> seen((size_t)num_blocks, 0);
    for (int32_t i = 0; i < num_blocks; ++i) {
      int32_t b = free_order[i];
      if (b < 0 || b >= num_blocks || seen[(size_t)b]) {
        delete p;
        return PA_ERR_INVALID_ARG;
      }
      seen[(size_t)b] = 1;
      p->free_list.push_back(b);
    }
  } else {
    for (int32_t b = 0; b < num_blocks; ++b) p->free_list.push_back(b);
  }
  *out = p;
  return PA_OK;
}

void pa_pool_destroy(pa_pool* pool) { delete pool; }

pa_status pa_pool_add_seq(pa_pool* pool, int64_t num_tokens, int64_t* seq_id) {
  if (!pool || !seq_id || num_tokens < 0) return PA_ERR_INVALID_ARG;
  const int64_t need = (num_tokens + pool->block_size - 1) / pool->block_size;
  if (need > (int64_t)pool->free_list.size()) return PA_ERR_OUT_OF_BLOCKS;
  Seq s;
  s.blocks.reserve((size_t)need);
  for (int64_t i = 0; i < need; ++i) s.blocks.push_back(pool->take_free());
  s.len = num_tokens;
  const int64_t id = pool->next_id++;
  pool->seqs.emplace(id, std::move(s));
  *seq_id = id;
  return PA_OK;
}

pa_status pa_pool_fork(pa_pool* pool, int64_t parent, int64_t* child) {
  if (!pool || !child) return PA_ERR_INVALID_ARG;
  const Seq* p = pool->find(parent);
  if (!p) return PA_ERR_BAD_STATE;
  Seq c = *p;
  for (int32_t b : c.blocks) pool->ref[b] += 1;
  const int64_t id = pool->next_id++;
  pool->seqs.emplace(id, std::move(c));
  *child = id;
  return PA_OK;
}

pa_status pa_pool_append_token(pa_pool* pool, int64_t seq, int64_t* slot, int64_t cow_pair[2]) {
  if (!pool || !slot || !cow_pair) return PA_ERR_INVALID_ARG;
  Seq* s = pool->find(seq);
  if (!s) return PA_ERR_BAD_STATE;
  AppendUndo undo;
  return pool->append(seq, *s, slot, cow_pair, &undo);
}

pa_status pa_pool_append_tokens(pa_pool* pool, const int64_t* seqs, int32_t n, int64_t* slots,
                                int64_t* cow_pairs, int32_t* num_pairs) {
  if (!pool || n < 0 || (n > 0 && (!seqs || !slots || !cow_pairs)) || !num_pairs)
    return PA_ERR_INVALID_ARG;
  for (int32_t i = 0; i < n; ++i)
    if (!pool->find(seqs[i])) return PA_ERR_BAD_STATE;
  std::vector<AppendUndo> done;
  done.reserve((size_t)n);
  int32_t npairs = 0;
  for (int32_t i = 0; i < n; ++i) {
    int64_t pair[2];
    AppendUndo undo;
    pa_status st = pool->append(seqs[i], *pool->find(seqs[i]), &slots[i], pair, &undo);
    if (st != PA_OK) {
      for (auto it = done.rbegin(); it != done.rend(); ++it) pool->rollback(*it);
      *num_pairs = 0;
      return st;
    }
    done.push_back(undo);
    if (pair[0] >= 0) {
      cow_pairs[2 * npairs] = pair[0];
      cow_pairs[2 * npairs + 1] = pair[1];
      ++npairs;
    }
  }
  *num_pairs = npairs;
  return PA_OK;
}

pa_status pa_pool_free_seq(pa_pool* pool, int64_t seq) {
  if (!pool) return PA_ERR_INVALID_ARG;
  auto it = pool->seqs.find(seq);
  if (it == pool->seqs.end()) return PA_ERR_BAD_STATE;
  const std::vector<int32_t>& blocks = it->second.blocks;
  for (auto b = blocks.rbegin(); b != blocks.rend(); ++b) {
    if (pool->ref[*b] <= 0) return PA_ERR_BAD_STATE;  // cannot happen unless corrupted
  }
  for (auto b = blocks.rbegin(); b != blocks.rend(); ++b) {
    if (--pool->ref[*b] == 0) pool->free_list.push_back(*b);
  }
  pool->seqs.erase(it);
  return PA_OK;
}

pa_status pa_pool_block_table(const pa_pool* pool, int64_t seq, int32_t* out, int32_t cap,
                              int32_t* num_table_blocks, int64_t* seq_len) {
  if (!pool || cap < 0 || (cap > 0 && !out)) return PA_ERR_INVALID_ARG;
  const Seq* s = pool->find(seq);
  if (!s) return PA_ERR_BAD_STATE;
  const int32_t n = (int32_t)s->blocks.size();
  for (int32_t i = 0; i < n && i < cap; ++i) out[i] = s->blocks[(size_t)i];
  if (num_table_blocks) *num_table_blocks = n;
  if (seq_len) *seq_len = s->len;
  return n > cap ? PA_ERR_INVALID_ARG : PA_OK;
}

pa_status pa_pool_fill_tables(const pa_pool* pool, const int64_t* seqs, int32_t n,
                              int32_t* block_tables, int32_t max_blocks_per_seq,
                              int32_t* seq_lens) {
  if (!pool || n < 0 || max_blocks_per_seq <= 0 ||
      (n > 0 && (!seqs || !block_tables || !seq_lens)))
    return PA_ERR_INVALID_ARG;
  for (int32_t i = 0; i < n; ++i) {
    const Seq* s = pool->find(seqs[i]);
    if (!s) return PA_ERR_BAD_STATE;
    if ((int64_t)s->blocks.size() > max_blocks_per_seq || s->len > INT32_MAX)
      return PA_ERR_INVALID_ARG;
  }
  for (int32_t i = 0; i < n; ++i) {
    const Seq* s = pool->find(seqs[i]);
    int32_t* row = block_tables + (size_t)i * (size_t)max_blocks_per_seq;
    const size_t nb = s->blocks.size();
    for (size_t j = 0; j < nb; ++j) row[j] = s->blocks[j];
    for (size_t j = nb; j < (size_t)max_blocks_per_seq; ++j) row[j] = 0;
    seq_lens[i] = (int32_t)s->len;
  }
  return PA_OK;
}

pa_status pa_pool_slot(const pa_pool* pool, int64_t seq, int64_t pos, int64_t* slot) {
  if (!pool || !slot) return PA_ERR_INVALID_ARG;
  const Seq* s = pool->find(seq);
  if (!s) return PA_ERR_BAD_STATE;
  if (pos < 0 || pos >= s->len) return PA_ERR_INVALID_ARG;
  *slot = (int64_t)s->blocks[(size_t)(pos / pool->block_size)] * pool->block_size +
          pos % pool->block_size;
  return PA_OK;
}

pa_status pa_pool_ref_count(const pa_pool* pool, int32_t block, int32_t* ref) {
  if (!pool || !ref || block < 0 || block >= pool->num_blocks) return PA_ERR_INVALID_ARG;
  *ref = pool->ref[(size_t)block];
  return PA_OK;
}

int32_t pa_pool_num_free(const pa_pool* pool) {
  return pool ? (int32_t)pool->free_list.size() : -1;
}

pa_status pa_slot_mapping(const int32_t* block_tables, int32_t num_seqs,
                          int32_t max_blocks_per_seq, int32_t block_size, int32_t num_blocks,
                          const int32_t* seq_idx, const int32_t* positions, int32_t n,
                          int64_t* slots) {
  if (n < 0 || num_seqs < 0 || max_blocks_per_seq <= 0 || block_size <= 0 || num_blocks <= 0)
    return PA_ERR_INVALID_ARG;
  if (n > 0 && (!block_tables || !seq_idx || !positions || !slots)) return PA_ERR_INVALID_ARG;
  for (int32_t i = 0; i < n; ++i) {
    const int32_t s = seq_idx[i], pos = positions[i];
    if (s < 0 || s >= num_seqs || pos < 0) return PA_ERR_INVALID_ARG;
    const int64_t logical = pos / block_size;
    if (logical >= max_blocks_per_seq) return PA_ERR_INVALID_ARG;
    const int32_t b = block_tables[(size_t)s * (size_t)max_blocks_per_seq + (size_t)logical];
    if (b < 0 || b >= num_blocks) return PA_ERR_INVALID_ARG;
    slots[i] = (int64_t)b * block_size + pos % block_size;
  }
  return PA_OK;
}

}  // extern "C"
