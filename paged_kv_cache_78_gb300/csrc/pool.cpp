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
// Prefix caching (itan.pw page, section "プレイフィックスキャッシュの詳細"):
//   * a full block of a sequence created with its token ids carries a chained
//     hash (the previous block's hash and the block's tokens) and is
//     registered under it; a partly filled block has none;
//   * a new request shares the longest run of leading blocks whose hashes are
//     registered, at most (tokens - 1) / block_size of them; shared blocks
//     leave the free queue before the request's other blocks are taken;
//   * freed blocks keep their hash until the free queue hands them out again.
// Every mutating call either completes or leaves the pool unchanged.
#include <cstdint>
#include <cstring>
#include <deque>
#include <new>
#include <unordered_map>
#include <vector>

#include "pa.h"

namespace {


// 128-bit chained block hash: two independent 64-bit mixes.
struct BlockHash {
  uint64_t a = 0, b = 0;
  bool operator==(const BlockHash& o) const { return a == o.a && b == o.b; }
};

struct BlockHashKey {
  size_t operator()(const BlockHash& h) const { return (size_t)(h.a ^ (h.b * 0x9e3779b97f4a7c15ull)); }
};

// splitmix64 finaliser (Steele, Lea and Flood, "Fast splittable pseudorandom
// number generators", 2014).
inline uint64_t mix64(uint64_t x) {
  x += 0x9e3779b97f4a7c15ull;
  x = (x ^ (x >> 30)) * 0xbf58476d1ce4e5b9ull;
  x = (x ^ (x >> 27)) * 0x94d049bb133111ebull;
  return x ^ (x >> 31);
}

// Hash of a block's tokens chained to the previous block's hash.
BlockHash chain_hash(const BlockHash& prev, const int32_t* tokens, int n) {
  BlockHash h{prev.a ^ 0x6a09e667f3bcc908ull, prev.b ^ 0xbb67ae8584caa73bull};
  for (int i = 0; i < n; ++i) {
    const uint64_t t = (uint64_t)(uint32_t)tokens[i];
    h.a = mix64(h.a ^ t);
    h.b = mix64(h.b + (t << 1 | 1) * 0xd6e8feb86659fd93ull);
  }
  h.a = mix64(h.a ^ (uint64_t)n);
  h.b = mix64(h.b ^ ((uint64_t)n << 32));
  return h;
}

// Free blocks as a doubly linked queue over the block ids: taken from the
// front, returned to the back, and a cached block that a new request shares
// leaves it from wherever it is.
struct FreeQueue {
  std::vector<int32_t> prev, next;
  std::vector<char> in;
  int32_t head = -1, tail = -1;
  int32_t count = 0;

  void init(int32_t n) {
    prev.assign((size_t)n, -1);
    next.assign((size_t)n, -1);
    in.assign((size_t)n, 0);
  }
  bool empty() const { return count == 0; }
  size_t size() const { return (size_t)count; }
  int32_t front() const { return head; }
  void push_back(int32_t b) {
    prev[b] = tail;
    next[b] = -1;
    if (tail >= 0) next[tail] = b; else head = b;
    tail = b;
    in[b] = 1;
    ++count;
  }
  void push_front(int32_t b) {
    next[b] = head;
    prev[b] = -1;
    if (head >= 0) prev[head] = b; else tail = b;
    head = b;
    in[b] = 1;
    ++count;
  }
  void remove(int32_t b) {
    if (prev[b] >= 0) next[prev[b]] = next[b]; else head = next[b];
    if (next[b] >= 0) prev[next[b]] = prev[b]; else tail = prev[b];
    prev[b] = next[b] = -1;
    in[b] = 0;
    --count;
  }
  void pop_front() { remove(head); }
};

struct Seq {
  std::vector<int32_t> blocks;  // logical block i -> physical block
  int64_t len = 0;              // tokens written
  bool tracked = false;         // created with token ids (takes part in prefix caching)
  std::vector<int32_t> tokens;  // tracked: every token id so far
  BlockHash chain;              // tracked: chained hash of the full blocks so far
  int64_t chained = 0;          // tracked: how many full blocks `chain` covers
  bool swapped = false;         // blocks are CPU block ids (swapped out)
};

// One reversible step of append_token, kept for rollback.
struct AppendUndo {
  int64_t seq;
  int kind;          // 0: filled an existing private block, 1: new block, 2: copy-on-write
  int32_t old_block; // kind 2: the shared block the sequence left
  int32_t new_block; // kind 1 and 2: the block taken from the free list
  bool had_hash;     // kind 1 and 2: new_block was registered before it was taken
  BlockHash hash;    //   ... under this hash
};

}  // namespace

struct pa_pool {
  int32_t num_blocks = 0;
  int32_t block_size = 0;
  std::vector<int32_t> ref;
  FreeQueue free_list;
  std::unordered_map<int64_t, Seq> seqs;
  int64_t next_id = 0;
  // CPU swap region: blocks 0..num_cpu_blocks-1, a FIFO free list and counts.
  int32_t num_cpu_blocks = 0;
  std::vector<int32_t> cpu_ref;
  std::deque<int32_t> cpu_free;
  // Prefix cache: registered full blocks by chained hash, and each block's hash.
  std::unordered_map<BlockHash, int32_t, BlockHashKey> cached;
  std::vector<BlockHash> block_hash;
  std::vector<char> hashed;

  void uncache(int32_t b) {
    if (!hashed[b]) return;
    auto it = cached.find(block_hash[b]);
    if (it != cached.end() && it->second == b) cached.erase(it);
    hashed[b] = 0;
  }

  // Register block b (full, of a tracked sequence) under h unless another
  // block already holds that hash.
  void register_block(int32_t b, const BlockHash& h) {
    if (hashed[b] || cached.count(h)) return;
    cached.emplace(h, b);
    block_hash[b] = h;
    hashed[b] = 1;
  }

  // Chained hash of logical block i of a tracked sequence (its tokens known).
  BlockHash hash_of(const Seq& s, int64_t i) const {
    BlockHash h;
    for (int64_t j = 0; j <= i; ++j)
      h = chain_hash(h, s.tokens.data() + j * block_size, block_size);
    return h;
  }

  Seq* find(int64_t id) {
    auto it = seqs.find(id);
    return it == seqs.end() ? nullptr : &it->second;
  }
  const Seq* find(int64_t id) const {
    auto it = seqs.find(id);
    return it == seqs.end() ? nullptr : &it->second;
  }

  // A block handed out for new content loses its cached hash (reported in
  // *had / *h so that a rollback can restore it).
  int32_t take_free(bool* had = nullptr, BlockHash* h = nullptr) {
    int32_t b = free_list.front();
    free_list.pop_front();
    if (had) *had = hashed[b] != 0;
    if (h) *h = block_hash[b];
    uncache(b);
    ref[b] = 1;
    return b;
  }

  // A tracked sequence whose block `logical` just became full: chain its hash
  // and register the block.
  void seal(Seq& s, int64_t logical) {
    if (!s.tracked || logical != s.chained) return;
    s.chain = chain_hash(s.chain, s.tokens.data() + logical * block_size, block_size);
    s.chained = logical + 1;
    register_block(s.blocks[(size_t)logical], s.chain);
  }

  // Reserve the next token's slot of `s` (id `id`); `token` is its id, or
  // null (a tracked sequence then stops taking part in prefix caching).
  // Returns PA_OK or PA_ERR_OUT_OF_BLOCKS with nothing changed.
  pa_status append(int64_t id, Seq& s, const int32_t* token, int64_t* slot, int64_t pair[2],
                   AppendUndo* undo) {
    const int64_t pos = s.len;
    const int64_t logical = pos / block_size;
    const int64_t offset = pos % block_size;
    pair[0] = pair[1] = -1;
    int32_t b;
    if (logical == (int64_t)s.blocks.size()) {
      if (free_list.empty()) return PA_ERR_OUT_OF_BLOCKS;
      *undo = {id, 1, -1, -1, false, BlockHash{}};
      b = take_free(&undo->had_hash, &undo->hash);
      undo->new_block = b;
      s.blocks.push_back(b);
    } else {
      b = s.blocks[(size_t)logical];
      if (ref[b] > 1) {
        if (free_list.empty()) return PA_ERR_OUT_OF_BLOCKS;
        *undo = {id, 2, b, -1, false, BlockHash{}};
        int32_t nb = take_free(&undo->had_hash, &undo->hash);
        undo->new_block = nb;
        ref[b] -= 1;
        s.blocks[(size_t)logical] = nb;
        pair[0] = b;
        pair[1] = nb;
        b = nb;
      } else {
        *undo = {id, 0, -1, -1, false, BlockHash{}};
      }
    }
    s.len = pos + 1;
    *slot = (int64_t)b * block_size + offset;
    if (s.tracked && token) {
      s.tokens.push_back(*token);
      if (offset == block_size - 1) seal(s, logical);
    }
    return PA_OK;
  }

  // A tracked sequence appended to without a token id (after the append
  // succeeded): it stops taking part in prefix caching.
  static void untrack(Seq& s) {
    if (!s.tracked) return;
    s.tracked = false;
    s.tokens.clear();
    s.tokens.shrink_to_fit();
  }

  // Undo an untracked append (the batch call appends without token ids).
  void rollback(const AppendUndo& u) {
    Seq& s = seqs[u.seq];
    s.len -= 1;
    if (u.kind == 1) {
      s.blocks.pop_back();
    } else if (u.kind == 2) {
      const int64_t logical = s.len / block_size;
      s.blocks[(size_t)logical] = u.old_block;
      ref[u.old_block] += 1;
    }
    if (u.kind != 0) {
      ref[u.new_block] = 0;
      free_list.push_front(u.new_block);
      if (u.had_hash) register_block(u.new_block, u.hash);
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
  p->free_list.init(num_blocks);
  p->block_hash.assign((size_t)num_blocks, BlockHash{});
  p->hashed.assign((size_t)num_blocks, 0);
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
  if (!p || p->swapped) return PA_ERR_BAD_STATE;
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
  if (!s || s->swapped) return PA_ERR_BAD_STATE;
  AppendUndo undo;
  const pa_status st = pool->append(seq, *s, nullptr, slot, cow_pair, &undo);
  if (st == PA_OK) pa_pool::untrack(*s);
  return st;
}

pa_status pa_pool_append_token_id(pa_pool* pool, int64_t seq, int32_t token, int64_t* slot,
                                  int64_t cow_pair[2]) {
  if (!pool || !slot || !cow_pair) return PA_ERR_INVALID_ARG;
  Seq* s = pool->find(seq);
  if (!s || s->swapped) return PA_ERR_BAD_STATE;
  AppendUndo undo;
  return pool->append(seq, *s, &token, slot, cow_pair, &undo);
}

pa_status pa_pool_add_seq_tokens(pa_pool* pool, const int32_t* tokens, int64_t num_tokens,
                                 int64_t* seq_id, int64_t* num_cached_tokens) {
  if (!pool || !seq_id || !num_cached_tokens || num_tokens < 0 || (num_tokens > 0 && !tokens))
    return PA_ERR_INVALID_ARG;
  const int32_t bs = pool->block_size;
  const int64_t need = (num_tokens + bs - 1) / bs;
  const int64_t full = num_tokens / bs;
  // The longest run of leading full blocks already registered, at most
  // (num_tokens - 1) / block_size: the last token is always computed.
  const int64_t max_hit = num_tokens > 0 ? (num_tokens - 1) / bs : 0;
  std::vector<int32_t> hit;
  std::vector<BlockHash> chain;
  chain.reserve((size_t)full);
  BlockHash h;
  for (int64_t i = 0; i < full; ++i) {
    h = chain_hash(h, tokens + i * bs, bs);
    chain.push_back(h);
  }
  for (int64_t i = 0; i < max_hit; ++i) {
    auto it = pool->cached.find(chain[(size_t)i]);
    if (it == pool->cached.end()) break;
    hit.push_back(it->second);
  }
  int64_t hits_in_queue = 0;
  for (int32_t b : hit) hits_in_queue += pool->free_list.in[b] ? 1 : 0;
  if (need - (int64_t)hit.size() > (int64_t)pool->free_list.size() - hits_in_queue)
    return PA_ERR_OUT_OF_BLOCKS;
  Seq s;
  s.blocks.reserve((size_t)need);
  // Shared blocks first leave the free queue, then the rest are taken.
  for (int32_t b : hit) {
    if (pool->free_list.in[b]) pool->free_list.remove(b);
    pool->ref[b] += 1;
    s.blocks.push_back(b);
  }
  for (int64_t i = (int64_t)hit.size(); i < need; ++i) s.blocks.push_back(pool->take_free());
  s.len = num_tokens;
  s.tracked = true;
  s.tokens.assign(tokens, tokens + num_tokens);
  // Register the new full blocks (their KV is the caller's to write).
  for (int64_t i = (int64_t)hit.size(); i < full; ++i)
    pool->register_block(s.blocks[(size_t)i], chain[(size_t)i]);
  s.chain = full > 0 ? chain[(size_t)full - 1] : BlockHash{};
  s.chained = full;
  const int64_t id = pool->next_id++;
  pool->seqs.emplace(id, std::move(s));
  *seq_id = id;
  *num_cached_tokens = (int64_t)hit.size() * bs;
  return PA_OK;
}

pa_status pa_pool_is_cached(const pa_pool* pool, int32_t block, int32_t* cached) {
  if (!pool || !cached || block < 0 || block >= pool->num_blocks) return PA_ERR_INVALID_ARG;
  *cached = pool->hashed[(size_t)block] ? 1 : 0;
  return PA_OK;
}

pa_status pa_pool_free_queue(const pa_pool* pool, int32_t* out, int32_t cap, int32_t* n) {
  if (!pool || !n || cap < 0 || (cap > 0 && !out)) return PA_ERR_INVALID_ARG;
  int32_t i = 0;
  for (int32_t b = pool->free_list.head; b >= 0; b = pool->free_list.next[(size_t)b], ++i)
    if (i < cap) out[i] = b;
  *n = i;
  return i > cap ? PA_ERR_INVALID_ARG : PA_OK;
}

pa_status pa_pool_reset_prefix_cache(pa_pool* pool) {
  if (!pool) return PA_ERR_INVALID_ARG;
  for (int32_t b = 0; b < pool->num_blocks; ++b) pool->hashed[(size_t)b] = 0;
  pool->cached.clear();
  return PA_OK;
}

pa_status pa_pool_append_tokens(pa_pool* pool, const int64_t* seqs, int32_t n, int64_t* slots,
                                int64_t* cow_pairs, int32_t* num_pairs) {
  if (!pool || n < 0 || (n > 0 && (!seqs || !slots || !cow_pairs)) || !num_pairs)
    return PA_ERR_INVALID_ARG;
  for (int32_t i = 0; i < n; ++i)
    if (!pool->find(seqs[i]) || pool->find(seqs[i])->swapped) return PA_ERR_BAD_STATE;
  std::vector<AppendUndo> done;
  done.reserve((size_t)n);
  int32_t npairs = 0;
  for (int32_t i = 0; i < n; ++i) {
    int64_t pair[2];
    AppendUndo undo;
    pa_status st = pool->append(seqs[i], *pool->find(seqs[i]), nullptr, &slots[i], pair, &undo);
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
  for (int32_t i = 0; i < n; ++i) pa_pool::untrack(*pool->find(seqs[i]));
  *num_pairs = npairs;
  return PA_OK;
}

pa_status pa_pool_free_seq(pa_pool* pool, int64_t seq) {
  if (!pool) return PA_ERR_INVALID_ARG;
  auto it = pool->seqs.find(seq);
  if (it == pool->seqs.end()) return PA_ERR_BAD_STATE;
  const std::vector<int32_t>& blocks = it->second.blocks;
  std::vector<int32_t>& ref = it->second.swapped ? pool->cpu_ref : pool->ref;
  for (auto b = blocks.rbegin(); b != blocks.rend(); ++b) {
    if (ref[*b] <= 0) return PA_ERR_BAD_STATE;  // cannot happen unless corrupted
  }
  for (auto b = blocks.rbegin(); b != blocks.rend(); ++b) {
    if (--ref[*b] == 0) {
      if (it->second.swapped) pool->cpu_free.push_back(*b); else pool->free_list.push_back(*b);
    }
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
    if (!s || s->swapped) return PA_ERR_BAD_STATE;
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
  if (!s || s->swapped) return PA_ERR_BAD_STATE;
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

pa_status pa_pool_set_cpu_blocks(pa_pool* pool, int32_t num_cpu_blocks) {
  if (!pool || num_cpu_blocks < 0 || num_cpu_blocks > pool->num_blocks) return PA_ERR_INVALID_ARG;
  for (const auto& kv : pool->seqs)
    if (kv.second.swapped) return PA_ERR_BAD_STATE;
  pool->num_cpu_blocks = num_cpu_blocks;
  pool->cpu_ref.assign((size_t)num_cpu_blocks, 0);
  pool->cpu_free.clear();
  for (int32_t b = 0; b < num_cpu_blocks; ++b) pool->cpu_free.push_back(b);
  return PA_OK;
}

// Swap a sequence group between GPU and CPU blocks (all or nothing).  `out`
// selects the direction; pairs receive (src, dst) block ids in first-use
// order, one per distinct block.
static pa_status swap_group(pa_pool* pool, const int64_t* seqs, int32_t n, int64_t* pairs,
                            int32_t* num_pairs, bool out) {
  if (!pool || n < 0 || (n > 0 && (!seqs || !pairs)) || !num_pairs) return PA_ERR_INVALID_ARG;
  *num_pairs = 0;
  std::vector<Seq*> group;
  for (int32_t i = 0; i < n; ++i) {
    Seq* s = pool->find(seqs[i]);
    if (!s || s->swapped == out) return PA_ERR_BAD_STATE;
    for (Seq* g : group)
      if (g == s) return PA_ERR_INVALID_ARG;  // listed twice
    group.push_back(s);
  }
  std::vector<int32_t>& from_ref = out ? pool->ref : pool->cpu_ref;
  // Distinct source blocks in first-use order, and the group's references.
  std::unordered_map<int32_t, int32_t> uses;
  std::vector<int32_t> order;
  for (Seq* s : group)
    for (int32_t b : s->blocks)
      if (uses[b]++ == 0) order.push_back(b);
  // A block also held outside the group would be split: refuse.
  for (int32_t b : order)
    if (uses[b] != from_ref[(size_t)b]) return PA_ERR_BAD_STATE;
  const size_t avail = out ? pool->cpu_free.size() : pool->free_list.size();
  if (order.size() > avail) return PA_ERR_OUT_OF_BLOCKS;
  std::unordered_map<int32_t, int32_t> to;
  for (size_t i = 0; i < order.size(); ++i) {
    const int32_t b = order[i];
    int32_t d;
    if (out) {
      d = pool->cpu_free.front();
      pool->cpu_free.pop_front();
      pool->cpu_ref[(size_t)d] = pool->ref[(size_t)b];
    } else {
      const int32_t r = pool->cpu_ref[(size_t)b];
      d = pool->take_free();
      pool->ref[(size_t)d] = r;
    }
    to[b] = d;
    pairs[2 * i] = b;
    pairs[2 * i + 1] = d;
  }
  // Release the source blocks, each sequence's last block first, and move
  // the tables to the destination blocks.
  for (Seq* s : group) {
    for (auto it = s->blocks.rbegin(); it != s->blocks.rend(); ++it) {
      if (--from_ref[(size_t)*it] == 0) {
        if (out) pool->free_list.push_back(*it); else pool->cpu_free.push_back(*it);
      }
    }
    for (int32_t& b : s->blocks) b = to[b];
    s->swapped = out;
  }
  *num_pairs = (int32_t)order.size();
  return PA_OK;
}

pa_status pa_pool_swap_out(pa_pool* pool, const int64_t* seqs, int32_t n, int64_t* pairs,
                           int32_t* num_pairs) {
  return swap_group(pool, seqs, n, pairs, num_pairs, true);
}

pa_status pa_pool_swap_in(pa_pool* pool, const int64_t* seqs, int32_t n, int64_t* pairs,
                          int32_t* num_pairs) {
  return swap_group(pool, seqs, n, pairs, num_pairs, false);
}

pa_status pa_pool_is_swapped(const pa_pool* pool, int64_t seq, int32_t* swapped) {
  if (!pool || !swapped) return PA_ERR_INVALID_ARG;
  const Seq* s = pool->find(seq);
  if (!s) return PA_ERR_BAD_STATE;
  *swapped = s->swapped ? 1 : 0;
  return PA_OK;
}

int32_t pa_pool_num_free_cpu(const pa_pool* pool) {
  return pool ? (int32_t)pool->cpu_free.size() : -1;
}

pa_status pa_pool_usage(const pa_pool* pool, int64_t* tokens, int64_t* blocks_in_use) {
  if (!pool || !tokens || !blocks_in_use) return PA_ERR_INVALID_ARG;
  int64_t t = 0, b = 0;
  for (const auto& kv : pool->seqs)
    if (!kv.second.swapped) t += kv.second.len;
  for (int32_t i = 0; i < pool->num_blocks; ++i) b += pool->ref[(size_t)i] > 0 ? 1 : 0;
  *tokens = t;
  *blocks_in_use = b;
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
