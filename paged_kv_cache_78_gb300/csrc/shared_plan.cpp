// Shared-prefix plan: which sequences of a decode batch hold the same
// physical blocks at the start of their block tables, and for how many
// tokens, cut into chunks of query rows for the shared-prefix decode.
//
// Sharing comes from the block pool: a fork shares every block of the parent
// by reference count until a write copies one (studying-code.tistory.com/16,
// section "생성 단계에서의 Copy-on-Write"; tech.blogsailing.com/?p=100,
// section 3), and prefix caching hands a new request the cached blocks of its
// longest known prefix (itan.pw "vLLMにおけるKVCacheマネージャーの詳細解説",
// section "プレイフィックスキャッシュの詳細").  Either way the shared blocks are
// the leading entries of the block tables, with the same ids, so the plan is
// found from the host copy of the tables alone.
//
// Grouping: sequences whose first block ids are equal form a candidate group
// (in increasing sequence order).  Its shared length is the longest run of
// leading block ids every member has in common with the first member, capped
// for every member at floor((L - 1) / block_size) blocks so that each member
// keeps at least its newest token to itself.  Groups of one member, or with
// fewer than min_shared_blocks shared blocks, are dropped.  A group is cut
// into chunks of 4 * floor(32 / G) members (G query heads per KV head): the
// decode tile's 128 rows are four warps of 32, and a member's G rows stay in
// one warp.
#include <algorithm>
#include <cstdint>
#include <unordered_map>
#include <vector>

#include "pa.h"

extern "C" pa_status pa_decode_shared_plan(const int32_t* block_tables, int32_t max_blocks_per_seq,
                                           const int32_t* seq_lens, int32_t num_seqs,
                                           int32_t block_size, int32_t num_heads,
                                           int32_t num_kv_heads, int32_t min_shared_blocks,
                                           int32_t* plan, size_t plan_ints,
                                           pa_shared_plan_info* info) {
  if (!info || num_seqs < 0 || max_blocks_per_seq < 1 || block_size < 1 || block_size > 256 ||
      (block_size & (block_size - 1)) != 0 || num_kv_heads < 1 || num_heads < 1 ||
      num_heads % num_kv_heads != 0 || min_shared_blocks < 1)
    return PA_ERR_INVALID_ARG;
  const int group = num_heads / num_kv_heads;
  if (group > 32) return PA_ERR_INVALID_ARG;
  if (!plan || plan_ints < (size_t)PA_SHARED_PLAN_INTS(num_seqs)) return PA_ERR_INVALID_ARG;
  if (num_seqs > 0 && (!block_tables || !seq_lens)) return PA_ERR_INVALID_ARG;
  for (int s = 0; s < num_seqs; ++s) {
    const int64_t L = seq_lens[s];
    if (L < 0 || (L + block_size - 1) / block_size > max_blocks_per_seq) return PA_ERR_INVALID_ARG;
  }
  // Four softmax warps of 32 rows; a member's G rows stay in one warp.
  const int per_chunk = 4 * (32 / group);

  std::unordered_map<int32_t, int> first_of;  // first block id -> candidate index
  std::vector<std::vector<int>> cand;
  for (int s = 0; s < num_seqs; ++s) {
    if ((seq_lens[s] - 1) / block_size < 1) continue;  // no full block before the newest token
    const int32_t b0 = block_tables[(size_t)s * max_blocks_per_seq];
    auto it = first_of.find(b0);
    if (it == first_of.end()) {
      first_of.emplace(b0, (int)cand.size());
      cand.push_back({s});
    } else {
      cand[it->second].push_back(s);
    }
  }

  struct Group {
    const std::vector<int>* members;
    int32_t shared_tokens;
  };
  std::vector<Group> groups;
  for (const auto& c : cand) {
    if (c.size() < 2) continue;
    const int32_t* t0 = block_tables + (size_t)c[0] * max_blocks_per_seq;
    int64_t shared = max_blocks_per_seq;
    for (int s : c) {
      const int32_t* t = block_tables + (size_t)s * max_blocks_per_seq;
      const int64_t cap = (seq_lens[s] - 1) / block_size;  // blocks before the newest token
      int64_t k = 0;
      while (k < cap && t[k] == t0[k]) ++k;
      shared = std::min(shared, k);
    }
    if (shared < min_shared_blocks) continue;
    groups.push_back({&c, (int32_t)(shared * block_size)});
  }

  // Layout (int32): header {chunks, sequences, members, G}; per chunk
  // {first member index, members, shared tokens, group}; per sequence the
  // first token of its own part (its group's shared tokens, 0 outside a
  // group); the members' sequence ids, chunk after chunk.
  int nc = 0;
  for (const auto& g : groups) nc += (int)((g.members->size() + per_chunk - 1) / per_chunk);
  int32_t* crec = plan + 4;
  int32_t* start = crec + 4 * (size_t)nc;
  int32_t* mem = start + num_seqs;
  for (int s = 0; s < num_seqs; ++s) start[s] = 0;
  // A chunk's stages (the decode's geometry): its shared tokens in 128-token
  // stages, then its members' own tokens in boxes of min(block_size, 128)
  // tokens, queued per softmax warp (ceil(members / 4) members to a warp):
  // boxes of up to 32 tokens fill one 32-column word per warp and stage,
  // wider boxes go 128 / box to a stage round robin over the four queues.
  const int64_t box = std::min<int64_t>(block_size, 128);
  int m = 0, ci = 0;
  int32_t min_tokens = 0, min_stages = 0;
  for (size_t g = 0; g < groups.size(); ++g) {
    const auto& mm = *groups[g].members;
    const int32_t tokens = groups[g].shared_tokens;
    min_tokens = (g == 0) ? tokens : std::min(min_tokens, tokens);
    for (size_t j0 = 0; j0 < mm.size(); j0 += per_chunk) {
      const int cnt = (int)std::min(mm.size() - j0, (size_t)per_chunk);
      crec[4 * ci + 0] = m;
      crec[4 * ci + 1] = cnt;
      crec[4 * ci + 2] = tokens;
      crec[4 * ci + 3] = (int32_t)g;
      const int per_warp = (cnt + 3) / 4;
      int64_t q[4] = {0, 0, 0, 0};
      for (int j = 0; j < cnt; ++j) {
        const int s = mm[j0 + j];
        start[s] = tokens;
        mem[m++] = s;
        q[j / per_warp] += (seq_lens[s] - tokens + box - 1) / box;
      }
      const int64_t qmax = std::max(std::max(q[0], q[1]), std::max(q[2], q[3]));
      const int64_t own = box <= 32 ? (qmax + 32 / box - 1) / (32 / box)
                                    : (4 * qmax + 128 / box - 1) / (128 / box);
      const int64_t stages = (tokens + 127) / 128 + own;
      const int32_t st = (int32_t)std::min<int64_t>(stages, 1 << 30);
      min_stages = (ci == 0) ? st : std::min(min_stages, st);
      ++ci;
    }
  }
  plan[0] = nc;
  plan[1] = num_seqs;
  plan[2] = m;
  plan[3] = group;
  info->num_chunks = nc;
  info->num_members = m;
  info->min_shared_tokens = min_tokens;
  info->min_chunk_stages = min_stages;
  info->group_size = group;
  info->plan_ints = 4 + 4 * nc + num_seqs + m;
  return PA_OK;
}
