// Shared-prefix decode on the tensor cores: the attention of a group of
// sequences that share leading K/V blocks, with every block read once.
//
// Sharing is what the block pool produces: parallel samples forked from one
// prompt hold the prompt's blocks by reference count until a write copies
// one (studying-code.tistory.com/16, section "생성 단계에서의 Copy-on-Write";
// tech.blogsailing.com/?p=100, section 3), and prefix caching gives a new
// request the cached blocks of its longest known prefix (itan.pw
// "vLLMにおけるKVCacheマネージャーの詳細解説", section "プレイフィックスキャッシュの詳細").
// Either way the shared blocks lead the members' block tables with the same
// ids.
//
// A CTA takes one (stage range, KV head, chunk); a chunk is up to 128 query
// rows (members x query heads of the KV head), the M dimension of both MMAs:
//   S [128 rows x 128 tokens] = Q [128 x D] . K_stage^T        (QK, N = 128)
//   O [128 rows x D]         += P [128 x 128 tokens] . V_stage  (PV, N = D)
// A chunk's stages are first its shared tokens [0, T), which every row
// attends, then its members' own tokens [T, L_j) in boxes (a box is
// min(block_size, 128) tokens of one block), where a row attends only the
// boxes of its own member (the other columns are masked).  Members are
// spread over the four softmax warps, ceil(members / 4) to a warp with each
// member's G rows in consecutive lanes, and every warp has a queue of its
// members' own boxes: in a packed stage, 32-column word w holds boxes from
// warp w's queue (boxes of up to 32 tokens), so each warp computes the
// softmax of one word of the stage and skips the others.  The stages are cut
// into `ranges` equal ranges, one per CTA: with one range the CTA writes the
// rows' final output, otherwise each range is a split-KV partial (O / l and
// the log2-domain log-sum-exp; zero weight for a row with no token in the
// range) that the log-sum-exp reduce combines.
//
// S and P (double-buffered) and O (accumulated over the range) live in
// tensor memory; PV reads P from there, which leaves shared memory to the
// query tile and three K/V stages (five at head size 64).  Each softmax
// thread owns one query row, so the online softmax needs no exchange between
// threads; when a stage's maximum exceeds the running one by more than
// kShLazyMax (log2 units) the thread rescales its row of O in tensor memory
// before the stage's PV.  Warps:
//   warp 0      producer: per stage, each lane resolves one box (member,
//               block id, tokens held), records it for the softmax and
//               issues its TMA load (the tensor-core decode's 5-D map and
//               stage layout); the next stage's boxes are prefetched into L2
//               as soon as they are resolved; a member's newest token (the
//               fused cache write) is written just before its last box loads;
//   warp 1      tensor-memory allocator and MMA issuer (an event loop);
//   warps 2..5  query tile (each thread gathers its row), softmax, output.
// Every wait is bounded (the decode's wait limit); a timeout records
// PA_DEVERR_TIMEOUT, drains the CTA's own TMA loads and MMAs, frees tensor
// memory and returns.
#pragma once

#include "decode_tc_kernel.cuh"

namespace pa {

constexpr int kShThreads = 192;
constexpr int kShRows = 128;        // query rows of a tile: M of both MMAs
constexpr int kShTokens = 128;      // tokens per stage: N of QK, K of PV
constexpr int kShTmemCols = 512;    // S x2 (128 columns each), P x2 (64 each), O (D)
constexpr float kShLazyMax = 8.f;

constexpr int kShMaxBoxes = 16;     // boxes per stage (boxes of 8 tokens or more)

struct SharedParams {
  const void* query;             // [S][Hq][D] bf16
  const int32_t* block_tables;   // [S][max_blocks_per_seq]
  const int32_t* seq_lens;       // [S]
  const int32_t* chunks;         // [num_chunks][4]: first member, members, shared tokens, group
  const int32_t* members;        // member sequence ids, chunk after chunk
  void* out;                     // [S][Hq][D] bf16: final rows (one range)
  float* part_o;                 // [S][Hq][max_parts][D] (several ranges)
  float* part_lse;               // [S][Hq][max_parts]
  int32_t* part_counts;          // [S][Hkv]: partials of each member pair for the reduce
  uint8_t* cache_w;              // the pool, for the fused cache write
  const void* new_k;             // [S][Hkv][D] newest tokens, or null
  const void* new_v;
  unsigned int* err;
  int num_chunks;
  int num_members;
  int num_seqs;
  int num_heads;
  int num_kv_heads;
  int group;
  int num_blocks;
  int block_size;
  int log2_block_size;
  int max_blocks_per_seq;
  int max_parts;
  int ranges;                    // stage ranges per (chunk, KV head) = gridDim.x
  int box_rows;                  // min(block_size, 128)
  int log2_box_rows;
  int num_stages;                // ring slots
  float scale_log2;
  long long wait_limit;
  unsigned long long* trace;     // timeline (pa_set_decode_trace), or null
  int trace_per_role;
  size_t trace_bytes;
  int trace_cta_base;            // record index of this grid's first CTA
};

// Shared-memory layout (byte offsets from a 1024-aligned base).
struct ShSmem {
  int stage, q_off, bar_off, misc_off, mem_off, len_off, pre_off, meta_off, total;
};

__host__ __device__ inline ShSmem sh_smem_layout(int head_size, int num_stages) {
  ShSmem l;
  const int groups = head_size / 64;
  l.stage = 2 * groups * kShTokens * 128;            // K and V of 128 tokens
  l.q_off = num_stages * l.stage;
  l.bar_off = l.q_off + groups * kShRows * 128;      // Q: [column group][128 rows][128 B]
  // full[NS], empty[NS], s_full[2], s_free[2], p_full[2], pv_done[2], q_full, drain
  l.misc_off = l.bar_off + 8 * (2 * num_stages + 10);
  l.mem_off = l.misc_off + 32;                        // member sequence ids [128]
  l.len_off = l.mem_off + kShRows * 4;                // member lengths [128]
  l.pre_off = l.len_off + kShRows * 4;                // own boxes before each member [129]
  l.meta_off = l.pre_off + (kShRows + 4) * 4;         // per slot, per box: owner + 1, tokens
  l.total = l.meta_off + num_stages * kShMaxBoxes * 4 + 1024;
  return l;
}

// Own stages of a chunk: the most own boxes any warp's queue holds (q_max),
// taken 32 / rb a stage when boxes are at most 32 tokens (one 32-column word
// per warp), else B = 128 / rb boxes a stage round robin over the warps.
__host__ __device__ inline int sh_own_stages(int q_max, int rb) {
  if (q_max <= 0) return 0;
  if (rb <= 32) return (q_max + 32 / rb - 1) / (32 / rb);
  const int b = 128 / rb;
  return (4 * q_max + b - 1) / b;
}

// Bits [lo, lo + n) of a 128-bit column mask held in four words.
__device__ __forceinline__ void sh_mask_set(uint32_t (&m)[4], int lo, int n) {
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const int a = max(lo, w * 32), b = min(lo + n, w * 32 + 32);
    if (a < b) m[w] |= (b - a == 32 ? 0xffffffffu : ((1u << (b - a)) - 1u)) << (a - w * 32);
  }
}

template <int N>
__device__ __forceinline__ float sh_tree_max(const float* v) {
  if constexpr (N == 1) {
    return v[0];
  } else {
    return fmaxf(sh_tree_max<N / 2>(v), sh_tree_max<N / 2>(v + N / 2));
  }
}

// A full stage (every column kept): the row's 128 scores (read at once by
// the caller), their maximum, then the weights of all of them from the same
// registers.  Whole warp.
__device__ __forceinline__ float sh_full_stage(float (&x)[kShTokens], float scale_log2,
                                               float& m_run, float& l_run, float& alpha,
                                               bool& rescale, int k, uint32_t prow) {
#pragma unroll
  for (int c = 0; c < kShTokens; ++c) x[c] *= scale_log2;
  const float mx = sh_tree_max<kShTokens>(x);
  alpha = 1.f;
  rescale = false;
  if (mx > m_run + kShLazyMax) {
    alpha = fast_exp2(m_run - mx);
    rescale = k > 0;
    m_run = mx;
  }
  l_run *= alpha;
  float lsum = 0.f;
#pragma unroll
  for (int w = 0; w < kShTokens / 32; ++w) {
    uint32_t pw[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const __nv_bfloat162 b = __floats2bfloat162_rn(fast_exp2(x[w * 32 + 2 * i] - m_run),
                                                     fast_exp2(x[w * 32 + 2 * i + 1] - m_run));
      pw[i] = *reinterpret_cast<const uint32_t*>(&b);
      lsum += bf16_lo(pw[i]) + bf16_hi(pw[i]);
    }
    tc::tmem_st16(prow + (uint32_t)(w * 16), pw);
  }
  return lsum;
}

// Word w (32 columns) of a 128-bit column mask.
__device__ __forceinline__ uint32_t sh_word(const uint32_t (&m)[4], int w) {
  return w == 0 ? m[0] : w == 1 ? m[1] : w == 2 ? m[2] : m[3];
}

// A packed stage with boxes of at most 32 tokens: this row attends only
// columns of its warp's word, whose 32 scores the caller read.  Their
// maximum under the mask, the lazy running maximum, then the weights of the
// word (0 outside the mask, rounded to bf16; the same rounded values enter
// P.V and the returned row sum) stored at `pword`.  Whole warp.
__device__ __forceinline__ float sh_word_stage(float (&v)[32], uint32_t bits, float scale_log2,
                                               float& m_run, float& l_run, float& alpha,
                                               bool& rescale, int k, uint32_t pword) {
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = ((bits >> i) & 1u) ? v[i] * scale_log2 : -INFINITY;
  const float mx = sh_tree_max<32>(v);
  alpha = 1.f;
  rescale = false;
  if (mx > m_run + kShLazyMax) {
    alpha = fast_exp2(m_run - mx);  // 0 while the row has seen nothing
    rescale = k > 0;
    m_run = mx;
  }
  l_run *= alpha;
  // (A row that has attended nothing yet keeps m = -inf: every weight 0.)
  const float m = m_run == -INFINITY ? 0.f : m_run;
  uint32_t pw[16];
  float part[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int t = q * 8 + 2 * i;
      pw[q * 4 + i] = pack_bf16x2(fast_exp2(v[t] - m), fast_exp2(v[t + 1] - m));
      acc += bf16_lo(pw[q * 4 + i]) + bf16_hi(pw[q * 4 + i]);
    }
    part[q] = acc;
  }
  tc::tmem_st16(pword, pw);
  return (part[0] + part[1]) + (part[2] + part[3]);
}

// Pass 1 of a stage: this row's largest score x = s * scale_log2 over the
// columns the mask keeps.  The stage's scores are read from tensor memory one
// 32-column word at a time, and a word no lane of the warp attends is
// skipped (not even read).  Whole warp.
__device__ __forceinline__ float sh_stage_max(uint32_t srow, const uint32_t (&mask)[4],
                                              float scale_log2) {
  float mx = -INFINITY;
#pragma unroll 1
  for (int w = 0; w < kShTokens / 32; ++w) {
    const uint32_t bits = sh_word(mask, w);
    if (!__any_sync(0xffffffffu, bits != 0u)) continue;
    float v[32];
    tc::tmem_ld<32>(srow + (uint32_t)(w * 32), v);
    tc::tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = ((bits >> i) & 1u) ? v[i] * scale_log2 : -INFINITY;
    mx = fmaxf(mx, sh_tree_max<32>(v));
  }
  return mx;
}

// Pass 2: the row's weights 2^(x - m) over the kept columns (0 elsewhere),
// rounded to bf16 (the same rounded values enter P.V and the row sum, which
// is returned), stored as the row of P in tensor memory at `prow` (two per
// 32-bit column).  A word no lane of the warp attends is stored as zeros
// without reading the scores.  Whole warp.
__device__ __forceinline__ float sh_stage_weights(uint32_t srow, const uint32_t (&mask)[4],
                                                  float scale_log2, float m, uint32_t prow) {
  float lsum = 0.f;
#pragma unroll 1
  for (int w = 0; w < kShTokens / 32; ++w) {
    const uint32_t bits = sh_word(mask, w);
    uint32_t pw[16];
    if (__any_sync(0xffffffffu, bits != 0u)) {
      float v[32];
      tc::tmem_ld<32>(srow + (uint32_t)(w * 32), v);
      tc::tmem_wait_ld();
      float part[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float acc = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int t = q * 8 + 2 * i;
          const float p0 = ((bits >> t) & 1u) ? fast_exp2(fmaf(v[t], scale_log2, -m)) : 0.f;
          const float p1 =
              ((bits >> (t + 1)) & 1u) ? fast_exp2(fmaf(v[t + 1], scale_log2, -m)) : 0.f;
          const __nv_bfloat162 b = __floats2bfloat162_rn(p0, p1);
          pw[q * 4 + i] = *reinterpret_cast<const uint32_t*>(&b);
          acc += bf16_lo(pw[q * 4 + i]) + bf16_hi(pw[q * 4 + i]);
        }
        part[q] = acc;
      }
      lsum += (part[0] + part[1]) + (part[2] + part[3]);
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) pw[i] = 0u;
    }
    tc::tmem_st16(prow + (uint32_t)(w * 16), pw);
  }
  return lsum;
}

// One event of the optional timeline: CTA (flattened grid index) and role
// (warp) select the record; compiled only into the timeline variant.
template <bool kTrace>
__device__ __forceinline__ void sh_trace(const SharedParams& p, int role, int& n, uint32_t tag,
                                         uint32_t arg) {
  if constexpr (kTrace) {
    if (p.trace != nullptr && n < p.trace_per_role) {
      const size_t cta = (size_t)p.trace_cta_base +
                         ((size_t)blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
      unsigned long long* e =
          p.trace + ((cta * kTcTraceRoles + role) * (size_t)p.trace_per_role + n) * 2;
      e[0] = (unsigned long long)clock64();
      e[1] = ((unsigned long long)tag << 32) | arg;
    }
    ++n;
  }
}

// One box of a stage, as the producer lane that owns it resolves it.
struct ShBox {
  int live;   // a box of this stage
  int seq;    // sequence whose table holds it
  int tok;    // its first token (position in that sequence)
  int cnt;    // tokens of it the sequence holds
  int owner;  // member index within the chunk, -1 for a shared box
  int last;   // holds the member's newest token
  int id;     // physical block
};

template <int D, bool kTrace>
__global__ void __launch_bounds__(kShThreads, 1)
    paged_decode_shared_kernel(const __grid_constant__ CUtensorMap kv_map,
                               const SharedParams p) {
  static_assert(D == 64 || D == 128, "shared-prefix decode handles head sizes 64 and 128");
  constexpr int kGroups = D / 64;
  constexpr int kChunkBytes = kGroups * 2048;  // one 8-token chunk of a stage: [group][8 K][8 V]
  constexpr uint32_t kIdescQK = tc::idesc_bf16_f32_ab(kShRows, kShTokens, 0, 0);
  constexpr uint32_t kIdescPV = tc::idesc_bf16_f32_ab(kShRows, D, 0, 1);
  constexpr uint32_t kQGroupBytes = kShRows * 128;   // a 64-column group of the query tile

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int NS = p.num_stages;
  const ShSmem lay = sh_smem_layout(D, NS);
  const int range = blockIdx.x;
  const int h = blockIdx.y;
  const int chunk = blockIdx.z;
  const int G = p.group;
  const int BS = p.block_size;
  const int l2bs = p.log2_block_size;
  const int Rb = p.box_rows;                   // tokens per box (one block, at most 128)
  const int l2rb = p.log2_box_rows;
  const int B = kShTokens >> l2rb;             // boxes per stage
  const int bw = Rb <= 32 ? 32 >> l2rb : 0;    // boxes per 32-column word (boxes of <= 32 tokens)

  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(base);
  const uint32_t q_s = sbase + lay.q_off;
  const uint32_t full0 = sbase + lay.bar_off;
  const uint32_t empty0 = full0 + 8u * NS;
  const uint32_t s_full = empty0 + 8u * NS;
  const uint32_t s_free = s_full + 16;
  const uint32_t p_full = s_full + 32;
  const uint32_t pv_done = s_full + 48;
  const uint32_t q_full = s_full + 64;
  const uint32_t drain = s_full + 72;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + lay.misc_off);
  volatile int* flags = reinterpret_cast<volatile int*>(base + lay.misc_off + 16);
  // flags[0] abort, flags[1] K/V stages issued, flags[2] unit refused
  int* mem_s = reinterpret_cast<int*>(base + lay.mem_off);
  int* mem_len = reinterpret_cast<int*>(base + lay.len_off);
  int* own_pre = reinterpret_cast<int*>(base + lay.pre_off);
  volatile int* meta = reinterpret_cast<volatile int*>(base + lay.meta_off);

  if (tid == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(full0 + 8u * i, 1);
      mbar_init(empty0 + 8u * i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(s_full + 8u * i, 1);
      mbar_init(s_free + 8u * i, 128);
      mbar_init(p_full + 8u * i, 128);
      mbar_init(pv_done + 8u * i, 1);
    }
    mbar_init(q_full, 128);
    mbar_init(drain, 1);
    flags[0] = 0;
    flags[1] = 0;
    flags[2] = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(smem_u32(tmem_slot), kShTmemCols);
    tc::tmem_relinquish();
  }
  if (tid == 32) tma_prefetch_desc(&kv_map);
  grid_dependency_wait();
  grid_dependents_launch();
  if (tid == 0) {
    int n0 = 0;
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    sh_trace<kTrace>(p, 0, n0, 30, (uint32_t)t);
  }

  // The unit: chunk record and members.  Every member must be a sequence of
  // the batch holding more than T tokens (its newest token stays its own)
  // within its table; otherwise the unit is refused.
  const int first = __ldg(p.chunks + 4 * chunk);
  const int nmem = __ldg(p.chunks + 4 * chunk + 1);
  const int T = __ldg(p.chunks + 4 * chunk + 2);
  // ceil(nmem / 4) members to a softmax warp, G rows each
  const bool bad = nmem < 1 || nmem > kShRows || ((nmem + 3) >> 2) * G > 32 || first < 0 ||
                   first > p.num_members - nmem || T < 1 || (T & (BS - 1)) != 0 ||
                   (T >> l2bs) > p.max_blocks_per_seq;
  tc::fence_before_sync();
  __syncthreads();  // barriers, flags and the tensor-memory address are set
  tc::fence_after_sync();
  if (!bad && tid < nmem) {
    const int s = __ldg(p.members + first + tid);
    const bool in_batch = s >= 0 && s < p.num_seqs;
    const int L = in_batch ? __ldg(p.seq_lens + s) : 0;
    const bool ok = in_batch && L > T && ((L + BS - 1) >> l2bs) <= p.max_blocks_per_seq;
    mem_s[tid] = ok ? s : -1;
    mem_len[tid] = ok ? L : T + 1;
    if (!ok) flags[2] = 1;
    // With one range the rows are final: the reduce leaves them alone.
    if (ok && range == 0) p.part_counts[s * p.num_kv_heads + h] = p.ranges > 1 ? p.ranges : 0;
  }
  if (bad && tid == 0) flags[2] = 1;
  __syncthreads();
  const bool refused = flags[2] != 0;
  // Own boxes before each member, in member order (a warp scan).
  if (warp == 0) {
    int carry = 0;
    if (lane == 0) own_pre[0] = 0;
    for (int c0 = 0; c0 < nmem && !refused && !bad; c0 += 32) {
      const int j = c0 + lane;
      int nb = j < nmem ? (mem_len[j] - T + Rb - 1) >> l2rb : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, nb, o);
        if (lane >= o) nb += v;
      }
      if (j < nmem) own_pre[j + 1] = carry + nb;
      carry += __shfl_sync(0xffffffffu, nb, 31);
    }
  }
  __syncthreads();
  const uint32_t tmem = *tmem_slot;
  // S0 S1 [128 columns each], P0 P1 [64 each: 128 bf16], O [D]
  const uint32_t tS = tmem, tP = tmem + 2 * kShTokens, tO = tmem + 3 * kShTokens;
  if (refused && tid == 0) record_error(p.err, PA_DEVERR_SEQ_LEN);
  const int per_warp = (nmem + 3) >> 2;  // members of each softmax warp
  // Own-box queue of warp w: the boxes of members [w * per_warp, ...).
  auto q_first = [&](int w) { return min(w * per_warp, max(nmem, 0)); };
  int q_max = 0;
  if (!refused && !bad)
    for (int w = 0; w < 4; ++w) q_max = max(q_max, own_pre[q_first(w + 1)] - own_pre[q_first(w)]);
  const int n_sh = (refused || bad) ? 0 : (int)(((long long)T + kShTokens - 1) / kShTokens);
  const int n_tot = n_sh + sh_own_stages(q_max, Rb);
  const int k_begin = (int)((long long)n_tot * range / p.ranges);
  const int k_end = (int)((long long)n_tot * (range + 1) / p.ranges);
  const int n = k_end - k_begin;  // this CTA's stages

  int ntr = warp == 0 ? 1 : 0;  // (the producer's record 0 is the start event)
  if (warp == 0) {
    // ---------------- producer ----------------
    if (lane == 0) sh_trace<kTrace>(p, 0, ntr, 31, (uint32_t)n);
    const uint32_t box_bytes = (uint32_t)Rb * (uint32_t)kGroups * 256u;
    const int chunks_per_block = BS >> 3;
    // Lane b resolves box b of global stage kg: a shared box of the first
    // member's table, or an own box: for boxes of up to 32 tokens, 32-column
    // word w of own stage o holds boxes o * bw .. o * bw + bw - 1 of warp w's
    // queue; wider boxes go round robin over the four queues.
    auto resolve = [&](int kg) {
      ShBox x{0, 0, 0, 0, -1, 0, 0};
      if (kg < n_sh) {
        x.tok = kg * kShTokens + lane * Rb;
        x.live = lane < B && x.tok < T;
        x.seq = mem_s[0];
        x.cnt = Rb;
      } else if (lane < B) {
        const int o = kg - n_sh;
        int w, pos;
        if (Rb <= 32) {
          w = lane / bw;
          pos = o * bw + (lane - w * bw);
        } else {
          const int gb = o * B + lane;
          w = gb & 3;
          pos = gb >> 2;
        }
        const int j0 = q_first(w), j1 = q_first(w + 1);
        const int qb = own_pre[j0];
        x.live = pos < own_pre[j1] - qb;
        if (x.live) {
          int lo = j0, hi = j1 - 1;  // the last member of the queue with own_pre[j] - qb <= pos
          while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (own_pre[mid] - qb <= pos) lo = mid; else hi = mid - 1;
          }
          x.owner = lo;
          x.seq = mem_s[lo];
          x.tok = T + (pos - (own_pre[lo] - qb)) * Rb;
          x.cnt = min(Rb, mem_len[lo] - x.tok);
          x.last = x.tok + x.cnt == mem_len[lo];
        }
      }
      if (x.live) x.id = __ldg(p.block_tables + (size_t)x.seq * p.max_blocks_per_seq + (x.tok >> l2bs));
      return x;
    };
    ShBox nx = n > 0 ? resolve(k_begin) : ShBox{0, 0, 0, 0, -1, 0, 0};
    bool ok = true;
    for (int k = 0; k < n; ++k) {
      const int slot = k % NS;
      const ShBox x = nx;
      if (k >= NS) {
        if (lane == 0) ok = mbar_wait_bounded(empty0 + 8u * slot, ((k / NS) - 1) & 1, p.err,
                                              p.wait_limit);
        ok = __shfl_sync(0xffffffffu, ok && !flags[0], 0);
        if (!ok) break;
      }
      if (lane == 0) sh_trace<kTrace>(p, 0, ntr, 32, (uint32_t)k);
      // What the softmax needs of each box: owner + 1 (0 = every row) and
      // the tokens it holds (0 = none: its rows are stale).
      if (lane < kShMaxBoxes)
        meta[slot * kShMaxBoxes + lane] = x.live ? ((x.owner + 1) << 16) | x.cnt : 0;
      const unsigned live_mask = __ballot_sync(0xffffffffu, x.live);
      // The fused cache write of each member whose newest token is here, into
      // the block the box is loaded from (its rows were fetched into L2 a
      // stage earlier, so each load is an L2 hit).
      unsigned wmask = __ballot_sync(0xffffffffu, x.live && x.last && p.new_k != nullptr);
      while (wmask) {
        const int b = __ffs(wmask) - 1;
        wmask &= wmask - 1;
        const int ws = __shfl_sync(0xffffffffu, x.seq, b);
        const int wpos = __shfl_sync(0xffffffffu, x.tok + x.cnt - 1, b);
        const int wid = __shfl_sync(0xffffffffu, x.id, b);
        const uint4 wv = load_new_token(p.new_k, p.new_v, ws, h, p.num_kv_heads, D * 2 / 16, lane);
        store_new_token(p.cache_w, wv, wid, h, wpos, p.num_kv_heads, D * 2 / 16, BS, p.num_blocks,
                        p.err, lane);
        fence_proxy_async_global();
        __syncwarp();
        fence_proxy_async_global();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive_expect_tx(full0 + 8u * slot, (uint32_t)__popc(live_mask) * box_bytes);
      __syncwarp();
      if (x.live) {
        const uint32_t kdst = sbase + (uint32_t)slot * (uint32_t)lay.stage;
        int c4 = x.id * chunks_per_block + ((x.tok & (BS - 1)) >> 3);
        if (x.id < 0 || x.id >= p.num_blocks) {
          record_error(p.err, PA_DEVERR_BLOCK_ID);
          c4 = p.num_blocks * chunks_per_block;  // outside the tensor: zero fill
        }
        tma_load_5d(kdst + (uint32_t)lane * box_bytes, &kv_map, full0 + 8u * slot, 0, 0, 0,
                    h * kGroups, c4);
      }
      if (lane == 0) {
        flags[1] = k + 1;
        sh_trace<kTrace>(p, 0, ntr, 33, (uint32_t)k);
      }
      // The next stage's boxes, resolved while this one loads and fetched
      // into L2 now: its slot frees only after a stage's round trip, and the
      // load then finds the rows in L2 instead of waiting on DRAM.
      if (k + 1 < n) {
        nx = resolve(k_begin + k + 1);
        if (nx.live && nx.id >= 0 && nx.id < p.num_blocks)
          tma_prefetch_l2_5d(&kv_map, 0, 0, 0, h * kGroups,
                             nx.id * chunks_per_block + ((nx.tok & (BS - 1)) >> 3));
        if (nx.live && nx.last && p.new_k != nullptr) {
          // The rows that stage writes (D * 2 bytes each of K and V).
          const size_t row = ((size_t)nx.seq * p.num_kv_heads + h) * (D * 2);
#pragma unroll
          for (int c = 0; c < D * 2; c += 128) {
            prefetch_l2(static_cast<const uint8_t*>(p.new_k) + row + c);
            prefetch_l2(static_cast<const uint8_t*>(p.new_v) + row + c);
          }
        }
      }
      if (lane == 0) sh_trace<kTrace>(p, 0, ntr, 34, (uint32_t)k);
    }
    if (!ok) flags[0] = 1;
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    // QK of stage k waits for its stage's data and for the softmax to have
    // read S of stage k - 2 (S is double-buffered; the softmax releases it
    // right after reading it), not for the PV of k - 2; PV waits for the
    // softmax's P (and any rescale of O) and then releases the stage slot.
    const bool leader = elect_one();
    int next_qk = 0, next_pv = 0;
    bool have_q = n == 0, ok = true;
    long long t_idle = clock64();
    const uint64_t qdesc = tc::smem_desc_sw128(q_s, 16, 1024);
    while (next_pv < n) {
      bool progress = false;
      if (!have_q && warp_test(q_full, 0)) {
        have_q = true;
        progress = true;
      }
      if (next_pv < next_qk) {
        const int j = next_pv, sb = j & 1, slot = j % NS;
        if (warp_test(p_full + 8u * sb, (j >> 1) & 1)) {
          tc::fence_after_sync();
          // A: P in tensor memory (16 tokens = 8 columns a step); B: the
          // stage's V rows read N-major (64-dimension groups 2048 apart,
          // 8-token groups kChunkBytes apart).
          const uint64_t b0 = tc::smem_desc_sw128(
              sbase + (uint32_t)slot * (uint32_t)lay.stage + 1024u, kGroups > 1 ? 2048 : 0,
              kChunkBytes);
          if (leader) {
#pragma unroll
            for (int kk = 0; kk < kShTokens / 16; ++kk) {
              const uint32_t boff = (uint32_t)(kk * 2 * kChunkBytes);
              tc::mma_bf16_tmem_a(tO, tP + (uint32_t)sb * 64u + (uint32_t)(kk * 8),
                                  b0 + (boff >> 4), kIdescPV, j > 0 || kk > 0);
            }
            tc::mma_commit(pv_done + 8u * sb);
            tc::mma_commit(empty0 + 8u * slot);
            sh_trace<kTrace>(p, 1, ntr, 36, (uint32_t)j);
          }
          __syncwarp();
          ++next_pv;
          progress = true;
        }
      }
      if (have_q && next_qk < n && next_qk < next_pv + 4) {
        const int k = next_qk, sb = k & 1, slot = k % NS;
        if (warp_test(full0 + 8u * slot, (k / NS) & 1) &&
            (k < 2 || warp_test(s_free + 8u * sb, ((k >> 1) - 1) & 1))) {
          tc::fence_after_sync();
          // A: the query tile (K-major, 8-row groups 1024 apart, 64-column
          // groups kQGroupBytes apart); B: the stage's K rows (K-major,
          // 8-token groups kChunkBytes apart, 64-column groups 2048 apart).
          const uint64_t b0 =
              tc::smem_desc_sw128(sbase + (uint32_t)slot * (uint32_t)lay.stage, 16, kChunkBytes);
          if (leader) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t aoff = (uint32_t)((kk >> 2) * kQGroupBytes + (kk & 3) * 32);
              const uint32_t boff = (uint32_t)((kk >> 2) * 2048 + (kk & 3) * 32);
              tc::mma_bf16(tS + (uint32_t)sb * kShTokens, qdesc + (aoff >> 4), b0 + (boff >> 4),
                           kIdescQK, kk > 0);
            }
            tc::mma_commit(s_full + 8u * sb);
            sh_trace<kTrace>(p, 1, ntr, 35, (uint32_t)k);
          }
          __syncwarp();
          ++next_qk;
          progress = true;
        }
      }
      const bool abort = __any_sync(0xffffffffu, flags[0] != 0);
      if (progress) {
        t_idle = clock64();
      } else if (abort) {
        ok = false;
        break;
      } else if (__any_sync(0xffffffffu, clock64() - t_idle > p.wait_limit)) {
        if (leader) record_error(p.err, PA_DEVERR_TIMEOUT);
        ok = false;
        break;
      } else if (next_pv < next_qk) {
        mbar_suspend(p_full + 8u * (next_pv & 1), (next_pv >> 1) & 1, 128);
      } else if (have_q && next_qk < n) {
        mbar_suspend(full0 + 8u * (next_qk % NS), (next_qk / NS) & 1, 128);
      } else if (!have_q) {
        mbar_suspend(q_full, 0, 128);
      }
    }
    if (!ok && leader) flags[0] = 1;
    if (leader) {
      tc::mma_commit(drain);
      mbar_wait_bounded(drain, 0, p.err);
    }
    __syncwarp();
  } else {
    // ---------------- query tile, softmax, output ----------------
    const int q4 = warp & 3;
    const int trow = q4 * 32 + lane;                 // tile row = tensor-memory lane
    const int jw = lane / G;
    const int g = lane - jw * G;
    const int jm0 = q4 * per_warp + jw;
    const bool row_ok = !refused && !bad && jw < per_warp && jm0 < nmem;  // a member's row
    const int jm = row_ok ? jm0 : -1;                // its member within the chunk
    const int s = row_ok ? mem_s[jm] : 0;
    const size_t grow = (size_t)s * p.num_heads + (size_t)h * G + g;  // global query row
    const uint32_t lane_addr = (uint32_t)(q4 * 32) << 16;
    // The query tile: this thread's row, 16 bytes at a time, into the
    // swizzled K-major layout (8-row atoms of 1024 bytes).
    {
      const uint4* src = reinterpret_cast<const uint4*>(p.query) + grow * (D / 8);
      const uint32_t rbase = q_s + (uint32_t)(trow >> 3) * 1024u + (uint32_t)(trow & 7) * 128u;
      uint4 v[D / 8];
#pragma unroll
      for (int c = 0; c < D / 8; ++c) v[c] = row_ok ? ldg_nc_v4(src + c) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int c = 0; c < D / 8; ++c) {
        const uint32_t addr = rbase + (uint32_t)(c >> 3) * kQGroupBytes +
                              (uint32_t)(((c & 7) ^ (trow & 7)) << 4);
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v[c].x),
                     "r"(v[c].y), "r"(v[c].z), "r"(v[c].w)
                     : "memory");
      }
      tc::fence_proxy_async_smem();
      mbar_arrive(q_full);
      if (lane == 0) sh_trace<kTrace>(p, warp, ntr, 37, 0u);
    }
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    uint32_t p_dirty = 3u;  // bit b: P buffer b may hold weights outside this warp's word
    for (int k = 0; k < n && ok; ++k) {
      const int kg = k_begin + k;
      const int sb = k & 1;
      const int slot = k % NS;
      // The stage's box table is readable once its data has landed, which
      // is before its scores are: the masks are built while QK runs.
      ok = mbar_wait_bounded(full0 + 8u * slot, (k / NS) & 1, p.err, p.wait_limit);
      ok = __all_sync(0xffffffffu, ok && !flags[0]);
      if (!ok) break;
      if (lane == 0) sh_trace<kTrace>(p, warp, ntr, 38, (uint32_t)k);
      // Columns this row attends: a shared stage's tokens below T, or the
      // boxes of this row's member (for boxes of up to 32 tokens only this
      // warp's word can hold them).  A token row of the stage is stale (its
      // V row is cleared before P.V) past its box's tokens.
      const bool shared_stage = kg < n_sh;
      const int nvalid = shared_stage ? min(kShTokens, T - kg * kShTokens) : 0;
      uint32_t mask[4] = {0u, 0u, 0u, 0u};
      uint32_t myword = 0u;   // packed stage, boxes of up to 32 tokens: word q4's bits
      int my_box_tokens = 0;  // tokens held by the box of token row trow
      if (shared_stage) {
        if (row_ok) sh_mask_set(mask, 0, nvalid);
        my_box_tokens = trow < nvalid ? Rb : 0;
      } else {
        my_box_tokens = meta[slot * kShMaxBoxes + (trow >> l2rb)] & 0xffff;
        const int mine = (jm + 1) << 16;  // owner field of this row's member
        if (Rb <= 32) {
          // Word q4 holds this warp's boxes: bw boxes of Rb columns.
          uint32_t m = 0u;
          for (int i = 0; i < bw; ++i) {
            const int e = meta[slot * kShMaxBoxes + q4 * bw + i];
            const int cnt = e & 0xffff;
            if (row_ok && (e & 0xffff0000) == mine)
              m |= (cnt >= 32 ? 0xffffffffu : ((1u << cnt) - 1u)) << (i * Rb);
          }
          myword = m;
        } else {
          for (int b = 0; b < B; ++b) {
            const int e = meta[slot * kShMaxBoxes + b];
            if (row_ok && (e & 0xffff0000) == mine) sh_mask_set(mask, b * Rb, e & 0xffff);
          }
        }
      }
      ok = mbar_wait_bounded(s_full + 8u * sb, (k >> 1) & 1, p.err, p.wait_limit);
      ok = __all_sync(0xffffffffu, ok && !flags[0]);
      if (!ok) break;
      tc::fence_after_sync();
      if (lane == 0) sh_trace<kTrace>(p, warp, ntr, 43, (uint32_t)k);
      const uint32_t srow = tS + (uint32_t)sb * kShTokens + lane_addr;
      const uint32_t prow = tP + (uint32_t)sb * 64u + lane_addr;
      float alpha = 1.f;
      bool rescale = false;
      float lw;
      const bool full_stage = shared_stage && nvalid == kShTokens;
      const bool word_stage = !shared_stage && Rb <= 32;
      // Scores of a full or a one-word stage are read first and S is
      // released at once, so the QK two stages on can start while this
      // stage's weights are computed.  P goes into buffer sb, which the PV of
      // stage k - 2 read.
      auto p_buffer_free = [&]() {
        bool w = true;
        if (k >= 2) w = mbar_wait_bounded(pv_done + 8u * sb, ((k >> 1) - 1) & 1, p.err,
                                          p.wait_limit);
        w = __all_sync(0xffffffffu, w && !flags[0]);
        tc::fence_after_sync();  // the P stores below come after that P.V
        return w;
      };
      if (full_stage) {
        float x[kShTokens];
#pragma unroll
        for (int c = 0; c < kShTokens / 32; ++c)
          tc::tmem_ld<32>(srow + (uint32_t)(c * 32), x + 32 * c);
        tc::tmem_wait_ld();
        tc::fence_before_sync();
        mbar_arrive(s_free + 8u * sb);
        if (!(ok = p_buffer_free())) break;
        // A full shared stage: every column, for every row (rows of no
        // member compute weights that are never stored).  The lazy maximum
        // is settled inside, before the weights.
        lw = sh_full_stage(x, p.scale_log2, m_run, l_run, alpha, rescale, k, prow);
        p_dirty |= 1u << sb;
      } else if (word_stage) {
        float v[32];
        tc::tmem_ld<32>(srow + (uint32_t)(q4 * 32), v);
        tc::tmem_wait_ld();
        tc::fence_before_sync();
        mbar_arrive(s_free + 8u * sb);
        if (!(ok = p_buffer_free())) break;
        lw = sh_word_stage(v, myword, p.scale_log2, m_run, l_run, alpha, rescale, k,
                           prow + (uint32_t)(q4 * 16));
        if (p_dirty & (1u << sb)) {
          // The other words of this buffer still hold an earlier stage's
          // weights: clear them once (later one-word stages keep them 0).
          uint32_t z[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) z[i] = 0u;
#pragma unroll
          for (int w = 0; w < 4; ++w)
            if (w != q4) tc::tmem_st16(prow + (uint32_t)(w * 16), z);
          p_dirty &= ~(1u << sb);
        }
      } else {
        // A shared stage with fewer than 128 tokens, or a packed stage of
        // boxes wider than 32 tokens: the mask's words, two passes.
        if (!(ok = p_buffer_free())) break;
        const float mx = sh_stage_max(srow, mask, p.scale_log2);
        // Lazy running maximum: moved only when this stage's scores exceed
        // it by more than kShLazyMax, so weights stay at most 2^kShLazyMax.
        if (mx > m_run + kShLazyMax) {
          alpha = fast_exp2(m_run - mx);  // 0 while the row has seen nothing
          rescale = k > 0;                // O holds earlier stages only from k = 1 on
          m_run = mx;
        }
        l_run *= alpha;
        // (A row that has attended nothing yet has m = -inf and weight 0.)
        lw = sh_stage_weights(srow, mask, p.scale_log2, m_run == -INFINITY ? 0.f : m_run, prow);
        tc::fence_before_sync();
        mbar_arrive(s_free + 8u * sb);
        p_dirty |= 1u << sb;
      }
      if (lane == 0) sh_trace<kTrace>(p, warp, ntr, 39, (uint32_t)k);
      if (row_ok) l_run += lw;
      if (__any_sync(0xffffffffu, rescale)) {
        // O holds the stages before k once the PV of stage k - 1 is done;
        // rescale this thread's row of it before the PV of stage k.  (P of
        // stage k is already written: only its P.V is held back.)
        ok = mbar_wait_bounded(pv_done + 8u * ((k - 1) & 1), ((k - 1) >> 1) & 1, p.err,
                               p.wait_limit);
        ok = __all_sync(0xffffffffu, ok && !flags[0]);
        if (!ok) break;
        tc::fence_after_sync();
        const float a = rescale ? alpha : 1.f;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          float o[32];
          tc::tmem_ld<32>(tO + lane_addr + (uint32_t)(c * 32), o);
          tc::tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= a;
          tc::tmem_st32(tO + lane_addr + (uint32_t)(c * 32), o);
        }
      }
      if (lane == 0) sh_trace<kTrace>(p, warp, ntr, 46, (uint32_t)k);
      tc::tmem_wait_st();
      if (lane == 0) sh_trace<kTrace>(p, warp, ntr, 47, (uint32_t)k);
      // Stale V rows (past a box's tokens, or boxes the stage does not have)
      // must not reach P.V: 0 * NaN would.  Each thread clears token row trow
      // if it is stale, its 16-byte pieces in a rotated order so that the
      // eight rows of an atom hit different banks.
      const bool stale = (trow & (Rb - 1)) >= my_box_tokens;
      if (stale) {
        const uint32_t vrow = sbase + (uint32_t)slot * (uint32_t)lay.stage + 1024u +
                              (uint32_t)((trow >> 3) * kChunkBytes + (trow & 7) * 128);
#pragma unroll
        for (int c = 0; c < 8; ++c)
#pragma unroll
          for (int gg = 0; gg < kGroups; ++gg)
            asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(
                             vrow + (uint32_t)(gg * 2048 + (((c + trow) & 7) << 4))),
                         "r"(0u)
                         : "memory");
      }
      if (__any_sync(0xffffffffu, stale)) tc::fence_proxy_async_smem();
      tc::fence_before_sync();
      mbar_arrive(p_full + 8u * sb);
      if (lane == 0) sh_trace<kTrace>(p, warp, ntr, 40, (uint32_t)k);
    }
    if (ok && n > 0) {
      ok = mbar_wait_bounded(pv_done + 8u * ((n - 1) & 1), ((n - 1) >> 1) & 1, p.err,
                             p.wait_limit);
      ok = __all_sync(0xffffffffu, ok && !flags[0]);
    }
    if (lane == 0) sh_trace<kTrace>(p, warp, ntr, 42, 0u);
    if (ok && n > 0) {
      // The rows go through shared memory (the stage ring, idle now that
      // every P.V is done; rows padded by 16 bytes), so that each warp then
      // stores its rows one whole row per instruction.
      tc::fence_after_sync();
      const bool some = l_run > 0.f;
      const float inv_l = some ? 1.f / l_run : 0.f;
      constexpr int kPitch = D + 4;  // floats per staged row
      float* rows = reinterpret_cast<float*>(base);
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        float o[32];
        tc::tmem_ld<32>(tO + lane_addr + (uint32_t)(c * 32), o);
        tc::tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; i += 4)
          *reinterpret_cast<float4*>(rows + trow * kPitch + c * 32 + i) =
              make_float4(o[i] * inv_l, o[i + 1] * inv_l, o[i + 2] * inv_l, o[i + 3] * inv_l);
      }
      const bool final_rows = p.ranges == 1;
      if (row_ok && !final_rows)
        p.part_lse[grow * (size_t)p.max_parts + (size_t)range] =
            some ? m_run + log2f(l_run) : -INFINITY;
      __syncwarp();
      // Row r of this warp: the global row and whether it is a member's,
      // from the lane that owns it.
      const size_t row_off = final_rows ? grow * D : (grow * (size_t)p.max_parts + range) * D;
#pragma unroll 4
      for (int r = 0; r < 32; ++r) {
        if (!__shfl_sync(0xffffffffu, row_ok, r)) continue;  // warp-uniform
        const size_t off = __shfl_sync(0xffffffffu, row_off, r);
        const float4 v = *reinterpret_cast<const float4*>(rows + (q4 * 32 + r) * kPitch + lane * 4);
        if (lane < D / 4) {
          if (final_rows) {
            const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
            const __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
            uint2 w;
            w.x = *reinterpret_cast<const uint32_t*>(&a);
            w.y = *reinterpret_cast<const uint32_t*>(&b);
            reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(p.out) + off)[lane] = w;
          } else {
            reinterpret_cast<float4*>(p.part_o + off)[lane] = v;
          }
        }
      }
    }
    if (lane == 0) sh_trace<kTrace>(p, warp, ntr, 41, 0u);
    if (!ok) flags[0] = 1;
  }

  tc::fence_before_sync();
  __syncthreads();
  if (tid == 0 && flags[0]) {
    // Wait (bounded, default limit) for every TMA load this CTA issued.
    const int issued = flags[1];
    for (int sl = 0; sl < NS && sl < issued; ++sl)
      mbar_wait_bounded(full0 + 8u * sl, ((issued - 1 - sl) / NS) & 1, p.err);
  }
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kShTmemCols);
  }
}

}  // namespace pa
