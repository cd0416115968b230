// Paged decode attention for sm_103a: TMA-staged K/V blocks, warp-level
// online softmax, fp32 accumulation; split-KV partials and their
// log-sum-exp reduce.
//
// The operation (studying-code.tistory.com/16, section "PagedAttention:
// 운영체제의 페이징 개념에서 영감을 받은 새로운 어텐션 알고리즘"; garden.houmin.site/
// infra/paged-attention, section "KV Cache 管理器"): the query of each sequence
// meets the key block K_j and value block V_j of every logical block j, found
// through the block table, and the per-block results are combined into o_i.
// Scores are scale * q.k with a softmax over the sequence's tokens.
//
// Work decomposition (one CTA = one (partition, KV head, sequence)):
//   warp 0      producer: walks the partition's block table (32 entries per
//               lane-parallel load) and issues TMA boxes into a ring of
//               shared-memory stages of 32 tokens, completing on the stage's
//               "full" mbarrier: with blocks of 8 tokens or more one box per
//               block holding its K and V rows of every 128-byte column group
//               (laid out [column group][K or V][rows]), else one box per
//               (block, column group, K or V);
//   warps 1..4  consumers: warp w takes stages w, w+C, ... (C consumer warps,
//               C dividing the number of stages, so that every ring slot has
//               a single owner and each slot's barrier phases are waited on in
//               order; a parity wait can only tell apart adjacent phases); per stage
//               QK      lane j owns token j and computes all G = Hq/Hkv query
//                       heads' scores (query heads of a GQA group share the K
//                       load), reading the row through the 128-byte swizzle;
//               softmax warp max per head, rescale factor 2^(m_old - m_new),
//                       p_j = 2^(s_j - m_new) written to a per-warp buffer;
//               PV      lane (chunk c, token group r) accumulates
//                       p_j[g] * v_j[c*8 .. c*8+7] for tokens j = r mod R;
//               then releases the stage ("empty" mbarrier) to the producer.
//   end         per-warp (m, l, o) merged across warps by log-sum-exp and
//               written as the final output or as a split-KV partial.
// Scores live in the log2 domain: q is pre-multiplied by scale * log2(e) so
// that exp(x - m) becomes 2^(x' - m').
#pragma once

#include "pa_device.cuh"

namespace pa {

constexpr int kConsumerWarps = 4;
constexpr int kDecodeThreads = 32 * (kConsumerWarps + 1);
constexpr int kStageTokens = 32;
constexpr int kPStride = 8;  // floats per token in the per-warp softmax-weight buffer
constexpr int kLongestFirstMaxSeqs = 128;  // batches the CUDA-core kernel ranks by length

struct DecodeParams {
  void* out;                    // [S][Hq][D] of T (final rows)
  const void* query;            // [S][Hq][D] of T
  const int32_t* block_tables;  // [S][max_blocks_per_seq]
  const int32_t* seq_lens;      // [S]
  float* part_o;                // [S][Hq][max_parts][D]: normalised partial outputs
  float* part_lse;              // [S][Hq][max_parts]: log2-domain log-sum-exp of each partial
  unsigned int* err;            // device error word
  unsigned int* sched;          // tensor-core kernel: [0] next work item, [1] CTAs finished
  int total_items;              // tensor-core kernel: num_seqs * num_kv_heads * max_parts
                                // (balanced split: the number of stage ranges)
  int dense_items;              // tensor-core kernel: number only the real work items
  int longest_first;            // CUDA-core kernel: grid z is a rank in decreasing length order
  int balanced;                 // tensor-core kernel: stage-balanced split (ranges of stages)
  int32_t* part_counts;         // balanced split: [S][Hkv] pieces of each pair (1 = final rows)
  int num_seqs;
  uint8_t* cache_w;             // the pool, for the fused cache write (pa_decode_append)
  const void* new_k;            // [S][Hkv][D] newest token's keys, or null (no fused write)
  const void* new_v;            // [S][Hkv][D] newest token's values
  unsigned long long* trace;    // tensor-core kernel timeline, or null
  int trace_per_role;
  size_t trace_bytes;
  int num_blocks;
  int block_size;
  int log2_block_size;
  int num_kv_heads;
  int num_heads;
  int group;             // query heads per KV head
  int max_blocks_per_seq;
  int partition_tokens;  // 0 = the whole sequence in one CTA
  int max_parts;         // grid.x in split mode
  float scale_log2;      // scale * log2(e)
  // shared-memory geometry, bytes
  int box_rows;          // tokens per TMA box: min(block_size, tokens per stage)
  int log2_box_rows;
  int group_slot;        // bytes between a box's 128-byte column groups
  int region_bytes;      // bytes from a K row to the same V row
  int box_stride;        // bytes between consecutive boxes of a stage
  int kv_boxes;          // 1: one TMA box per block holds K and V of every column group
  int stage_bytes;       // bytes of one stage
  int num_stages;        // a multiple of num_consumers
  int num_consumers;     // consumer warps that take stages (1..kConsumerWarps)
  int stage_area;        // bytes before the query buffer (stages, or the merge overlay)
  long long wait_limit;  // tensor-core kernel: SM cycles a pipeline wait may take
  // Tensor-core kernel next to a shared-prefix decode: sequences with
  // seq_start[s] > 0 belong to a group the group kernel covers (rows and
  // partial counts) and are skipped; the others are decoded as usual.
  const int32_t* seq_start;
};

// Dynamic shared memory a decode launch needs (the kernel aligns its base to 1024).
inline int decode_smem_bytes(int stage_area, int group, int head_size) {
  int bytes = 1024 + stage_area;
  bytes += group * head_size * 4;                      // pre-scaled fp32 query
  bytes += kConsumerWarps * kStageTokens * kPStride * 4;  // softmax weights
  bytes += 2 * 64 * 8;                                 // up to 64 stages x (full, empty)
  bytes += 16;                                         // flags
  return bytes;
}

// Bytes of the cross-warp merge overlay: m, l and o of every consumer warp.
inline int decode_merge_bytes(int group, int head_size) {
  return kConsumerWarps * group * (head_size + 2) * 4;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <typename T, int D, int G>
__global__ void __launch_bounds__(kDecodeThreads, 2)
    paged_decode_kernel(const __grid_constant__ CUtensorMap kv_map, const DecodeParams p) {
  using E = ElemTraits<T>;
  constexpr int kRowBytes = D * E::kBytes;
  constexpr int kChunks = kRowBytes / 16;             // 16-byte chunks per token row
  constexpr int kGroups = kRowBytes / 128;            // 128-byte column groups per row
  constexpr int kEPC = E::kPerChunk;                  // elements per chunk
  constexpr int kCPL = kChunks > 32 ? kChunks / 32 : 1;  // PV chunks per lane
  constexpr int kRpv = kChunks >= 32 ? 1 : 32 / kChunks;  // PV token groups per warp
  static_assert(kRowBytes % 128 == 0, "head rows must be whole 128-byte groups");
  static_assert(G >= 1 && G <= kPStride, "group size");

  const int part = blockIdx.x;
  const int h = blockIdx.y;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

  grid_dependency_wait();
  int s = blockIdx.z;
  int L;
  if (p.longest_first) {
    // Longest first: CTAs are dispatched in grid order, so grid z = r takes
    // the sequence of rank r in decreasing length (ties by index) and the
    // shortest work is left for the tail.  The lengths sit in the stage
    // area, unused until the barrier after the query load.
    __shared__ int pick[2];
    int* lens = reinterpret_cast<int*>(base);
    for (int i = tid; i < p.num_seqs; i += blockDim.x) lens[i] = p.seq_lens[i];
    __syncthreads();
    for (int i = tid; i < p.num_seqs; i += blockDim.x) {
      const int li = lens[i];
      int r = 0;
      for (int u = 0; u < p.num_seqs; ++u) {
        const int lu = lens[u];
        r += (lu > li) || (lu == li && u < i);
      }
      if (r == (int)blockIdx.z) {
        pick[0] = i;
        pick[1] = li;
      }
    }
    __syncthreads();
    s = pick[0];
    L = pick[1];
  } else {
    L = p.seq_lens[s];
  }
  const int P = p.partition_tokens;
  const bool split = P > 0;
  const int nparts = L <= 0 ? 0 : (split ? (L + P - 1) / P : 1);
  const size_t row0 = (size_t)s * p.num_heads + (size_t)h * G;  // first query row

  if (L <= 0) {
    if (part == 0) {
      T* out = reinterpret_cast<T*>(p.out) + row0 * D;
      for (int i = tid; i < G * D; i += blockDim.x) out[i] = E::from_float(0.f);
    }
    return;
  }
  if ((split && nparts > p.max_parts) ||
      ((L + p.block_size - 1) >> p.log2_block_size) > p.max_blocks_per_seq) {
    if (part == 0 && tid == 0) record_error(p.err, PA_DEVERR_SEQ_LEN);
    return;
  }
  if (part >= nparts) return;

  const int tok0 = split ? part * P : 0;
  const int tok1 = split ? min(L, tok0 + P) : L;
  const int n_stages = (tok1 - tok0 + kStageTokens - 1) / kStageTokens;
  const int NS = p.num_stages;

  const uint32_t sbase = smem_u32(base);
  float* q_s = reinterpret_cast<float*>(base + p.stage_area);
  float* p_all = q_s + G * D;
  uint64_t* bars = reinterpret_cast<uint64_t*>(p_all + kConsumerWarps * kStageTokens * kPStride);
  volatile int* flags = reinterpret_cast<volatile int*>(bars + 2 * 64);
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8u * NS;

  if (tid == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(full0 + 8u * i, 1);
      mbar_init(empty0 + 8u * i, 1);
    }
    flags[0] = 0;  // abort
    flags[1] = 0;  // stages issued
    fence_mbar_init();
  }
  if (tid == 32) tma_prefetch_desc(&kv_map);
  {
    const T* qg = reinterpret_cast<const T*>(p.query) + row0 * D;
    for (int i = tid; i < G * D; i += blockDim.x) q_s[i] = E::to_float(qg[i]) * p.scale_log2;
  }
  __syncthreads();

  const int R = p.box_rows;
  const int log2R = p.log2_box_rows;
  const int gslot = p.group_slot;
  const int region = p.region_bytes;

  // Consumer state (the producer warp leaves it unused).
  float m_run[G], l_run[G];
  float o[G][kCPL * kEPC];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    m_run[g] = -INFINITY;
    l_run[g] = 0.f;
#pragma unroll
    for (int e = 0; e < kCPL * kEPC; ++e) o[g][e] = 0.f;
  }
  // PV lane roles: chunk index (first of kCPL) and token group.
  const int pv_c = kChunks >= 32 ? lane : lane % kChunks;
  const int pv_r = kChunks >= 32 ? 0 : lane / kChunks;

  if (warp == 0) {
    // ---------------- producer ----------------
    const int BS = p.block_size;
    const int l2bs = p.log2_block_size;
    const int32_t* table = p.block_tables + (size_t)s * p.max_blocks_per_seq;
    const int lb_end = (tok1 + BS - 1) >> l2bs;  // one past the last logical block
    int win = tok0 >> l2bs;                      // logical block held by lane 0 of `cur`
    int cur = (win + lane < lb_end) ? __ldg(table + win + lane) : 0;
    int nxt = (win + 32 + lane < lb_end) ? __ldg(table + win + 32 + lane) : 0;
    const uint32_t box_bytes = p.kv_boxes ? (uint32_t)R * (uint32_t)kGroups * 256u : (uint32_t)R * 128u;
    const uint32_t stage_tx = p.kv_boxes ? box_bytes : (uint32_t)(kGroups * 2) * box_bytes;
    int issued = 0;
    for (int k = 0; k < n_stages; ++k) {
      const int slot = k % NS;
      if (k >= NS) {
        bool ok = true;
        if (lane == 0) ok = mbar_wait_bounded(empty0 + 8u * slot, ((k / NS) - 1) & 1, p.err);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok || flags[0]) {
          flags[0] = 1;
          break;
        }
      }
      const int st_tok = tok0 + k * kStageTokens;
      const int st_n = min(kStageTokens, tok1 - st_tok);
      const int nbox = (st_n + R - 1) >> log2R;
      if (p.new_k != nullptr && tok1 == L && k == n_stages - 1)  // fused write of the newest token
        write_new_token(p.cache_w, p.new_k, p.new_v, table, s, h, L - 1, p.num_kv_heads,
                        kRowBytes / 16, BS, l2bs, p.num_blocks, p.err, lane);
      if (lane == 0) mbar_arrive_expect_tx(full0 + 8u * slot, (uint32_t)nbox * stage_tx);
      __syncwarp();
      const uint32_t kdst = sbase + (uint32_t)slot * (uint32_t)p.stage_bytes;
      if (p.kv_boxes) {
        // One box per block, issued by one lane each (a stage holds at most
        // 32 / 8 = 4 boxes, all inside the table window).
        const int tk = st_tok + (min(lane, nbox - 1) << log2R);
        const int lb = tk >> l2bs;
        while ((st_tok >> l2bs) >= win + 32) {
          cur = nxt;
          win += 32;
          nxt = (win + 32 + lane < lb_end) ? __ldg(table + win + 32 + lane) : 0;
        }
        const int src = lb - win;  // 0 .. 34
        const int id_cur = __shfl_sync(0xffffffffu, cur, src & 31);
        const int id_nxt = __shfl_sync(0xffffffffu, nxt, src & 31);
        if (lane < nbox) {
          int id = src < 32 ? id_cur : id_nxt;
          if (id < 0 || id >= p.num_blocks) {
            record_error(p.err, PA_DEVERR_BLOCK_ID);
            id = p.num_blocks;  // outside the tensor: zero fill
          }
          tma_load_5d(kdst + (uint32_t)lane * (uint32_t)p.box_stride, &kv_map, full0 + 8u * slot,
                      0, tk & (BS - 1), 0, h * kGroups, id);
        }
      }
      for (int i = 0; !p.kv_boxes && i < nbox; ++i) {
        const int tk = st_tok + (i << log2R);
        const int lb = tk >> l2bs;
        const int t0 = tk & (BS - 1);
        while (lb >= win + 32) {
          cur = nxt;
          win += 32;
          nxt = (win + 32 + lane < lb_end) ? __ldg(table + win + 32 + lane) : 0;
        }
        const int id = __shfl_sync(0xffffffffu, cur, lb - win);
        if (lane == 0) {
          int ck = id, cv = p.num_blocks + id;
          if (id < 0 || id >= p.num_blocks) {
            // Outside the tensor: the box reads the zero fill instead of another block.
            record_error(p.err, PA_DEVERR_BLOCK_ID);
            ck = cv = 2 * p.num_blocks;
          }
#pragma unroll
          for (int g = 0; g < kGroups; ++g) {
            const uint32_t dst = kdst + (uint32_t)i * (uint32_t)p.box_stride + (uint32_t)g * gslot;
            tma_load_5d(dst, &kv_map, full0 + 8u * slot, 0, g, h, t0, ck);
            tma_load_5d(dst + region, &kv_map, full0 + 8u * slot, 0, g, h, t0, cv);
          }
        }
      }
      issued = k + 1;
    }
    if (lane == 0) flags[1] = issued;
  } else {
    // ---------------- consumers ----------------
    const int w = warp - 1;
    float* p_w = p_all + w * kStageTokens * kPStride;
    const uint32_t p_w_s = smem_u32(p_w);
    const uint32_t q_s_s = smem_u32(q_s);


    // This lane's token in the QK phase and its row position inside a stage.
    const int qk_box = lane >> log2R;
    const int qk_t = lane & (R - 1);
    const uint32_t qk_off = (uint32_t)qk_box * (uint32_t)p.box_stride + (uint32_t)qk_t * 128u;
    const uint32_t qk_swz = (uint32_t)(qk_t & 7);

    const int nc = p.num_consumers;
    for (int k = w; w < nc && k < n_stages; k += nc) {
      if (flags[0]) break;
      const int slot = k % NS;
      bool ok = mbar_wait_bounded(full0 + 8u * slot, (k / NS) & 1, p.err);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) {
        flags[0] = 1;
        break;
      }
      const int st_tok = tok0 + k * kStageTokens;
      const int nvalid = min(kStageTokens, tok1 - st_tok);
      const uint32_t kreg = sbase + (uint32_t)slot * (uint32_t)p.stage_bytes;
      const uint32_t vreg = kreg + region;

      // ---- scores: lane = token ----
      float acc[G];
#pragma unroll
      for (int g = 0; g < G; ++g) acc[g] = 0.f;
#pragma unroll
      for (int c = 0; c < kChunks; ++c) {
        const uint32_t addr = kreg + qk_off + (uint32_t)(c >> 3) * gslot +
                              ((((uint32_t)c & 7u) ^ qk_swz) << 4);
        float kf[kEPC];
        E::unpack(lds128(addr), kf);
#pragma unroll
        for (int g = 0; g < G; ++g) {
#pragma unroll
          for (int e4 = 0; e4 < kEPC; e4 += 4) {
            const float4 qv = lds128f(q_s_s + (uint32_t)((g * D + c * kEPC + e4) * 4));
            acc[g] = fmaf(qv.x, kf[e4 + 0], acc[g]);
            acc[g] = fmaf(qv.y, kf[e4 + 1], acc[g]);
            acc[g] = fmaf(qv.z, kf[e4 + 2], acc[g]);
            acc[g] = fmaf(qv.w, kf[e4 + 3], acc[g]);
          }
        }
      }
      const bool valid = lane < nvalid;

      // ---- online softmax over this stage (log2 domain) ----
      float alpha[G];
      float pj[kPStride];
#pragma unroll
      for (int g = 0; g < kPStride; ++g) pj[g] = 0.f;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float sc = valid ? acc[g] : -INFINITY;
        const float m_new = fmaxf(m_run[g], warp_max(sc));
        alpha[g] = fast_exp2(m_run[g] - m_new);
        m_run[g] = m_new;
        pj[g] = fast_exp2(sc - m_new);
        l_run[g] = fmaf(l_run[g], alpha[g], pj[g]);
      }
      {
        float4* dst = reinterpret_cast<float4*>(p_w + lane * kPStride);
        dst[0] = make_float4(pj[0], pj[1], pj[2], pj[3]);
        if (G > 4) dst[1] = make_float4(pj[4], pj[5], pj[6], pj[7]);
      }
      __syncwarp();

      // ---- values: lane = (chunk, token group) ----
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int e = 0; e < kCPL * kEPC; ++e) o[g][e] *= alpha[g];
      for (int j = pv_r; j < nvalid; j += kRpv) {
        const int box = j >> log2R;
        const int t = j & (R - 1);
        const uint32_t rowbase = vreg + (uint32_t)box * (uint32_t)p.box_stride + (uint32_t)t * 128u;
        float pw[kPStride];
        {
          const float4 a = lds128f(p_w_s + (uint32_t)(j * kPStride * 4));
          pw[0] = a.x; pw[1] = a.y; pw[2] = a.z; pw[3] = a.w;
          if (G > 4) {
            const float4 b = lds128f(p_w_s + (uint32_t)(j * kPStride * 4 + 16));
            pw[4] = b.x; pw[5] = b.y; pw[6] = b.z; pw[7] = b.w;
          }
        }
#pragma unroll
        for (int cc = 0; cc < kCPL; ++cc) {
          const int c = pv_c + cc * 32;
          const uint32_t addr = rowbase + (uint32_t)(c >> 3) * gslot +
                                ((((uint32_t)c & 7u) ^ ((uint32_t)t & 7u)) << 4);
          float vf[kEPC];
          E::unpack(lds128(addr), vf);
#pragma unroll
          for (int g = 0; g < G; ++g)
#pragma unroll
            for (int e = 0; e < kEPC; ++e) o[g][cc * kEPC + e] = fmaf(pw[g], vf[e], o[g][cc * kEPC + e]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8u * slot);
    }

    // Per-warp totals: l over lanes, o over token groups.
#pragma unroll
    for (int g = 0; g < G; ++g) l_run[g] = warp_sum(l_run[g]);
    if (kRpv > 1) {
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int e = 0; e < kCPL * kEPC; ++e)
#pragma unroll
          for (int off = kChunks; off < 32; off <<= 1)
            o[g][e] += __shfl_xor_sync(0xffffffffu, o[g][e], off);
    }
  }
  __syncthreads();  // (A) every stage consumed: the stage area is free for the merge
  if (warp > 0 && !flags[0]) {
    const int w = warp - 1;
    float* Mw = reinterpret_cast<float*>(base);
    float* Lw = Mw + kConsumerWarps * G;
    float* Ow = Lw + kConsumerWarps * G;
    if (lane == 0) {
#pragma unroll
      for (int g = 0; g < G; ++g) {
        Mw[w * G + g] = m_run[g];
        Lw[w * G + g] = l_run[g];
      }
    }
    if (pv_r == 0) {
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int cc = 0; cc < kCPL; ++cc)
#pragma unroll
          for (int e = 0; e < kEPC; ++e)
            Ow[(w * G + g) * D + (pv_c + cc * 32) * kEPC + e] = o[g][cc * kEPC + e];
    }
  }

  if (flags[0]) {
    // A wait gave up.  Before leaving, wait (bounded) for every TMA load this
    // CTA issued, so that no copy into its shared memory is still in flight.
    if (tid == 0) {
      const int issued = flags[1];
      for (int sl = 0; sl < NS && sl < issued; ++sl) {
        const int last_use = (issued - 1 - sl) / NS;
        mbar_wait_bounded(full0 + 8u * sl, last_use & 1, p.err);
      }
    }
    return;
  }
  __syncthreads();  // (B) merge data written

  {
    const float* Mw = reinterpret_cast<const float*>(base);
    const float* Lw = Mw + kConsumerWarps * G;
    const float* Ow = Lw + kConsumerWarps * G;
    for (int i = tid; i < G * D; i += blockDim.x) {
      const int g = i / D;
      const int d = i - g * D;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, Mw[w * G + g]);
      float lsum = 0.f, osum = 0.f;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) {
        const float sc = fast_exp2(Mw[w * G + g] - M);
        lsum = fmaf(Lw[w * G + g], sc, lsum);
        osum = fmaf(Ow[(w * G + g) * D + d], sc, osum);
      }
      const float val = osum / lsum;
      if (nparts == 1) {
        reinterpret_cast<T*>(p.out)[(row0 + g) * D + d] = E::from_float(val);
      } else {
        const size_t prow = (row0 + g) * (size_t)p.max_parts + part;
        p.part_o[prow * D + d] = val;
        if (d == 0) p.part_lse[prow] = M + log2f(lsum);
      }
    }
  }
}

// Log-sum-exp combination for rows of few partitions (up to
// kReduceRowParts): one warp per (sequence, query head) row, eight rows per
// CTA; each lane owns D/32 output columns and walks the row's partitions
// with four loads in flight.  Same arithmetic as lse_reduce_kernel.
constexpr int kReduceRowParts = 16;
constexpr int kReduceRowSpec = 4;  // partials loaded before the row's count is known

template <typename T, int D>
__global__ void __launch_bounds__(256)
    lse_reduce_rows_kernel(void* out_, const float* __restrict__ part_o,
                           const float* __restrict__ part_lse,
                           const int32_t* __restrict__ seq_lens,
                           const int32_t* __restrict__ counts, int group, int num_seqs,
                           int num_heads, int partition_tokens, int max_parts) {
  using E = ElemTraits<T>;
  constexpr int kPer = D / 32;  // columns per lane: 2, 4 or 8
  static_assert(D % 64 == 0, "row reduce columns");
  const int lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  grid_dependency_wait();
  if (row >= (long long)num_seqs * num_heads) return;
  // Every load of a row of up to kReduceRowSpec partials is issued at once,
  // before the row's partial count arrives (one round trip instead of
  // three): the count, lane q's log-sum-exp and the first partials'
  // columns.  Slots past the count hold stale values and are masked.
  const float* lse = part_lse + (size_t)row * max_parts;
  const float* po = part_o + (size_t)row * max_parts * D + lane * kPer;
  const float lse_l = lane < max_parts ? lse[lane] : -INFINITY;
  float v0[kReduceRowSpec][kPer];
#pragma unroll
  for (int q = 0; q < kReduceRowSpec; ++q)
#pragma unroll
    for (int e = 0; e < kPer; e += 2) {
      float2 t = make_float2(0.f, 0.f);
      if (q < max_parts) t = *reinterpret_cast<const float2*>(po + (size_t)q * D + e);
      v0[q][e] = t.x;
      v0[q][e + 1] = t.y;
    }
  int nparts;
  if (counts != nullptr) {
    nparts = counts[row / group];  // pieces of the row's (sequence, KV head) pair
  } else {
    const int L = seq_lens[row / num_heads];
    nparts = L <= 0 ? 0 : (L + partition_tokens - 1) / partition_tokens;
  }
  if (nparts <= 1 || nparts > max_parts) return;  // written by the decode kernel (or an error)
  const float M = warp_max(lane < nparts ? lse_l : -INFINITY);
  float w_own = lane < nparts ? fast_exp2(lse_l - M) : 0.f;
  const float wsum = warp_sum(w_own);
  float acc[kPer];
#pragma unroll
  for (int e = 0; e < kPer; ++e) acc[e] = 0.f;
#pragma unroll
  for (int q = 0; q < kReduceRowSpec; ++q) {
    const float w = __shfl_sync(0xffffffffu, w_own, q);
    if (q < nparts)  // a stale slot may hold anything, even NaN
#pragma unroll
      for (int e = 0; e < kPer; ++e) acc[e] = fmaf(w, v0[q][e], acc[e]);
  }
  for (int q = kReduceRowSpec; q < nparts; ++q) {
    const float w = __shfl_sync(0xffffffffu, w_own, q);
    float v[kPer];
#pragma unroll
    for (int e = 0; e < kPer; e += 2) {
      const float2 t = *reinterpret_cast<const float2*>(po + (size_t)q * D + e);
      v[e] = t.x;
      v[e + 1] = t.y;
    }
#pragma unroll
    for (int e = 0; e < kPer; ++e) acc[e] = fmaf(w, v[e], acc[e]);
  }
  T* out = reinterpret_cast<T*>(out_) + (size_t)row * D + lane * kPer;
#pragma unroll
  for (int e = 0; e < kPer; ++e) out[e] = E::from_float(acc[e] / wsum);
}

// Log-sum-exp combination of split-KV partials:
//   M = max_p lse_p,  w_p = 2^(lse_p - M),  out = sum_p w_p o_p / sum_p w_p.
// One CTA per (query head, sequence, `cols` output columns): cols = D, or 32
// when rows have many partitions (more CTAs share a long row).  Its threads
// are cols/4 float4 columns x (1024/cols) partition slices; each sums its
// slice's partials (four loads in flight), and the slices are added through
// shared memory.  The weights of up to kReduceChunk partitions at a time are
// staged in shared memory.
constexpr int kReduceThreads = 256;
constexpr int kReduceChunk = 1024;
constexpr int kReduceMinCols = 32;

template <typename T, int D>
__global__ void __launch_bounds__(kReduceThreads, 4)
    lse_reduce_kernel(void* out_, const float* __restrict__ part_o,
                      const float* __restrict__ part_lse, const int32_t* __restrict__ seq_lens,
                      const int32_t* __restrict__ counts, int group, int num_heads,
                      int partition_tokens, int max_parts, int cols) {
  using E = ElemTraits<T>;
  static_assert(D % kReduceMinCols == 0, "reduce columns");
  constexpr int kRowF4 = D / 4;  // float4 columns of a partial row
  __shared__ float w_s[kReduceChunk];
  __shared__ __align__(16) float acc_s[kReduceThreads * 4];
  __shared__ float red_s[kReduceThreads / 32];
  __shared__ float bcast_s;

  const int hq = blockIdx.x;
  const int s = blockIdx.y;
  const int col0 = blockIdx.z * cols;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  grid_dependency_wait();
  const size_t row = (size_t)s * num_heads + hq;
  int nparts;
  if (counts != nullptr) {
    nparts = counts[row / group];  // pieces of the row's (sequence, KV head) pair
  } else {
    const int L = seq_lens[s];
    nparts = L <= 0 ? 0 : (L + partition_tokens - 1) / partition_tokens;
  }
  if (nparts <= 1 || nparts > max_parts) return;  // written by the decode kernel (or an error)
  const float* lse = part_lse + row * max_parts;
  const float4* po = reinterpret_cast<const float4*>(part_o + row * max_parts * D + col0);

  // M over the row's partitions.
  float m = -INFINITY;
  for (int q = tid; q < nparts; q += kReduceThreads) m = fmaxf(m, lse[q]);
  m = warp_max(m);
  if (lane == 0) red_s[warp] = m;
  __syncthreads();
  if (tid == 0) {
    float v = red_s[0];
    for (int i = 1; i < kReduceThreads / 32; ++i) v = fmaxf(v, red_s[i]);
    bcast_s = v;
  }
  __syncthreads();
  const float M = bcast_s;

  const int ncol4 = cols >> 2;
  const int col = tid % ncol4;
  const int slice = tid / ncol4;
  const int nslices = kReduceThreads / ncol4;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float wsum = 0.f;
  for (int c0 = 0; c0 < nparts; c0 += kReduceChunk) {
    const int cn = min(kReduceChunk, nparts - c0);
    if (c0 > 0) __syncthreads();  // the previous chunk's weights are consumed
    for (int q = tid; q < cn; q += kReduceThreads) {
      const float w = fast_exp2(lse[c0 + q] - M);
      w_s[q] = w;
      wsum += w;
    }
    __syncthreads();
    int q = slice;
    for (; q + 3 * nslices < cn; q += 4 * nslices) {
      const float4 a = po[(size_t)(c0 + q) * kRowF4 + col];
      const float4 b = po[(size_t)(c0 + q + nslices) * kRowF4 + col];
      const float4 c = po[(size_t)(c0 + q + 2 * nslices) * kRowF4 + col];
      const float4 d = po[(size_t)(c0 + q + 3 * nslices) * kRowF4 + col];
      const float wa = w_s[q], wb = w_s[q + nslices], wc = w_s[q + 2 * nslices],
                  wd = w_s[q + 3 * nslices];
      acc.x = fmaf(wa, a.x, acc.x); acc.y = fmaf(wa, a.y, acc.y);
      acc.z = fmaf(wa, a.z, acc.z); acc.w = fmaf(wa, a.w, acc.w);
      acc.x = fmaf(wb, b.x, acc.x); acc.y = fmaf(wb, b.y, acc.y);
      acc.z = fmaf(wb, b.z, acc.z); acc.w = fmaf(wb, b.w, acc.w);
      acc.x = fmaf(wc, c.x, acc.x); acc.y = fmaf(wc, c.y, acc.y);
      acc.z = fmaf(wc, c.z, acc.z); acc.w = fmaf(wc, c.w, acc.w);
      acc.x = fmaf(wd, d.x, acc.x); acc.y = fmaf(wd, d.y, acc.y);
      acc.z = fmaf(wd, d.z, acc.z); acc.w = fmaf(wd, d.w, acc.w);
    }
    for (; q < cn; q += nslices) {
      const float4 a = po[(size_t)(c0 + q) * kRowF4 + col];
      const float wa = w_s[q];
      acc.x = fmaf(wa, a.x, acc.x); acc.y = fmaf(wa, a.y, acc.y);
      acc.z = fmaf(wa, a.z, acc.z); acc.w = fmaf(wa, a.w, acc.w);
    }
  }
  reinterpret_cast<float4*>(acc_s)[tid] = acc;  // float index slice * cols + col * 4
  wsum = warp_sum(wsum);
  if (lane == 0) red_s[warp] = wsum;
  __syncthreads();
  if (tid < cols) {
    float ws = 0.f;
    for (int i = 0; i < kReduceThreads / 32; ++i) ws += red_s[i];
    float v = 0.f;
    for (int i = 0; i < nslices; ++i) v += acc_s[i * cols + tid];
    reinterpret_cast<T*>(out_)[row * D + col0 + tid] = E::from_float(v / ws);
  }
}

}  // namespace pa
