// Paged decode attention on the 5th-generation tensor cores (tcgen05, bf16),
// persistent.
//
// The same operation as paged_decode_kernel (studying-code.tistory.com/16,
// section "PagedAttention: 운영체제의 페이징 개념에서 영감을 받은 새로운 어텐션
// 알고리즘": the query multiplies each block's keys, the scores weight each
// block's values, the per-block results combine into o_i), with the two
// contractions of a GQA group on the tensor cores:
//
//   S^T [128 tokens x 16]   = K_tile [128 x D] . Q^T [D x 16]        (QK)
//   O^T [D x 16]            = V_tile^T [D x 128] . P^T [128 x 16]     (PV)
//
// The 16 columns are the query heads of one KV head (G <= 16; rows past G
// are masked).  A work item is one (partition, KV head, sequence).  The grid
// is persistent: each CTA takes items from an atomic counter until they run
// out (or, in the balanced split, the pieces of its own ranges of stages),
// and its six warps stream every item's stages through one pipeline:
//   warp 0      producer: takes the next item, publishes it in a 4-entry ring,
//               loads the item's 16 query rows by TMA straight into the
//               swizzled B-operand layout, and streams the item's 128-token
//               K/V stages, one TMA box per block holding the block's K and V
//               rows of every column group (in the 128-byte swizzle the MMA
//               descriptors read), the boxes of a stage issued by all 32
//               lanes at once;
//   warp 1      tensor-memory allocator and MMA issuer (one thread), an event
//               loop that issues QK (up to two stages ahead) and PV (in order)
//               as soon as each one's inputs are ready;
//   warps 2..5  softmax warpgroup, one token (QK) or one head dimension (PV)
//               per tensor-memory lane: online softmax in fp32 (log2 domain),
//               P^T to shared memory as bf16; each stage's PV adds into one
//               fp32 O tile in tensor memory (rescaled there when the running
//               maximum moves), read once for the item's output (final rows,
//               or a split-KV partial) at its end.
// Stage ring slots, S and P double buffers and their barriers are indexed by a
// stage counter that runs across items, so the pipeline never drains between
// items.  Every wait is bounded; a timeout records PA_DEVERR_TIMEOUT, the CTA
// drains its MMAs and TMA loads, frees its tensor memory and returns.  The
// last CTA to finish resets the work counter, so it is zero for the next call.
#pragma once

#include "decode_kernel.cuh"
#include "pa_tcgen05.cuh"

namespace pa {

constexpr int kTcTokens = 128;   // tokens per stage = M of the QK MMA
constexpr int kTcHeads = 16;     // N of both MMAs: query heads, G padded
constexpr int kTcThreads = 192;  // producer, MMA, 4 softmax warps
constexpr int kTcTmemCols = 64;  // S x2, O x2, 16 columns each
constexpr int kTcItemRing = 4;
constexpr int kTcLensCache = 256;  // batches up to this size keep seq_lens in shared memory
constexpr int kTcTraceRoles = 6;   // timeline regions per CTA: one per warp
constexpr float kTcLazyMax = 8.f;  // a stage's scores may exceed the running maximum by this much

// Kinds of ring entries.
constexpr int kItemAttend = 0;  // attention over tokens [tok0, tok1)
constexpr int kItemZero = 1;    // a sequence of length 0: zero output rows
constexpr int kItemEnd = 2;     // no more work

struct TcItem {
  int s, h, part, tok0, tok1, nstages, final_out, kind;
};

// Shared-memory layout (byte offsets from a 1024-aligned base).
struct TcSmem {
  int region;    // K (or V) tile of one stage
  int stage;
  int q_off;     // two Q tiles
  int p_off;     // two P^T tiles
  int red_off;   // max / sum exchange of the softmax warpgroup
  int item_off;  // item ring
  int bar_off;
  int misc_off;
  int lens_off;  // cached sequence lengths (batches of up to kTcLensCache)
  int pre_off;   // work items before each sequence (dense numbering), kTcLensCache + 1
  int starts_off;  // cached first tokens of each sequence's own part (after a shared prefix)
  int total;     // bytes to request (includes 1024 of alignment slack)
};

// with_starts: room for the own-part start tokens of a launch after a
// shared-prefix decode (other launches leave it out: at head size 64 the
// extra kilobyte would cost the second resident CTA of an SM).
__host__ __device__ inline TcSmem tc_smem_layout(int head_size, int num_stages,
                                                 bool with_starts = false) {
  TcSmem l;
  const int groups = head_size / 64;
  l.region = groups * kTcTokens * 128;
  l.stage = 2 * l.region;
  l.q_off = num_stages * l.stage;
  l.p_off = l.q_off + 2 * groups * kTcHeads * 128;
  l.red_off = l.p_off + 2 * 2 * kTcHeads * 128;
  l.item_off = l.red_off + 3 * 4 * kTcHeads * 4;
  l.bar_off = l.item_off + kTcItemRing * (int)sizeof(TcItem);
  // full[NS], empty[NS], s full/free, p full, o full and q full/free [2
  // each], item full/free [ring], drain
  l.misc_off = l.bar_off + 8 * (2 * num_stages + 12 + 2 * kTcItemRing + 1);
  l.lens_off = l.misc_off + 64;
  l.pre_off = l.lens_off + kTcLensCache * 4;
  l.starts_off = l.pre_off + (kTcLensCache + 4) * 4;
  l.total = l.starts_off + (with_starts ? kTcLensCache * 4 : 0) + 1024;
  return l;
}

// True in one lane of the (fully active) warp.
__device__ __forceinline__ bool elect_one() {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "elect.sync _|p, 0xffffffff;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r));
  return r != 0;
}

// Has the phase with the given parity completed, as observed by every lane
// of the warp?  (Each lane's own test gives it the acquire.)
__device__ __forceinline__ bool warp_test(uint32_t bar, uint32_t parity) {
  return __all_sync(0xffffffffu, mbar_test(bar, parity));
}

// Named barrier of the softmax warpgroup that also ORs a predicate across it.
__device__ __forceinline__ bool softmax_group_any(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v)
      : "memory");
  return r != 0;
}

// Named barrier of the softmax warpgroup that also ANDs a predicate across it.
__device__ __forceinline__ bool softmax_group_all(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

__device__ __forceinline__ void st_shared_zero16(uint32_t addr) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0u) : "memory");
}

// 3-D tiled tensor load (the query map), completing on `bar`.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}

// Barrier addresses of the tensor-core decode (shared-memory byte addresses).
struct TcBars {
  uint32_t full0, empty0, s_full, s_free, p_full, o_full, q_full, q_free, it_full, it_free,
      drain;
  __device__ __forceinline__ TcBars(uint32_t base, int ns) {
    full0 = base;
    empty0 = base + 8u * ns;
    s_full = base + 16u * ns;
    s_free = s_full + 16;
    p_full = s_full + 32;
    o_full = s_full + 48;
    q_full = s_full + 64;
    q_free = s_full + 80;
    it_full = s_full + 96;
    it_free = it_full + 8u * kTcItemRing;
    drain = it_free + 8u * kTcItemRing;
  }
};

// One event of the optional timeline (see pa_set_decode_trace); compiled
// only into the kernels launched while a timeline is requested.
template <bool kTrace>
__device__ __forceinline__ void tc_trace(const DecodeParams& p, int role, int& n, uint32_t tag,
                                         uint32_t arg) {
  if constexpr (kTrace) {
    if (p.trace != nullptr && n < p.trace_per_role) {
      unsigned long long* e =
          p.trace + (((size_t)blockIdx.x * kTcTraceRoles + role) * (size_t)p.trace_per_role + n) * 2;
      e[0] = (unsigned long long)clock64();
      e[1] = ((unsigned long long)tag << 32) | arg;
    }
    ++n;
  }
}

// floor(a / b) for 0 <= a < 2^24 and b >= 1, from a float reciprocal of b:
// the product is within one of the quotient, and one step corrects it.
__device__ __forceinline__ int div_by_recip(int a, int b, float inv_b) {
  int q = __float2int_rz(__int2float_rn(a) * inv_b);
  const int r = a - q * b;
  if (r >= b) ++q;
  else if (r < 0) --q;
  return q;
}

__device__ __forceinline__ unsigned long long global_timer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// GP: the query group size G rounded up to a power of two (1..16); the
// softmax warpgroup handles GP heads (the MMAs always compute 16 columns).
// kBal: the balanced split (else fixed partitions, or none); kTrace: record
// the timeline.  Each is a separate kernel so that a launch carries only the
// code it runs.
template <int D, int GP, bool kBal, bool kTrace>
__global__ void __launch_bounds__(kTcThreads, 1)
    paged_decode_tc_kernel(const __grid_constant__ CUtensorMap kv_map,
                           const __grid_constant__ CUtensorMap q_map, const DecodeParams p) {
  static_assert(D == 64 || D == 128, "tensor-core decode handles head sizes 64 and 128");
  static_assert(GP >= 1 && GP <= kTcHeads && (GP & (GP - 1)) == 0, "padded group");
  constexpr int kGroups = D / 64;                 // 128-byte column groups of a row
  // A stage holds 16 chunks of 8 tokens; a chunk holds, per column group, the
  // group's 8 K rows (1024 bytes, one 128-byte swizzle atom) then its 8 V rows.
  constexpr int kChunkBytes = kGroups * 2048;
  constexpr int kQTile = kGroups * kTcHeads * 128;
  constexpr int kKSteps = D / 16;                 // QK: K = head dimension
  constexpr int kPvSteps = kTcTokens / 16;        // PV: K = tokens
  constexpr uint32_t kIdescQK = tc::idesc_bf16_f32(128, kTcHeads, 0);
  constexpr uint32_t kIdescPV = tc::idesc_bf16_f32(128, kTcHeads, 1);
  // PV's A operand (V^T) spans 128 rows = two 64-dimension groups; with one
  // group (D = 64) both halves read the same group and rows 64..127 repeat.
  constexpr uint32_t kPvLbo = kGroups > 1 ? 2048 : 0;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int G = p.group;
  const int NS = p.num_stages;
  const TcSmem lay = tc_smem_layout(D, NS, p.seq_start != nullptr);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(base);
  const uint32_t q_s = sbase + lay.q_off;
  const uint32_t p_s = sbase + lay.p_off;
  float* red = reinterpret_cast<float*>(base + lay.red_off);  // [3][4 warps][16 heads]
  volatile TcItem* ring = reinterpret_cast<volatile TcItem*>(base + lay.item_off);
  const TcBars bars(sbase + lay.bar_off, NS);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + lay.misc_off);
  volatile int* flags = reinterpret_cast<volatile int*>(base + lay.misc_off + 16);
  // flags[0] abort, flags[1] K/V stages issued, flags[2] Q tiles issued

  if (tid == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(bars.full0 + 8u * i, 1);
      mbar_init(bars.empty0 + 8u * i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bars.s_full + 8u * i, 1);
      mbar_init(bars.s_free + 8u * i, 128);
      mbar_init(bars.p_full + 8u * i, 128);
      mbar_init(bars.o_full + 8u * i, 1);
      mbar_init(bars.q_full + 8u * i, 1);
      mbar_init(bars.q_free + 8u * i, 1);
    }
    for (int i = 0; i < kTcItemRing; ++i) {
      mbar_init(bars.it_full + 8u * i, 1);
      mbar_init(bars.it_free + 8u * i, 2);  // the MMA thread and the softmax warpgroup
    }
    mbar_init(bars.drain, 1);
    flags[0] = 0;
    flags[1] = 0;
    flags[2] = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(smem_u32(tmem_slot), kTcTmemCols);
    tc::tmem_relinquish();
  }
  if (tid == 32) {
    tma_prefetch_desc(&kv_map);
    tma_prefetch_desc(&q_map);
  }
  // Both P^T tiles start at zero: the softmax writes only rows below GP.
  for (int i = tid; i < 2 * 2 * kTcHeads * 128 / 16; i += kTcThreads)
    st_shared_zero16(p_s + (uint32_t)i * 16u);
  // Everything above touches only this CTA's own resources and may overlap
  // the previous kernel; from here on global memory is read.  The next
  // kernel (the split-KV reduce) may start launching: this grid is resident
  // as a whole, so its CTAs only take room this grid does not use.
  grid_dependency_wait();
  grid_dependents_launch();
  // The first work item of CTA b is item b (later ones come from the work
  // counter); the producer loads its block-table window now, overlapping the
  // sequence-length loads below.
  int pf_win = -1, pf_s = -1, pf_cur = 0, pf_nxt = 0;
  if (!kBal && warp == 0 && !p.dense_items && (int)blockIdx.x < p.total_items) {
    const int sh = p.num_seqs * p.num_kv_heads;
    const int part = (int)blockIdx.x / sh;
    pf_s = ((int)blockIdx.x - part * sh) / p.num_kv_heads;
    pf_win = (p.partition_tokens > 0 ? part * p.partition_tokens : 0) >> p.log2_block_size;
    const int32_t* row = p.block_tables + (size_t)pf_s * p.max_blocks_per_seq;
    pf_cur = pf_win + lane < p.max_blocks_per_seq ? __ldg(row + pf_win + lane) : 0;
    pf_nxt = pf_win + 32 + lane < p.max_blocks_per_seq ? __ldg(row + pf_win + 32 + lane) : 0;
  }
  // Sequence lengths in shared memory, so classifying a work item needs no
  // global load.
  int* lens_s = p.num_seqs <= kTcLensCache ? reinterpret_cast<int*>(base + lay.lens_off) : nullptr;
  // After a shared-prefix decode, the first token of each sequence's own part.
  int* starts_s =
      (p.seq_start != nullptr && lens_s) ? reinterpret_cast<int*>(base + lay.starts_off) : nullptr;
  if (lens_s)
    for (int i = tid; i < p.num_seqs; i += kTcThreads) {
      lens_s[i] = p.seq_lens[i];
      if (starts_s) starts_s[i] = p.seq_start[i];
    }
  tc::fence_proxy_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS0 = tmem, tO0 = tmem + 32;

  if (warp == 0) {
    // ---------------- producer ----------------
    const int BS = p.block_size;
    const int l2bs = p.log2_block_size;
    const int R = p.box_rows;  // min(block_size, 128)
    const int log2R = p.log2_box_rows;
    // A box = one block's rows (at most 128) of K and V, every column group.
    const uint32_t box_bytes = (uint32_t)R * (uint32_t)kGroups * 256u;
    const int chunks_per_block = BS >> 3;
    const int sh = p.num_seqs * p.num_kv_heads;
    const int P = p.partition_tokens;
    int gk = 0, qi = 0, ii = 0, ntr = 0;
    if (lane == 0) tc_trace<kTrace>(p, 0, ntr, 9, kTrace ? (uint32_t)global_timer() : 0u);
    // Dense numbering (many partitions per sequence, batches of up to
    // kTcLensCache): sequence s owns items pre[s] .. pre[s+1]-1, its
    // partitions in order with the KV heads fastest, so no index is spent on
    // a partition past a sequence's end.  pre[] is a warp scan of the
    // per-sequence item counts.  Otherwise item = (partition, sequence, KV
    // head) over the whole grid, partitions past a sequence's end skipped.
    //
    // Balanced split: the stages of every (sequence, KV head) pair, laid end
    // to end (sequences in order, KV heads fastest), are cut into
    // p.total_items ranges of Q = ceil(stages / ranges) stages; CTA b takes
    // ranges b, b + grid, ...  A range covers the end of one pair and the
    // start of the next ones; each such piece is a work item.  pre[s] then
    // counts the stages before sequence s, the pieces of a pair are its
    // partials (numbered by range), and the CTA holding a pair's first piece
    // records the pair's piece count for the reduce.  Sequences without
    // stages (length 0, or a length error) are handled after the ranges,
    // sequence s by CTA s mod grid.
    int* pre = reinterpret_cast<int*>(base + lay.pre_off);
    unsigned int total = (unsigned)p.total_items;
    // The balanced split needs the lengths in shared memory (the host
    // launches it only for batches that fit); without them nothing is done.
    constexpr bool bal = kBal;
    if (kBal && lens_s == nullptr && blockIdx.x == 0 && lane == 0)
      record_error(p.err, PA_DEVERR_SEQ_LEN);
    const bool dense = (p.dense_items || bal) && lens_s != nullptr;
    if (dense) {
      int carry = 0;
      if (lane == 0) pre[0] = 0;
      for (int c0 = 0; c0 < p.num_seqs; c0 += 32) {
        const int sq = c0 + lane;
        int n = 0;
        if (sq < p.num_seqs) {
          const int L = lens_s[sq];
          const int np = L <= 0 ? 1 : (P > 0 ? (L + P - 1) / P : 1);
          if (L > 0 && ((!bal && P > 0 && np > p.max_parts) ||
                        ((L + BS - 1) >> l2bs) > p.max_blocks_per_seq)) {
            if (blockIdx.x == 0) record_error(p.err, PA_DEVERR_SEQ_LEN);
          } else if (bal) {
            // Members of a shared-prefix group (start > 0) are the group
            // kernel's: no stages here.
            const bool member = starts_s && starts_s[sq] > 0;
            n = (L <= 0 || member) ? 0 : ((L + kTcTokens - 1) / kTcTokens) * p.num_kv_heads;
          } else {
            n = np * p.num_kv_heads;
          }
        }
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int v = __shfl_up_sync(0xffffffffu, n, o);
          if (lane >= o) n += v;
        }
        if (sq < p.num_seqs) pre[sq + 1] = carry + n;
        carry += __shfl_sync(0xffffffffu, n, 31);
      }
      __syncwarp();
      total = (unsigned)carry;
    }
    unsigned int idx = blockIdx.x;
    // Balanced split cursor (every lane holds the same): stages [bg, bg_end)
    // of range brange, then sequence zs (KV head zh) of the zero-stage pass.
    // Stage counts stay below 2^24 there (the reciprocal divisions need it;
    // beyond, no work is done and the length error is recorded).
    const int ranges = p.total_items;
    const int bq = bal ? max(1, (int)((total + (unsigned)ranges - 1) / (unsigned)ranges)) : 1;
    const float inv_bq = 1.f / (float)bq;
    // Past that, every pair goes through the zero-stage pass below, which
    // records a piece count of 0 for it: the reduce then leaves its rows
    // alone instead of combining whatever partials an earlier call left.
    const bool overflow = kBal && total >= (1u << 24);
    if (overflow) {
      if (blockIdx.x == 0 && lane == 0) record_error(p.err, PA_DEVERR_SEQ_LEN);
      total = 0;
    }
    int brange = (int)blockIdx.x, bg = 0, bg_end = 0, zs = (int)blockIdx.x, zh = 0;
    if (bal && brange < ranges) {
      bg = brange * bq;
      bg_end = min((int)total, bg + bq);
    }
    // An item's last stage is held back (its boxes resolved, one per lane)
    // and issued only once the next item is classified, published and its
    // query load issued: that work then overlaps the wait for the last
    // stage's slot instead of leaving freed slots idle after it.
    bool def_have = false, def_fence = false, def_live = false;
    int def_gk = 0, def_nbox = 0, def_c4 = 0, def_h = 0;
    auto issue_deferred = [&]() -> bool {
      if (!def_have) return true;
      def_have = false;
      const int slot = def_gk % NS;
      bool w = true;
      if (def_gk >= NS) {
        if (lane == 0)
          w = mbar_wait_bounded(bars.empty0 + 8u * slot, ((def_gk / NS) - 1) & 1, p.err,
                                p.wait_limit);
        w = __shfl_sync(0xffffffffu, w, 0);
        if (!w) return false;
      }
      if (def_fence) {
        fence_proxy_async_global();
        __syncwarp();
        fence_proxy_async_global();
      }
      if (lane == 0) {
        mbar_arrive_expect_tx(bars.full0 + 8u * slot, (uint32_t)def_nbox * box_bytes);
        tc_trace<kTrace>(p, 0, ntr, 20, (uint32_t)def_gk);
      }
      __syncwarp();
      if (def_live)
        tma_load_5d(sbase + (uint32_t)slot * (uint32_t)lay.stage + (uint32_t)lane * box_bytes,
                    &kv_map, bars.full0 + 8u * slot, 0, 0, 0, def_h * kGroups, def_c4);
      if (lane == 0) {
        flags[1] = def_gk + 1;
        tc_trace<kTrace>(p, 0, ntr, 2, (uint32_t)def_gk);
      }
      return true;
    };
    while (true) {
      if (flags[0]) break;
      // Lane 0 classifies the item; the warp follows its decision.
      TcItem it{0, 0, 0, 0, 0, 0, 0, kItemEnd};
      bool skip = false;
      int wnew = 0;  // this item holds the sequence's newest token and writes it (fused write)
      if (kBal && lens_s != nullptr) {
        // Warp-uniform: every lane computes the same item, lane 0 writes.
        if (bg < bg_end) {
          // The sequence whose stages contain bg: the last s with
          // pre[s] <= bg (pre is non-decreasing, so count the s that qualify).
          int lo = -1;
          for (int c0 = 0; c0 < p.num_seqs; c0 += 32)
            lo += __popc(__ballot_sync(0xffffffffu, c0 + lane < p.num_seqs && pre[c0 + lane] <= bg));
          const int L = lens_s[lo];
          const int n = (L + kTcTokens - 1) / kTcTokens;  // stages of each of its pairs
          const int off = bg - pre[lo];
          const int h = div_by_recip(off, n, 1.f / (float)n);
          const int k0 = off - h * n;
          const int len = min(n - k0, bg_end - bg);
          const int pair0 = pre[lo] + h * n;  // the pair's first stage
          const int first = div_by_recip(pair0, bq, inv_bq);
          const int npieces = div_by_recip(pair0 + n - 1, bq, inv_bq) - first + 1;
          it.s = lo;
          it.h = h;
          it.part = div_by_recip(bg, bq, inv_bq) - first;
          it.tok0 = k0 * kTcTokens;
          it.tok1 = min(L, (k0 + len) * kTcTokens);
          it.nstages = len;
          it.final_out = npieces == 1;
          it.kind = kItemAttend;
          if (it.part == 0 && lane == 0) {
            p.part_counts[lo * p.num_kv_heads + h] = npieces <= p.max_parts ? npieces : 0;
            if (npieces > p.max_parts) record_error(p.err, PA_DEVERR_SEQ_LEN);
          }
          skip = npieces > p.max_parts;
          wnew = p.new_k != nullptr && it.tok1 == L;
          bg += len;
          if (bg >= bg_end) {
            brange += (int)gridDim.x;
            if (brange < ranges) {
              bg = brange * bq;
              bg_end = min((int)total, bg + bq);
            }
          }
        } else if (zs < p.num_seqs) {
          if (starts_s && starts_s[zs] > 0 && lens_s[zs] > 0 && !overflow) {
            // A shared-prefix group member: the group kernel's rows and counts.
            skip = true;
            zs += (int)gridDim.x;
          } else if (pre[zs + 1] == pre[zs] || overflow) {
            // No stages: zero rows for length 0 (a length error leaves its
            // rows undefined); no partials either way.
            if (lane == 0) p.part_counts[zs * p.num_kv_heads + zh] = 0;
            it.s = zs;
            it.h = zh;
            it.kind = kItemZero;
            skip = lens_s[zs] > 0;
            if (++zh == p.num_kv_heads) {
              zh = 0;
              zs += (int)gridDim.x;
            }
          } else {
            skip = true;
            zs += (int)gridDim.x;
          }
        }
      } else if (!kBal && lane == 0 && dense && idx < total) {
        // The sequence whose items contain idx: the last s with pre[s] <= idx.
        int lo = 0, hi = p.num_seqs - 1;
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (pre[mid] <= (int)idx) lo = mid; else hi = mid - 1;
        }
        const int r = (int)idx - pre[lo];
        it.s = lo;
        it.part = r / p.num_kv_heads;
        it.h = r - it.part * p.num_kv_heads;
        const int L = lens_s[lo];
        if (L <= 0) {
          it.kind = kItemZero;
        } else {
          const int nparts = P > 0 ? (L + P - 1) / P : 1;
          it.kind = kItemAttend;
          it.tok0 = P > 0 ? it.part * P : 0;
          it.tok1 = P > 0 ? min(L, it.tok0 + P) : L;
          it.nstages = (it.tok1 - it.tok0 + kTcTokens - 1) / kTcTokens;
          it.final_out = nparts == 1;
          wnew = p.new_k != nullptr && it.tok1 == L;
        }
      } else if (!kBal && lane == 0 && !dense && idx < total) {
        it.part = (int)(idx / (unsigned)sh);
        const int rem = (int)(idx % (unsigned)sh);
        it.s = rem / p.num_kv_heads;
        it.h = rem - it.s * p.num_kv_heads;
        const int L = lens_s ? lens_s[it.s] : p.seq_lens[it.s];
        const int nparts = L <= 0 ? 0 : (P > 0 ? (L + P - 1) / P : 1);
        if (L <= 0) {
          it.kind = kItemZero;
          skip = it.part != 0;
        } else if ((P > 0 && nparts > p.max_parts) ||
                   ((L + BS - 1) >> l2bs) > p.max_blocks_per_seq) {
          if (it.part == 0 && it.h == 0) record_error(p.err, PA_DEVERR_SEQ_LEN);
          skip = true;
        } else if (it.part >= nparts) {
          skip = true;
        } else {
          it.kind = kItemAttend;
          it.tok0 = P > 0 ? it.part * P : 0;
          it.tok1 = P > 0 ? min(L, it.tok0 + P) : L;
          it.nstages = (it.tok1 - it.tok0 + kTcTokens - 1) / kTcTokens;
          it.final_out = nparts == 1;
          wnew = p.new_k != nullptr && it.tok1 == L;
        }
        if (p.seq_start != nullptr && it.part == 0) {
          // Next to a shared-prefix decode: members of a group (start > 0)
          // are the group kernel's; the others' rows are final here.
          const int st = starts_s ? starts_s[it.s] : __ldg(p.seq_start + it.s);
          if (st > 0 && L > 0) skip = true;
          else p.part_counts[it.s * p.num_kv_heads + it.h] = 0;
        }
      }
      if (lane == 0) tc_trace<kTrace>(p, 0, ntr, 10, bal ? (uint32_t)bg : idx);
      if constexpr (!kBal) {
        wnew = __shfl_sync(0xffffffffu, wnew, 0);
        skip = __shfl_sync(0xffffffffu, skip, 0);
      }
      if (skip) {
        if (!kBal && lane == 0) idx = gridDim.x + atomicAdd(p.sched, 1u);
        continue;
      }
      if constexpr (!kBal) {
        it.s = __shfl_sync(0xffffffffu, it.s, 0);
        it.h = __shfl_sync(0xffffffffu, it.h, 0);
        it.part = __shfl_sync(0xffffffffu, it.part, 0);
        it.tok0 = __shfl_sync(0xffffffffu, it.tok0, 0);
        it.tok1 = __shfl_sync(0xffffffffu, it.tok1, 0);
        it.nstages = __shfl_sync(0xffffffffu, it.nstages, 0);
        it.final_out = __shfl_sync(0xffffffffu, it.final_out, 0);
        it.kind = __shfl_sync(0xffffffffu, it.kind, 0);
      }
      // The item's block-table window, loaded now so that its latency
      // overlaps the item's publication and query load: [win, win+32) in
      // `cur`, [win+32, win+64) in `nxt` (a stage spans at most 16 blocks).
      const int32_t* table = p.block_tables + (size_t)it.s * p.max_blocks_per_seq;
      const int lb_end = (it.tok1 + BS - 1) >> l2bs;
      int win = it.tok0 >> l2bs;
      int cur, nxt;
      if (win == pf_win && it.s == pf_s) {  // the first item's window, loaded early
        cur = pf_cur;
        nxt = pf_nxt;
      } else {
        cur = (win + lane < lb_end) ? __ldg(table + win + lane) : 0;
        nxt = (win + 32 + lane < lb_end) ? __ldg(table + win + 32 + lane) : 0;
      }
      pf_win = -1;
      // Publish it in the ring.
      const int j = ii % kTcItemRing;
      bool ok = true;
      if (lane == 0) {
        if (ii >= kTcItemRing)
          ok = mbar_wait_bounded(bars.it_free + 8u * j, ((ii / kTcItemRing) - 1) & 1, p.err,
                                 p.wait_limit);
        if (ok) {
          ring[j].s = it.s;
          ring[j].h = it.h;
          ring[j].part = it.part;
          ring[j].tok0 = it.tok0;
          ring[j].tok1 = it.tok1;
          ring[j].nstages = it.nstages;
          ring[j].final_out = it.final_out;
          ring[j].kind = it.kind;
          mbar_arrive(bars.it_full + 8u * j);
          tc_trace<kTrace>(p, 0, ntr, 1, (uint32_t)ii);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) {
        flags[0] = 1;
        break;
      }
      ++ii;
      if (it.kind == kItemEnd) {
        if (!issue_deferred()) {
          flags[0] = 1;
          break;
        }
        if (lane == 0) tc_trace<kTrace>(p, 0, ntr, 8, (uint32_t)ii);
        break;
      }
      if (it.kind != kItemAttend) {
        if (!kBal && lane == 0) idx = gridDim.x + atomicAdd(p.sched, 1u);  // the next item
        if (!issue_deferred()) {
          flags[0] = 1;
          break;
        }
        continue;
      }
      // The fused write's rows and target block, loaded now so that their
      // latency overlaps the query load and the first stage's issue; stored
      // before the item's second stage (or its only one) is issued, fenced
      // before its last.
      uint4 new_kv = make_uint4(0u, 0u, 0u, 0u);
      int new_id = 0, k_store = -1, k_fence = -1;
      if (wnew) {
        new_kv = load_new_token(p.new_k, p.new_v, it.s, it.h, p.num_kv_heads, D * 2 / 16, lane);
        new_id = __ldg(table + lb_end - 1);
        k_store = min(1, it.nstages - 1);
        k_fence = it.nstages - 1;
      }

      // Query rows h*G .. h*G+15 of sequence s (rows past G are masked).
      const int qb = qi & 1;
      if (lane == 0) {
        if (qi >= 2)
          ok = mbar_wait_bounded(bars.q_free + 8u * qb, ((qi >> 1) - 1) & 1, p.err, p.wait_limit);
        if (ok) {
          mbar_arrive_expect_tx(bars.q_full + 8u * qb, (uint32_t)kQTile);
          const int row0 = it.s * p.num_heads + it.h * G;
#pragma unroll
          for (int g = 0; g < kGroups; ++g)
            tma_load_3d(q_s + (uint32_t)(qb * kQTile + g * kTcHeads * 128), &q_map,
                        bars.q_full + 8u * qb, 0, g, row0);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) {
        flags[0] = 1;
        break;
      }
      ++qi;
      if (lane == 0) {
        flags[2] = qi;
        tc_trace<kTrace>(p, 0, ntr, 11, (uint32_t)qi);
      }
      if (!issue_deferred()) {
        flags[0] = 1;
        break;
      }

      // The item's K/V stages.  Every lane issues TMA boxes (a box = one
      // block's rows of one 128-byte column group of K or of V): one thread
      // issuing them in sequence cannot keep HBM busy.
      if (lane == 0) tc_trace<kTrace>(p, 0, ntr, 12, (uint32_t)(cur + nxt));
      for (int k = 0; k < it.nstages; ++k, ++gk) {
        const int slot = gk % NS;
        const int st_tok = it.tok0 + k * kTcTokens;
        const int st_n = min(kTcTokens, it.tok1 - st_tok);
        const int nbox = (st_n + R - 1) >> log2R;
        const int lb0 = st_tok >> l2bs;
        // The last stage is held back for the next item's set-up.  Under the
        // balanced split (pieces of one or two stages are common) only when
        // its slot is still busy, so that the set-up fills that wait; with
        // fixed partitions (items of several stages) always.
        bool defer = k == it.nstages - 1 && nbox <= 32 && gk >= NS;
        if (kBal && defer) {
          bool busy = false;
          if (lane == 0) busy = !mbar_test(bars.empty0 + 8u * slot, ((gk / NS) - 1) & 1);
          defer = __shfl_sync(0xffffffffu, busy, 0);
        }
        if (gk >= NS && !defer) {
          if (lane == 0)
            ok = mbar_wait_bounded(bars.empty0 + 8u * slot, ((gk / NS) - 1) & 1, p.err,
                                   p.wait_limit);
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) break;
        }
        while (lb0 >= win + 32) {
          cur = nxt;
          win += 32;
          nxt = (win + 32 + lane < lb_end) ? __ldg(table + win + 32 + lane) : 0;
        }
        if (k == k_store)
          store_new_token(p.cache_w, new_kv, new_id, it.h, it.tok1 - 1, p.num_kv_heads, D * 2 / 16,
                          BS, p.num_blocks, p.err, lane);
        if (defer) {
          // Resolve the last stage's boxes now (this item's table window is
          // replaced by the next item's) and issue them later.
          const bool live = lane < nbox;
          const int tk = st_tok + ((live ? lane : 0) << log2R);
          const int src = (tk >> l2bs) - win;  // 0 .. 47
          const int id_cur = __shfl_sync(0xffffffffu, cur, src & 31);
          const int id_nxt = __shfl_sync(0xffffffffu, nxt, src & 31);
          const int id = src < 32 ? id_cur : id_nxt;
          int c4 = id * chunks_per_block + ((tk & (BS - 1)) >> 3);
          if (live && (id < 0 || id >= p.num_blocks)) {
            record_error(p.err, PA_DEVERR_BLOCK_ID);
            c4 = p.num_blocks * chunks_per_block;  // outside the tensor: zero fill
          }
          def_have = true;
          def_live = live;
          def_c4 = c4;
          def_gk = gk;
          def_nbox = nbox;
          def_h = it.h;
          def_fence = k == k_fence;
          if (!kBal && k == 0 && lane == 0) idx = gridDim.x + atomicAdd(p.sched, 1u);
          continue;
        }
        if (k == k_fence) {
          // The newest token lands in this stage: its store is ordered before
          // the stage's TMA reads.
          fence_proxy_async_global();
          __syncwarp();
          fence_proxy_async_global();
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(bars.full0 + 8u * slot, (uint32_t)nbox * box_bytes);
          tc_trace<kTrace>(p, 0, ntr, 20, (uint32_t)gk);
        }
        __syncwarp();
        const uint32_t kdst = sbase + (uint32_t)slot * (uint32_t)lay.stage;
        for (int b0 = 0; b0 < nbox; b0 += 32) {
          const int i = b0 + lane;
          const bool live = i < nbox;
          const int tk = st_tok + ((live ? i : 0) << log2R);
          const int src = (tk >> l2bs) - win;  // 0 .. 47
          const int id_cur = __shfl_sync(0xffffffffu, cur, src & 31);
          const int id_nxt = __shfl_sync(0xffffffffu, nxt, src & 31);
          if (live) {
            const int id = src < 32 ? id_cur : id_nxt;
            // 8-token chunk of the plane: block * (BS / 8) + chunk within the block.
            int c4 = id * chunks_per_block + ((tk & (BS - 1)) >> 3);
            if (id < 0 || id >= p.num_blocks) {
              record_error(p.err, PA_DEVERR_BLOCK_ID);
              c4 = p.num_blocks * chunks_per_block;  // outside the tensor: zero fill
            }
            tma_load_5d(kdst + (uint32_t)i * box_bytes, &kv_map, bars.full0 + 8u * slot, 0, 0, 0,
                        it.h * kGroups, c4);
          }
        }
        if (lane == 0) {
          flags[1] = gk + 1;
          tc_trace<kTrace>(p, 0, ntr, 2, (uint32_t)gk);
          // The next item's index, fetched once this item's first stage is
          // on its way (its round trip then overlaps the stages, not the
          // query load).
          if (!kBal && k == 0) idx = gridDim.x + atomicAdd(p.sched, 1u);
        }
      }
      if (!ok) {
        flags[0] = 1;
        break;
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    // An event loop: QK of the next stage and PV of the oldest stage are
    // issued as soon as their inputs are ready, independently, so a PV never
    // waits for an unrelated TMA load (PV releases the stage slot the loads
    // refill).  QK runs at most two stages ahead (S is double-buffered).
    // The whole warp runs the loop with warp-uniform state (a barrier counts
    // as complete once every lane has observed it, which also gives every
    // lane its acquire), so the MMA operands are warp-uniform values; one
    // elected lane issues the MMAs, commits and arrivals.
    const bool leader = elect_one();
    int next_qk = 0, next_pv = 0;  // global stage counters
    int ii = 0, qi = 0, qb = 0, qk_k = 0, qk_n = 0;
    // Bit gk % 4: stage gk is its item's first (its P.V starts the item's O
    // accumulator instead of adding to it).  QK runs at most two ahead of PV.
    uint32_t first_bits = 0;
    bool have_item = false, need_q = false, end_seen = false, ok = true;
    int ntr = 0;
    long long t_idle = clock64();
    while (true) {
      bool progress = false;
      if (!have_item && !end_seen) {
        const int j = ii % kTcItemRing;
        if (warp_test(bars.it_full + 8u * j, (ii / kTcItemRing) & 1)) {
          const int kind = ring[j].kind;
          const int n = ring[j].nstages;
          __syncwarp();
          if (leader) {
            mbar_arrive(bars.it_free + 8u * j);
            tc_trace<kTrace>(p, 1, ntr, 13, (uint32_t)ii);
          }
          ++ii;
          progress = true;
          if (kind == kItemEnd) {
            end_seen = true;
          } else if (kind == kItemAttend) {
            have_item = true;
            need_q = true;
            qk_k = 0;
            qk_n = n;
            qb = qi & 1;
          }
        }
      }
      if (have_item && need_q && warp_test(bars.q_full + 8u * qb, (qi >> 1) & 1)) {
        need_q = false;
        progress = true;
      }
      if (next_pv < next_qk) {
        const int gk = next_pv;
        const int slot = gk % NS;
        const int sb = gk & 1;
        if (warp_test(bars.p_full + 8u * sb, (gk >> 1) & 1)) {
          tc::fence_after_sync();
          // A: the stage's V rows read MN-major (V^T), 64-dimension groups
          // kPvLbo apart, 8-token groups kChunkBytes apart; B: P^T.
          const uint64_t a0 = tc::smem_desc_sw128(
              sbase + (uint32_t)slot * (uint32_t)lay.stage + 1024u, kPvLbo, kChunkBytes);
          const uint64_t b0 = tc::smem_desc_sw128(p_s + (uint32_t)sb * 2u * kTcHeads * 128u, 16,
                                                  1024);
          if (leader) {
            tc_trace<kTrace>(p, 1, ntr, 17, (uint32_t)gk);
#pragma unroll
            for (int kk = 0; kk < kPvSteps; ++kk) {
              const uint32_t aoff = (uint32_t)(kk * 2 * kChunkBytes);
              const uint32_t boff = (uint32_t)((kk >> 2) * kTcHeads * 128 + (kk & 3) * 32);
              tc::mma_bf16(tO0, a0 + (aoff >> 4), b0 + (boff >> 4), kIdescPV,
                           kk > 0 || !((first_bits >> (gk & 3)) & 1u));
            }
            tc::mma_commit(bars.o_full + 8u * sb);
            tc::mma_commit(bars.empty0 + 8u * slot);
            tc_trace<kTrace>(p, 1, ntr, 4, (uint32_t)gk);
          }
          __syncwarp();
          ++next_pv;
          progress = true;
        }
      }
      if (have_item && !need_q && next_qk < next_pv + 2) {
        const int gk = next_qk;
        const int slot = gk % NS;
        const int sb = gk & 1;
        if (warp_test(bars.full0 + 8u * slot, (gk / NS) & 1) &&
            (gk < 2 || warp_test(bars.s_free + 8u * sb, ((gk >> 1) - 1) & 1))) {
          tc::fence_after_sync();
          // A: the stage's K rows, K-major, 8-row groups kChunkBytes apart;
          // B: the item's Q tile.  Descriptors advance by address / 16.
          const uint64_t a0 = tc::smem_desc_sw128(sbase + (uint32_t)slot * (uint32_t)lay.stage,
                                                  16, kChunkBytes);
          const uint64_t b0 = tc::smem_desc_sw128(q_s + (uint32_t)(qb * kQTile), 16, 1024);
          const bool last = qk_k + 1 == qk_n;
          first_bits = (first_bits & ~(1u << (gk & 3))) | ((uint32_t)(qk_k == 0) << (gk & 3));
          if (leader) {
#pragma unroll
            for (int kk = 0; kk < kKSteps; ++kk) {
              const uint32_t aoff = (uint32_t)((kk >> 2) * 2048 + (kk & 3) * 32);
              const uint32_t boff = (uint32_t)((kk >> 2) * kTcHeads * 128 + (kk & 3) * 32);
              tc::mma_bf16(tS0 + 16u * sb, a0 + (aoff >> 4), b0 + (boff >> 4), kIdescQK, kk > 0);
            }
            tc::mma_commit(bars.s_full + 8u * sb);
            if (last) tc::mma_commit(bars.q_free + 8u * qb);  // the item's Q tile is no longer read
            tc_trace<kTrace>(p, 1, ntr, 3, (uint32_t)gk);
          }
          __syncwarp();
          ++next_qk;
          if (++qk_k == qk_n) {
            ++qi;
            have_item = false;
          }
          progress = true;
        }
      }
      if (end_seen && !have_item && next_pv == next_qk) break;
      const bool abort = __any_sync(0xffffffffu, flags[0] != 0);
      if (progress) {
        t_idle = clock64();
      } else if (!abort) {
        // Nothing ready: suspend briefly (128 ns at most) on the barrier most
        // likely to unblock this loop (the oldest pending PV's P tile, else
        // the next QK's stage); it wakes early when that barrier completes,
        // and leaves issue slots to the softmax warp sharing its scheduler.
        if (next_pv < next_qk)
          mbar_suspend(bars.p_full + 8u * (next_pv & 1), (next_pv >> 1) & 1, 128);
        else if (have_item && !need_q)
          mbar_suspend(bars.full0 + 8u * (next_qk % NS), (next_qk / NS) & 1, 128);
        else if (have_item)
          mbar_suspend(bars.q_full + 8u * qb, (qi >> 1) & 1, 128);
        else if (!end_seen)
          mbar_suspend(bars.it_full + 8u * (ii % kTcItemRing), (ii / kTcItemRing) & 1, 128);
      }
      if (progress) {
      } else if (abort) {
        ok = false;
        break;
      } else if (__any_sync(0xffffffffu, clock64() - t_idle > p.wait_limit)) {
        if (leader) record_error(p.err, PA_DEVERR_TIMEOUT);
        ok = false;
        break;
      }
    }
    if (!ok && leader) flags[0] = 1;
    // Every MMA the leader issued completes before the CTA may free its
    // tensor memory (this wait and the TMA drains below keep the full limit,
    // whatever limit the pipeline waits had).
    if (leader) {
      tc::mma_commit(bars.drain);
      mbar_wait_bounded(bars.drain, 0, p.err);
    }
    __syncwarp();
  } else {
    // ---------------- softmax warpgroup ----------------
    const int q4 = warp & 3;                  // tensor-memory lane quarter
    const int row = q4 * 32 + lane;           // token (QK) / head dimension (PV)
    const uint32_t lane_addr = (uint32_t)(q4 * 32) << 16;
    const uint32_t tO_lane = tO0 + lane_addr;
    float* red2 = red + 2 * 4 * kTcHeads;
    int gk = 0, ntr = 0;
    bool ok = true;
    for (int ii = 0;; ++ii) {
      const int j = ii % kTcItemRing;
      const bool w =
          mbar_wait_bounded(bars.it_full + 8u * j, (ii / kTcItemRing) & 1, p.err, p.wait_limit);
      TcItem it;
      it.s = ring[j].s;
      it.h = ring[j].h;
      it.part = ring[j].part;
      it.tok0 = ring[j].tok0;
      it.tok1 = ring[j].tok1;
      it.nstages = ring[j].nstages;
      it.final_out = ring[j].final_out;
      it.kind = ring[j].kind;
      if (lane == 0) tc_trace<kTrace>(p, warp, ntr, 21, (uint32_t)((warp << 16) | ii));
      ok = softmax_group_all(w && ok && !flags[0]);  // every thread has read the entry
      if (!ok) break;
      if (tid == 64) {
        mbar_arrive(bars.it_free + 8u * j);
        tc_trace<kTrace>(p, 2, ntr, 14, (uint32_t)ii);
      }
      if (it.kind == kItemEnd) break;
      const size_t row0 = (size_t)it.s * p.num_heads + (size_t)it.h * G;
      if (it.kind == kItemZero) {
        if (row < D)
          for (int g = 0; g < G; ++g)
            reinterpret_cast<__nv_bfloat16*>(p.out)[(row0 + g) * D + row] = __float2bfloat16_rn(0.f);
        continue;
      }

      float m_run[GP], l_run[GP], o_acc[GP];
#pragma unroll
      for (int g = 0; g < GP; ++g) {
        m_run[g] = -INFINITY;
        l_run[g] = 0.f;
      }
      const int n = it.nstages;
      for (int k = 0; k < n; ++k) {
        const int g_k = gk + k;
        const int sb = g_k & 1;
        const int slot = g_k % NS;
        const bool ws = mbar_wait_bounded(bars.s_full + 8u * sb, (g_k >> 1) & 1, p.err,
                                          p.wait_limit);
        if (tid == 64) tc_trace<kTrace>(p, 2, ntr, 15, (uint32_t)g_k);
        __syncwarp();
        tc::fence_after_sync();
        float sc[GP];
        tc::tmem_ld<GP>(tS0 + 16u * sb + lane_addr, sc);
        tc::tmem_wait_ld();
        tc::fence_before_sync();
        mbar_arrive(bars.s_free + 8u * sb);
        if (tid == 64) tc_trace<kTrace>(p, 2, ntr, 5, (uint32_t)g_k);

        const int nvalid = min(kTcTokens, it.tok1 - (it.tok0 + k * kTcTokens));
        const bool valid = row < nvalid;
        if (nvalid < kTcTokens) {
          // Stale rows of V (past the sequence, or never loaded) must not
          // reach the PV product: 0 * NaN would.  The rows of the ragged
          // 8-token chunk are cleared one per thread; the whole chunks after
          // it by the warpgroup in consecutive 16-byte pieces (a row per
          // thread would put eight threads on the same banks).
          const uint32_t vst = sbase + (uint32_t)slot * (uint32_t)lay.stage + 1024u;
          const int clear0 = (nvalid + 7) >> 3;  // the first chunk with no valid row
          if (!valid && row < clear0 * 8) {
            const uint32_t vrow = vst + (uint32_t)((row >> 3) * kChunkBytes + (row & 7) * 128);
#pragma unroll
            for (int g = 0; g < kGroups; ++g)
#pragma unroll
              for (int c = 0; c < 8; ++c)
                st_shared_zero16(vrow + (uint32_t)(g * 2048 + c * 16));
          }
          const int pieces = (kTcTokens / 8 - clear0) * kGroups * 64;
          for (int i = row; i < pieces; i += 128) {
            const int ch = clear0 + i / (kGroups * 64);
            const int rem = i % (kGroups * 64);
            st_shared_zero16(vst + (uint32_t)(ch * kChunkBytes + (rem >> 6) * 2048 + (rem & 63) * 16));
          }
        }
        float x[GP];
#pragma unroll
        for (int g = 0; g < GP; ++g)
          x[g] = (valid && g < G) ? sc[g] * p.scale_log2 : -INFINITY;
        // Lazy reference maximum: m_run[g] only has to bound this stage's
        // scores to within kTcLazyMax (log2 units), so the weights 2^(x - m)
        // stay at most 2^kTcLazyMax, exact in bf16 and fp32 sums.  Only when
        // some score in the warpgroup exceeds it (always on an item's first
        // stage) is the maximum exchanged and the running sums rescaled;
        // otherwise the stage costs one barrier.  A failed wait anywhere also
        // takes the exchange path, whose AND-barrier makes every thread agree.
        bool need = !(ws && ok) || flags[0];
#pragma unroll
        for (int g = 0; g < GP; ++g) need |= x[g] > m_run[g] + kTcLazyMax;
        float alpha[GP], pr[GP];
#pragma unroll
        for (int g = 0; g < GP; ++g) alpha[g] = 1.f;
        const bool need_any = softmax_group_any(need);
        if (tid == 64) tc_trace<kTrace>(p, 2, ntr, 24, (uint32_t)g_k);
        if (need_any) {
          float* redk = red + sb * 4 * kTcHeads;
#pragma unroll
          for (int g = 0; g < GP; ++g) {
            const float wm = warp_max_redux(x[g]);
            if (lane == 0) redk[q4 * kTcHeads + g] = wm;
          }
          if (!(ok = softmax_group_all(ws && ok && !flags[0]))) break;
#pragma unroll
          for (int g = 0; g < GP; ++g) {
            // Heads g >= G are padding: their scores are all -inf, the
            // maximum stays -inf, and they are given weight 0 and factor 1.
            const float tmax = fmaxf(fmaxf(redk[g], redk[kTcHeads + g]),
                                     fmaxf(redk[2 * kTcHeads + g], redk[3 * kTcHeads + g]));
            const float m_new = fmaxf(m_run[g], tmax);
            if (g < G) alpha[g] = fast_exp2(m_run[g] - m_new);
            m_run[g] = m_new;
          }
          if (k >= 1) {
            // O (in tensor memory, the sum of this item's P.V tiles so far)
            // is rescaled to the new maximum once the previous stage's P.V
            // has landed, before this stage's P releases the next P.V.
            const int gp = g_k - 1;
            const bool wo = mbar_wait_bounded(bars.o_full + 8u * (gp & 1), (gp >> 1) & 1, p.err,
                                              p.wait_limit);
            __syncwarp();
            tc::fence_after_sync();
            float ot[GP];
            tc::tmem_ld<GP>(tO_lane, ot);
            tc::tmem_wait_ld();
#pragma unroll
            for (int g = 0; g < GP; ++g) ot[g] *= alpha[g];
            tc::tmem_st<GP>(tO_lane, ot);
            tc::tmem_wait_st();
            tc::fence_before_sync();
            ok = wo && ok;
          }
        }
        // The weight enters P.V rounded to bf16; the denominator sums the
        // same rounded weights, so the output stays a convex combination.
        // Two heads' weights are rounded and packed by one conversion.
        uint32_t pw[(GP + 1) / 2];
#pragma unroll
        for (int i = 0; i < (GP + 1) / 2; ++i) {
          const int g0 = 2 * i, g1 = 2 * i + 1 < GP ? 2 * i + 1 : 2 * i;
          const float e0 = g0 < G ? fast_exp2(x[g0] - m_run[g0]) : 0.f;
          const float e1 = (2 * i + 1 < GP && g1 < G) ? fast_exp2(x[g1] - m_run[g1]) : 0.f;
          pw[i] = pack_bf16x2(e0, e1);
        }
#pragma unroll
        for (int g = 0; g < GP; ++g) {
          pr[g] = (g & 1) ? bf16_hi(pw[g >> 1]) : bf16_lo(pw[g >> 1]);
          l_run[g] = fmaf(l_run[g], alpha[g], pr[g]);
        }
        // P^T as the PV's B operand: [64-token group][16 rows][128 bytes], swizzled.
        {
          const uint32_t pb = p_s + (uint32_t)sb * 2u * kTcHeads * 128u +
                              (uint32_t)((row >> 6) * kTcHeads * 128);
          const int col = row & 63;
#pragma unroll
          for (int g = 0; g < GP; ++g) {
            const uint32_t addr = pb + (uint32_t)((g >> 3) * 1024 + (g & 7) * 128 +
                                                  ((((col >> 3) ^ (g & 7))) << 4) + (col & 7) * 2);
            st_shared_u16(addr, (uint16_t)((g & 1) ? (pw[g >> 1] >> 16) : (pw[g >> 1] & 0xffffu)));
          }
        }
        if (tid == 64) tc_trace<kTrace>(p, 2, ntr, 25, (uint32_t)g_k);
        tc::fence_proxy_async_smem();
        mbar_arrive(bars.p_full + 8u * sb);
        if (tid == 64) tc_trace<kTrace>(p, 2, ntr, 6, (uint32_t)g_k);
        else if (lane == 0) tc_trace<kTrace>(p, warp, ntr, 19, (uint32_t)((warp << 16) | g_k));
      }
      // A failed wait above is per thread: the barrier below settles it for
      // the warpgroup (a thread leaving alone would strand the others).
      // l over the warpgroup's 128 token rows (final after the last stage's
      // weights, so it is summed while the last P.V runs), then the item's
      // last PV tile; the barrier also decides for the whole warpgroup, so
      // that every warp executes the tensor-memory load convergently or not
      // at all.
#pragma unroll
      for (int g = 0; g < GP; ++g) {
        const float s_ = warp_sum(l_run[g]);
        if (lane == 0) red2[q4 * kTcHeads + g] = s_;
      }
      if (!(ok = softmax_group_all(ok && !flags[0]))) break;
      {
        const int gl = gk + n - 1;
        ok = mbar_wait_bounded(bars.o_full + 8u * (gl & 1), (gl >> 1) & 1, p.err, p.wait_limit);
        __syncwarp();
        tc::fence_after_sync();
        tc::tmem_ld<GP>(tO_lane, o_acc);
        tc::tmem_wait_ld();
        tc::fence_before_sync();
      }
      if (tid == 64) tc_trace<kTrace>(p, 2, ntr, 16, (uint32_t)(gk + n - 1));
      gk += n;
      {
        // One warp runs this once per item, so its instruction count is its
        // latency: per-head work (the sum over the four quarters, the
        // reciprocal, the log-sum-exp) is done by lane g for head g, in
        // parallel, and broadcast; lane i then writes column d of its heads.
        // For D = 128 each warp holds 32 columns of every head.  For D = 64
        // rows 64..127 of O^T repeat rows 0..63, so warps 2, 3 hold the same
        // columns as warps 4, 5, and the heads are split between the pairs.
        const int d = row & (D - 1);
        const int g_lo = D == 64 ? (q4 >> 1) * ((G + 1) >> 1) : 0;
        const int g_hi = D == 64 ? min(G, g_lo + ((G + 1) >> 1)) : G;
        float lsum_l = 1.f, m_l = 0.f;
        if (lane < GP) {
          lsum_l = red2[lane] + red2[kTcHeads + lane] + red2[2 * kTcHeads + lane] +
                   red2[3 * kTcHeads + lane];
#pragma unroll
          for (int g = 0; g < GP; ++g)
            if (lane == g) m_l = m_run[g];
        }
        const float inv_l = 1.f / lsum_l;
#pragma unroll
        for (int g = 0; g < GP; ++g) {
          const float val = o_acc[g] * __shfl_sync(0xffffffffu, inv_l, g);
          if (g < g_lo || g >= g_hi) continue;
          if (it.final_out)
            reinterpret_cast<__nv_bfloat16*>(p.out)[(row0 + g) * D + d] = __float2bfloat16_rn(val);
          else
            p.part_o[((row0 + g) * (size_t)p.max_parts + it.part) * D + d] = val;
        }
        if (!it.final_out && q4 == 0 && lane < G)
          p.part_lse[(row0 + lane) * (size_t)p.max_parts + it.part] = m_l + log2f(lsum_l);
      }
      if (tid == 64) tc_trace<kTrace>(p, 2, ntr, 7, (uint32_t)ii);
      else if (lane == 0) tc_trace<kTrace>(p, warp, ntr, 22, (uint32_t)((warp << 16) | ii));
    }
    if (!ok) flags[0] = 1;
  }

  tc::fence_before_sync();
  __syncthreads();
  if (tid == 0) {
    if (flags[0]) {
      // Wait (bounded) for every TMA load this CTA issued.
      const int issued = flags[1];
      for (int sl = 0; sl < NS && sl < issued; ++sl)
        mbar_wait_bounded(bars.full0 + 8u * sl, ((issued - 1 - sl) / NS) & 1, p.err);
      const int qissued = flags[2];
      for (int b = 0; b < 2 && b < qissued; ++b)
        mbar_wait_bounded(bars.q_full + 8u * b, ((qissued - 1 - b) / 2) & 1, p.err);
    }
    // The last CTA to finish resets the work counter for the next call.
    __threadfence();
    if (atomicAdd(p.sched + 1, 1u) == gridDim.x - 1) {
      p.sched[0] = 0u;
      p.sched[1] = 0u;
      __threadfence();
    }
  }
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTcTmemCols);
  }
}

}  // namespace pa
