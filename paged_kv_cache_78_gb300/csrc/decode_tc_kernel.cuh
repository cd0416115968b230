// Paged decode attention on the 5th-generation tensor cores (tcgen05, bf16).
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
// The 16 columns are the query heads of one KV head (G <= 16, padded with
// zero rows).  One CTA = one (partition, KV head, sequence); six warps:
//   warp 0      TMA producer: 128-token stages, one box per (block, 128-byte
//               column group, K or V), written in the 128-byte swizzle that
//               the MMA descriptors read directly (K tile: K-major A operand;
//               V tile: M-major A operand);
//   warp 1      tensor-memory allocator and MMA issuer (one thread): QK of
//               stage k+1 is issued before PV of stage k, so the QK overlaps
//               the softmax of stage k;
//   warps 2..5  softmax warpgroup, one token (QK) or one head dimension (PV)
//               per tensor-memory lane: online softmax in fp32 (log2 domain),
//               P^T written to shared memory as bf16, and the PV result of each
//               stage added into fp32 registers with the running rescale.
// Tensor memory: S double buffer (2 x 16 columns), O double buffer (2 x 16).
// Every wait is bounded; a timeout records PA_DEVERR_TIMEOUT, the CTA drains
// its MMAs and TMA loads, frees its tensor memory and returns.
#pragma once

#include "decode_kernel.cuh"
#include "pa_tcgen05.cuh"

namespace pa {

constexpr int kTcTokens = 128;   // tokens per stage = M of the QK MMA
constexpr int kTcHeads = 16;     // N of both MMAs: query heads, G padded
constexpr int kTcThreads = 192;  // producer, MMA, 4 softmax warps
constexpr int kTcTmemCols = 64;

// Shared-memory layout of the tensor-core decode kernel (byte offsets from
// a 1024-aligned base).
struct TcSmem {
  int region;  // K (or V) tile of one stage
  int stage;
  int q_off;
  int p_off;
  int red_off;
  int bar_off;
  int misc_off;
  int total;   // bytes to request (includes 1024 of alignment slack)
};

__host__ __device__ inline TcSmem tc_smem_layout(int head_size, int num_stages) {
  TcSmem l;
  l.region = (head_size / 64) * kTcTokens * 128;
  l.stage = 2 * l.region;
  l.q_off = num_stages * l.stage;
  l.p_off = l.q_off + (head_size / 64) * kTcHeads * 128;
  l.red_off = l.p_off + 2 * 2 * kTcHeads * 128;
  l.bar_off = l.red_off + 3 * 4 * kTcHeads * 4;
  l.misc_off = l.bar_off + 8 * (2 * num_stages + 11);
  l.total = l.misc_off + 64 + 1024;
  return l;
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

// MMA issuer: QK of stage k (S^T = K_tile . Q^T) into tensor-memory buffer
// k % 2, once the stage has landed and that buffer has been read.
template <int kKSteps, int kGroupBytes, uint32_t kIdesc>
__device__ __forceinline__ bool tc_issue_qk(int k, int NS, uint32_t full0, uint32_t s_full,
                                            uint32_t s_free, uint32_t sbase, int stage_bytes,
                                            uint32_t q_s, uint32_t t_s, unsigned int* err) {
  const int slot = k % NS;
  const int sb = k & 1;
  if (!mbar_wait_bounded(full0 + 8u * slot, (k / NS) & 1, err)) return false;
  if (k >= 2 && !mbar_wait_bounded(s_free + 8u * sb, ((k >> 1) - 1) & 1, err)) return false;
  tc::fence_after_sync();
  const uint32_t ka = sbase + (uint32_t)slot * (uint32_t)stage_bytes;
#pragma unroll
  for (int kk = 0; kk < kKSteps; ++kk) {
    const uint32_t goff = (uint32_t)((kk >> 2) * kGroupBytes) + (uint32_t)((kk & 3) * 32);
    const uint64_t a = tc::smem_desc_sw128(ka + goff, 16, 1024);
    const uint64_t b =
        tc::smem_desc_sw128(q_s + (uint32_t)((kk >> 2) * kTcHeads * 128 + (kk & 3) * 32), 16, 1024);
    tc::mma_bf16(t_s + 16u * sb, a, b, kIdesc, kk > 0);
  }
  tc::mma_commit(s_full + 8u * sb);
  return true;
}

// Softmax warpgroup: add the PV tile of stage j (tensor-memory buffer j % 2)
// into the fp32 accumulator, rescaled by that stage's factor.
__device__ __forceinline__ bool tc_epilogue(int j, uint32_t o_full, uint32_t o_free,
                                            uint32_t t_o_lane, unsigned int* err,
                                            float (&o_acc)[kTcHeads],
                                            const float (&alpha)[kTcHeads]) {
  const int sb = j & 1;
  const bool w = mbar_wait_bounded(o_full + 8u * sb, (j >> 1) & 1, err);
  __syncwarp();
  tc::fence_after_sync();
  float ot[kTcHeads];
  tc::tmem_ld16(t_o_lane + 16u * sb, ot);
  tc::tmem_wait_ld();
  tc::fence_before_sync();
  mbar_arrive(o_free + 8u * sb);
#pragma unroll
  for (int g = 0; g < kTcHeads; ++g) o_acc[g] = fmaf(o_acc[g], alpha[g], ot[g]);
  return w;
}

template <int D>
__global__ void __launch_bounds__(kTcThreads, 1)
    paged_decode_tc_kernel(const __grid_constant__ CUtensorMap kv_map, const DecodeParams p) {
  static_assert(D == 64 || D == 128, "tensor-core decode handles head sizes 64 and 128");
  constexpr int kGroups = D / 64;                 // 128-byte column groups of a row
  constexpr int kGroupBytes = kTcTokens * 128;    // one column group of a 128-token tile
  constexpr int kRegion = kGroups * kGroupBytes;  // K (or V) tile of a stage
  constexpr int kKSteps = D / 16;                 // QK: K = head dimension
  constexpr int kPvSteps = kTcTokens / 16;        // PV: K = tokens
  constexpr uint32_t kIdescQK = tc::idesc_bf16_f32(128, kTcHeads, 0);
  constexpr uint32_t kIdescPV = tc::idesc_bf16_f32(128, kTcHeads, 1);
  // PV's A operand (V^T) spans 128 rows = two 64-dimension groups; with one
  // group (D = 64) both halves read the same group and rows 64..127 repeat.
  constexpr uint32_t kPvLbo = kGroups > 1 ? kGroupBytes : 0;

  const int part = blockIdx.x;
  const int h = blockIdx.y;
  const int s = blockIdx.z;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int G = p.group;

  const int L = p.seq_lens[s];
  const int P = p.partition_tokens;
  const bool split = P > 0;
  const int nparts = L <= 0 ? 0 : (split ? (L + P - 1) / P : 1);
  const size_t row0 = (size_t)s * p.num_heads + (size_t)h * G;

  if (L <= 0) {
    if (part == 0) {
      __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out) + row0 * D;
      for (int i = tid; i < G * D; i += blockDim.x) out[i] = __float2bfloat16_rn(0.f);
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
  const int n_stages = (tok1 - tok0 + kTcTokens - 1) / kTcTokens;
  const int NS = p.num_stages;
  const TcSmem lay = tc_smem_layout(D, NS);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(base);
  const uint32_t q_s = sbase + lay.q_off;
  const uint32_t p_s = sbase + lay.p_off;
  float* red = reinterpret_cast<float*>(base + lay.red_off);  // [3][4 warps][16 heads]
  const uint32_t bars = sbase + lay.bar_off;
  const uint32_t full0 = bars;
  const uint32_t empty0 = bars + 8u * NS;
  const uint32_t s_full = bars + 16u * NS;   // [2]
  const uint32_t s_free = s_full + 16;       // [2]
  const uint32_t p_full = s_full + 32;       // [2]
  const uint32_t o_full = s_full + 48;       // [2]
  const uint32_t o_free = s_full + 64;       // [2]
  const uint32_t drain = s_full + 80;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + lay.misc_off);
  volatile int* flags = reinterpret_cast<volatile int*>(base + lay.misc_off + 16);

  if (tid == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(full0 + 8u * i, 1);
      mbar_init(empty0 + 8u * i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(s_full + 8u * i, 1);
      mbar_init(s_free + 8u * i, 128);
      mbar_init(p_full + 8u * i, 128);
      mbar_init(o_full + 8u * i, 1);
      mbar_init(o_free + 8u * i, 128);
    }
    mbar_init(drain, 1);
    flags[0] = 0;  // abort
    flags[1] = 0;  // stages issued
    fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(smem_u32(tmem_slot), kTcTmemCols);
    tc::tmem_relinquish();
  }
  if (tid == 32) tma_prefetch_desc(&kv_map);
  // Q^T as the QK's B operand: [column group][16 rows][128 bytes], 128-byte
  // swizzle (16-byte chunk c of row r stored at chunk c ^ (r % 8)); rows at or
  // beyond G are zero.
  {
    const __nv_bfloat16* qg = reinterpret_cast<const __nv_bfloat16*>(p.query) + row0 * D;
    for (int i = tid; i < kTcHeads * D; i += blockDim.x) {
      const int r = i / D;
      const int d = i - r * D;
      const __nv_bfloat16 v = r < G ? qg[r * D + d] : __float2bfloat16_rn(0.f);
      const int col = d & 63;
      const uint32_t addr = q_s + (uint32_t)((d >> 6) * kTcHeads * 128 + (r >> 3) * 1024 +
                                             (r & 7) * 128 + ((((col >> 3) ^ (r & 7))) << 4) +
                                             (col & 7) * 2);
      st_shared_u16(addr, __bfloat16_as_ushort(v));
    }
  }
  tc::fence_proxy_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS0 = tmem, tO0 = tmem + 32;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    const int BS = p.block_size;
    const int l2bs = p.log2_block_size;
    const int R = p.box_rows;  // min(block_size, 128)
    const int log2R = p.log2_box_rows;
    const int32_t* table = p.block_tables + (size_t)s * p.max_blocks_per_seq;
    const int lb_end = (tok1 + BS - 1) >> l2bs;
    int win = tok0 >> l2bs;
    int cur = (win + lane < lb_end) ? __ldg(table + win + lane) : 0;
    int nxt = (win + 32 + lane < lb_end) ? __ldg(table + win + 32 + lane) : 0;
    const uint32_t box_bytes = (uint32_t)R * 128u;
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
      const int st_tok = tok0 + k * kTcTokens;
      const int st_n = min(kTcTokens, tok1 - st_tok);
      const int nbox = (st_n + R - 1) >> log2R;
      if (lane == 0)
        mbar_arrive_expect_tx(full0 + 8u * slot, (uint32_t)(nbox * kGroups * 2) * box_bytes);
      const uint32_t kdst = sbase + (uint32_t)slot * (uint32_t)lay.stage;
      for (int i = 0; i < nbox; ++i) {
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
            record_error(p.err, PA_DEVERR_BLOCK_ID);
            ck = cv = 2 * p.num_blocks;  // outside the tensor: zero fill
          }
#pragma unroll
          for (int g = 0; g < kGroups; ++g) {
            const uint32_t dst = kdst + (uint32_t)(g * kGroupBytes) + (uint32_t)i * box_bytes;
            tma_load_5d(dst, &kv_map, full0 + 8u * slot, 0, g, h, t0, ck);
            tma_load_5d(dst + kRegion, &kv_map, full0 + 8u * slot, 0, g, h, t0, cv);
          }
        }
      }
      issued = k + 1;
    }
    if (lane == 0) flags[1] = issued;
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      bool ok = true;
      if (n_stages > 0) ok = tc_issue_qk<kKSteps, kGroupBytes, kIdescQK>(0, NS, full0, s_full, s_free, sbase, lay.stage, q_s, tS0, p.err);
      for (int k = 0; ok && k < n_stages; ++k) {
        if (k + 1 < n_stages &&
            !(ok = tc_issue_qk<kKSteps, kGroupBytes, kIdescQK>(k + 1, NS, full0, s_full, s_free,
                                                              sbase, lay.stage, q_s, tS0, p.err)))
          break;
        const int slot = k % NS;
        const int sb = k & 1;
        if (!(ok = mbar_wait_bounded(p_full + 8u * sb, (k >> 1) & 1, p.err))) break;
        if (k >= 2 && !(ok = mbar_wait_bounded(o_free + 8u * sb, ((k >> 1) - 1) & 1, p.err)))
          break;
        tc::fence_after_sync();
        const uint32_t va = sbase + (uint32_t)slot * (uint32_t)lay.stage + (uint32_t)kRegion;
        const uint32_t pa_ = p_s + (uint32_t)sb * 2u * kTcHeads * 128u;
#pragma unroll
        for (int kk = 0; kk < kPvSteps; ++kk) {
          const uint64_t a = tc::smem_desc_sw128(va + (uint32_t)kk * 2048u, kPvLbo, 1024);
          const uint64_t b = tc::smem_desc_sw128(
              pa_ + (uint32_t)((kk >> 2) * kTcHeads * 128 + (kk & 3) * 32), 16, 1024);
          tc::mma_bf16(tO0 + 16u * sb, a, b, kIdescPV, kk > 0);
        }
        tc::mma_commit(o_full + 8u * sb);
        tc::mma_commit(empty0 + 8u * slot);
      }
      if (!ok) flags[0] = 1;
      // Every MMA this thread issued completes before the CTA may free its
      // tensor memory.
      tc::mma_commit(drain);
      mbar_wait_bounded(drain, 0, p.err);
    }
    __syncwarp();
  } else {
    // ---------------- softmax warpgroup ----------------
    const int q4 = warp & 3;                  // tensor-memory lane quarter
    const int row = q4 * 32 + lane;           // token (QK) / head dimension (PV)
    const uint32_t lane_addr = (uint32_t)(q4 * 32) << 16;
    float m_run[kTcHeads], l_run[kTcHeads], o_acc[kTcHeads], alpha_prev[kTcHeads];
#pragma unroll
    for (int g = 0; g < kTcHeads; ++g) {
      m_run[g] = -INFINITY;
      l_run[g] = 0.f;
      o_acc[g] = 0.f;
      alpha_prev[g] = 1.f;
    }
    bool ok = true;

    for (int k = 0; k < n_stages; ++k) {
      const int sb = k & 1;
      const int slot = k % NS;
      bool w = mbar_wait_bounded(s_full + 8u * sb, (k >> 1) & 1, p.err);
      __syncwarp();
      tc::fence_after_sync();
      float sc[kTcHeads];
      tc::tmem_ld16(tS0 + 16u * sb + lane_addr, sc);
      tc::tmem_wait_ld();
      tc::fence_before_sync();
      mbar_arrive(s_free + 8u * sb);

      const int nvalid = min(kTcTokens, tok1 - (tok0 + k * kTcTokens));
      const bool valid = row < nvalid;
      if (!valid) {
        // A stale row of V (past the sequence, or never loaded) must not reach
        // the PV product: 0 * NaN would.
        const uint32_t vrow = sbase + (uint32_t)slot * (uint32_t)lay.stage + (uint32_t)kRegion +
                              (uint32_t)row * 128u;
#pragma unroll
        for (int g = 0; g < kGroups; ++g)
#pragma unroll
          for (int c = 0; c < 8; ++c) st_shared_zero16(vrow + (uint32_t)(g * kGroupBytes + c * 16));
      }
      float x[kTcHeads];
#pragma unroll
      for (int g = 0; g < kTcHeads; ++g)
        x[g] = (valid && g < G) ? sc[g] * p.scale_log2 : -INFINITY;
      float* redk = red + sb * 4 * kTcHeads;
#pragma unroll
      for (int g = 0; g < kTcHeads; ++g) {
        if (g < G) {
          const float wm = warp_max(x[g]);
          if (lane == 0) redk[q4 * kTcHeads + g] = wm;
        }
      }
      if (!softmax_group_all(w && ok && !flags[0])) {
        ok = false;
        break;
      }
      float alpha[kTcHeads], pr[kTcHeads];
#pragma unroll
      for (int g = 0; g < kTcHeads; ++g) {
        if (g < G) {
          const float tmax = fmaxf(fmaxf(redk[g], redk[kTcHeads + g]),
                                   fmaxf(redk[2 * kTcHeads + g], redk[3 * kTcHeads + g]));
          const float m_new = fmaxf(m_run[g], tmax);
          alpha[g] = fast_exp2(m_run[g] - m_new);
          m_run[g] = m_new;
          // The weight enters P.V rounded to bf16; the denominator sums the
          // same rounded weights, so the output stays a convex combination.
          pr[g] = __bfloat162float(__float2bfloat16_rn(fast_exp2(x[g] - m_new)));
          l_run[g] = fmaf(l_run[g], alpha[g], pr[g]);
        } else {
          alpha[g] = 1.f;
          pr[g] = 0.f;
        }
      }
      // P^T as the PV's B operand: [64-token group][16 rows][128 bytes], swizzled.
      {
        const uint32_t pb = p_s + (uint32_t)sb * 2u * kTcHeads * 128u +
                            (uint32_t)((row >> 6) * kTcHeads * 128);
        const int col = row & 63;
#pragma unroll
        for (int g = 0; g < kTcHeads; ++g) {
          const uint32_t addr = pb + (uint32_t)((g >> 3) * 1024 + (g & 7) * 128 +
                                                ((((col >> 3) ^ (g & 7))) << 4) + (col & 7) * 2);
          st_shared_u16(addr, __bfloat16_as_ushort(__float2bfloat16_rn(pr[g])));
        }
      }
      tc::fence_proxy_async_smem();
      mbar_arrive(p_full + 8u * sb);
      if (k >= 1) ok = tc_epilogue(k - 1, o_full, o_free, tO0 + lane_addr, p.err, o_acc, alpha_prev) && ok;
#pragma unroll
      for (int g = 0; g < kTcHeads; ++g) alpha_prev[g] = alpha[g];
    }
    // The last PV tile; the decision is taken by the whole warpgroup so that
    // every warp executes the tensor-memory load convergently or not at all.
    ok = softmax_group_all(ok && !flags[0]);
    if (ok && n_stages > 0)
      ok = tc_epilogue(n_stages - 1, o_full, o_free, tO0 + lane_addr, p.err, o_acc, alpha_prev);

    // l over the warpgroup's 128 token rows.
    float* red2 = red + 2 * 4 * kTcHeads;
#pragma unroll
    for (int g = 0; g < kTcHeads; ++g) {
      if (g < G) {
        const float ws = warp_sum(l_run[g]);
        if (lane == 0) red2[q4 * kTcHeads + g] = ws;
      }
    }
    ok = softmax_group_all(ok && !flags[0]);
    if (!ok) {
      flags[0] = 1;
    } else if (row < D) {
      const int d = row;
#pragma unroll
      for (int g = 0; g < kTcHeads; ++g) {
        if (g >= G) continue;
        const float lsum = red2[g] + red2[kTcHeads + g] + red2[2 * kTcHeads + g] +
                           red2[3 * kTcHeads + g];
        const float val = o_acc[g] / lsum;
        if (nparts == 1) {
          reinterpret_cast<__nv_bfloat16*>(p.out)[(row0 + g) * D + d] = __float2bfloat16_rn(val);
        } else {
          const size_t prow = (row0 + g) * (size_t)p.max_parts + part;
          p.part_o[prow * D + d] = val;
          if (d == 0) p.part_lse[prow] = m_run[g] + log2f(lsum);
        }
      }
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (flags[0] && tid == 0) {
    // Wait (bounded) for every TMA load this CTA issued.
    const int issued = flags[1];
    for (int sl = 0; sl < NS && sl < issued; ++sl) {
      const int last_use = (issued - 1 - sl) / NS;
      mbar_wait_bounded(full0 + 8u * sl, last_use & 1, p.err);
    }
  }
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTcTmemCols);
  }
}

}  // namespace pa
