// Device-side helpers for the sm_103a kernels: shared-memory barriers, TMA
// tensor loads, bounded waits, bf16 unpacking and the device error word.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pa.h"

namespace pa {

// A bounded wait gives up after this many SM clock cycles (about two seconds
// at 2 GHz), records PA_DEVERR_TIMEOUT and lets the kernel return.  The
// clock is read only every 64 polls, so a wait that succeeds quickly costs
// nothing beyond the polls.
constexpr long long kWaitLimitCycles = 4000000000ll;

__device__ __forceinline__ void record_error(unsigned int* err, unsigned int bits) {
  if (err) atomicOr(err, bits);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- programmatic dependent launch ------------------------------------------
// Every kernel of the library is launched so that it may start while the
// previous kernel on its stream is still finishing.  Before its first access
// to global memory each thread waits until the grids it depends on have
// completed and their writes are visible (a no-op for a kernel launched
// without the attribute).  Every thread executes the wait, so no grid of the
// library completes before the grid it follows: completion stays ordered
// along the stream.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Let the next grid on the stream start launching (its own wait still holds
// it back until this grid has completed).
__device__ __forceinline__ void grid_dependents_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- mbarrier -------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Non-blocking test: has the phase with the given parity completed?
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Suspend until the phase with the given parity completes or about `ns`
// nanoseconds pass, whichever comes first (the result is not reported).
__device__ __forceinline__ void mbar_suspend(uint32_t bar, uint32_t parity, uint32_t ns) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%0], %1, %2;\n\t}" ::"r"(bar),
      "r"(parity), "r"(ns)
      : "memory");
}

// Wait until the phase with the given parity has completed.  Returns false
// (and records PA_DEVERR_TIMEOUT) if that takes longer than `limit` SM clock
// cycles (kWaitLimitCycles unless the launch asked for another limit).
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  unsigned int* err,
                                                  long long limit = kWaitLimitCycles) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0 && clock64() - t0 > limit) {
      record_error(err, PA_DEVERR_TIMEOUT);
      return false;
    }
  }
}

// ---- TMA ------------------------------------------------------------------

// Fetch the 128-byte line holding p into L2.
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 5-D tiled tensor load into this CTA's shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_5d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1, int c2, int c3, int c4) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4),
      "r"(bar)
      : "memory");
}

// Prefetch a 5-D box of the map into L2 (no shared memory, no completion).
__device__ __forceinline__ void tma_prefetch_l2_5d(const CUtensorMap* map, int c0, int c1, int c2,
                                                   int c3, int c4) {
  asm volatile(
      "cp.async.bulk.prefetch.tensor.5d.L2.global.tile [%0, {%1, %2, %3, %4, %5}];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
      : "memory");
}

// ---- loads ------------------------------------------------------------------

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ float4 lds128f(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void stg_v4(void* p, uint4 v) {
  asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

// ---- the fused cache write ----------------------------------------------------

// Order this thread's generic-proxy global writes before later async-proxy
// (TMA) reads of the same memory.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// The fused write split in two, so that the load's latency can overlap other
// work: load_new_token fetches the newest token's K and V rows of KV head h of
// sequence s into the warp's lanes (lane i < 2 * chunks holds 16-byte chunk i,
// keys first; 2 * chunks <= 32, i.e. rows of at most 256 bytes), and
// store_new_token writes them into slot `pos` of block `id` (warp-uniform).
// An id outside the pool skips the store and records PA_DEVERR_BLOCK_ID.  The
// caller fences (fence_proxy_async_global, every lane) before a TMA read of
// the slot.
__device__ __forceinline__ uint4 load_new_token(const void* new_k, const void* new_v, int s,
                                                int h, int num_kv_heads, int chunks, int lane) {
  uint4 v = make_uint4(0u, 0u, 0u, 0u);
  if (lane < 2 * chunks) {
    const int kv = lane >= chunks;
    const int c = lane - kv * chunks;
    v = ldg_nc_v4(reinterpret_cast<const uint4*>(kv ? new_v : new_k) +
                  ((size_t)s * num_kv_heads + h) * chunks + c);
  }
  return v;
}

__device__ __forceinline__ void store_new_token(uint8_t* cache, uint4 v, int id, int h, int pos,
                                                int num_kv_heads, int chunks, int block_size,
                                                int num_blocks, unsigned int* err, int lane) {
  const bool ok = id >= 0 && id < num_blocks;
  if (!ok && lane == 0) record_error(err, PA_DEVERR_BLOCK_ID);
  if (ok && lane < 2 * chunks) {
    const int kv = lane >= chunks;
    const int c = lane - kv * chunks;
    const size_t row_bytes = (size_t)num_kv_heads * chunks * 16;
    uint8_t* dst = cache + (size_t)kv * num_blocks * block_size * row_bytes +
                   ((size_t)id * block_size + (pos & (block_size - 1))) * row_bytes +
                   (size_t)h * chunks * 16 + (size_t)c * 16;
    stg_v4(dst, v);
  }
}

// Write the newest token (position `pos` of sequence s) of KV head h into
// its cache slot, keys and values, one 16-byte chunk per lane (rows of
// `chunks` chunks), then make the writes visible to TMA reads by the warp.
// The slot's block comes from the sequence's table row; an id outside the
// pool skips the write and records PA_DEVERR_BLOCK_ID.  Whole warp.
__device__ __forceinline__ void write_new_token(uint8_t* cache, const void* new_k,
                                                const void* new_v, const int32_t* table_row,
                                                int s, int h, int pos, int num_kv_heads,
                                                int chunks, int block_size, int log2_block_size,
                                                int num_blocks, unsigned int* err, int lane) {
  const int id = __ldg(table_row + (pos >> log2_block_size));
  const bool ok = id >= 0 && id < num_blocks;
  if (!ok && lane == 0) record_error(err, PA_DEVERR_BLOCK_ID);
  const size_t row_bytes = (size_t)num_kv_heads * chunks * 16;
  for (int i = lane; ok && i < 2 * chunks; i += 32) {
    const int kv = i >= chunks;
    const int c = i - kv * chunks;
    const uint4* src = reinterpret_cast<const uint4*>(kv ? new_v : new_k) +
                       ((size_t)s * num_kv_heads + h) * chunks + c;
    uint8_t* dst = cache + (size_t)kv * num_blocks * block_size * row_bytes +
                   ((size_t)id * block_size + (pos & (block_size - 1))) * row_bytes +
                   (size_t)h * chunks * 16 + (size_t)c * 16;
    stg_v4(dst, ldg_nc_v4(src));
  }
  fence_proxy_async_global();
  __syncwarp();
  fence_proxy_async_global();
}

// ---- arithmetic -------------------------------------------------------------

// 2^x on the MUFU unit (x = -inf gives +0).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Maximum of v over the full warp, in one warp reduction instruction.
__device__ __forceinline__ float warp_max_redux(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}

// lo and hi rounded to bf16 (nearest even) and packed, lo in bits 0..15.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// The two bf16 halves of a 32-bit word as fp32 (exact).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

template <typename T>
struct ElemTraits;

template <>
struct ElemTraits<__nv_bfloat16> {
  static constexpr int kBytes = 2;
  static constexpr int kPerChunk = 8;  // elements in 16 bytes
  // Unpack 16 bytes into 8 floats.
  static __device__ __forceinline__ void unpack(const uint4& w, float* f) {
    f[0] = bf16_lo(w.x); f[1] = bf16_hi(w.x);
    f[2] = bf16_lo(w.y); f[3] = bf16_hi(w.y);
    f[4] = bf16_lo(w.z); f[5] = bf16_hi(w.z);
    f[6] = bf16_lo(w.w); f[7] = bf16_hi(w.w);
  }
  static __device__ __forceinline__ float to_float(__nv_bfloat16 x) { return __bfloat162float(x); }
  static __device__ __forceinline__ __nv_bfloat16 from_float(float x) {
    return __float2bfloat16_rn(x);
  }
};

template <>
struct ElemTraits<float> {
  static constexpr int kBytes = 4;
  static constexpr int kPerChunk = 4;
  static __device__ __forceinline__ void unpack(const uint4& w, float* f) {
    f[0] = __uint_as_float(w.x); f[1] = __uint_as_float(w.y);
    f[2] = __uint_as_float(w.z); f[3] = __uint_as_float(w.w);
  }
  static __device__ __forceinline__ float to_float(float x) { return x; }
  static __device__ __forceinline__ float from_float(float x) { return x; }
};

}  // namespace pa
