// Launch of the tensor-core decode kernels: one translation unit per (head
// size, timeline on or off) instantiates its query-group and split-mode
// variants, so the build stays parallel.
#pragma once

#include <algorithm>
#include <atomic>

#include "decode_tc_kernel.cuh"
#include "pa_launch.h"

namespace pa {

template <int D, int GP, bool kBal, bool kTrace>
static cudaError_t launch_tc(int num_sms, int smem_bytes, cudaStream_t stream,
                             const CUtensorMap& kv_map, const CUtensorMap& q_map,
                             const DecodeParams& params) {
  static std::atomic<int> configured[64];
  static std::atomic<int> smem_per_sm[64];
  static std::atomic<int> ctas_by_regs[64];
  auto kernel = paged_decode_tc_kernel<D, GP, kBal, kTrace>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (smem_bytes > configured[dev].load(std::memory_order_relaxed)) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, kernel);
    if (e != cudaSuccess) return e;
    int sm_smem = 0, regs_per_sm = 0;
    e = cudaDeviceGetAttribute(&sm_smem, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&regs_per_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev);
    if (e != cudaSuccess) return e;
    const int regs_per_warp = (fa.numRegs * 32 + 255) / 256 * 256;
    smem_per_sm[dev].store(sm_smem, std::memory_order_relaxed);
    ctas_by_regs[dev].store(regs_per_sm / (regs_per_warp * (kTcThreads / 32)),
                            std::memory_order_relaxed);
    configured[dev].store(smem_bytes, std::memory_order_relaxed);
  }
  // Resident CTAs per SM at this launch's shared memory (plus the 1 KB the
  // driver reserves per CTA), registers and tensor-memory columns.
  int per_sm = smem_per_sm[dev].load(std::memory_order_relaxed) / (smem_bytes + 1024);
  per_sm = std::min(per_sm, ctas_by_regs[dev].load(std::memory_order_relaxed));
  per_sm = std::min(per_sm, 512 / kTcTmemCols);
  if (per_sm < 1) per_sm = 1;
  // Persistent grid: as many CTAs as fit at once, at most one per work item.
  long long grid = (long long)num_sms * per_sm;
  if (grid > params.total_items) grid = params.total_items;
  if (grid < 1) return cudaSuccess;
  DecodeParams prm = params;
  if (kTrace && prm.trace != nullptr &&
      (size_t)grid * kTcTraceRoles * (size_t)prm.trace_per_role * 16 > (size_t)prm.trace_bytes)
    prm.trace = nullptr;  // the buffer cannot hold this launch's timeline: record nothing
  void* args[] = {const_cast<CUtensorMap*>(&kv_map), const_cast<CUtensorMap*>(&q_map), &prm};
  return launch_overlapped((const void*)kernel, dim3((unsigned)grid), dim3(kTcThreads),
                           (size_t)smem_bytes, stream, args);
}

template <int D, int GP, bool kTrace>
static cudaError_t launch_tc_mode(int num_sms, int smem_bytes, cudaStream_t stream,
                                  const CUtensorMap& kv_map, const CUtensorMap& q_map,
                                  const DecodeParams& params) {
  return params.balanced
             ? launch_tc<D, GP, true, kTrace>(num_sms, smem_bytes, stream, kv_map, q_map, params)
             : launch_tc<D, GP, false, kTrace>(num_sms, smem_bytes, stream, kv_map, q_map, params);
}

template <int D, bool kTrace>
cudaError_t launch_tc_head_size(int num_sms, int smem_bytes, cudaStream_t stream,
                                const CUtensorMap& kv_map, const CUtensorMap& q_map,
                                const DecodeParams& params) {
  const int g = params.group;
  if (g <= 1) return launch_tc_mode<D, 1, kTrace>(num_sms, smem_bytes, stream, kv_map, q_map, params);
  if (g <= 2) return launch_tc_mode<D, 2, kTrace>(num_sms, smem_bytes, stream, kv_map, q_map, params);
  if (g <= 4) return launch_tc_mode<D, 4, kTrace>(num_sms, smem_bytes, stream, kv_map, q_map, params);
  if (g <= 8) return launch_tc_mode<D, 8, kTrace>(num_sms, smem_bytes, stream, kv_map, q_map, params);
  return launch_tc_mode<D, 16, kTrace>(num_sms, smem_bytes, stream, kv_map, q_map, params);
}

}  // namespace pa

#define PA_DEFINE_TC_UNIT(D, TRACE, NAME)                                                    \
  namespace pa {                                                                             \
  cudaError_t NAME(int num_sms, int smem_bytes, cudaStream_t stream,                         \
                   const CUtensorMap& kv_map, const CUtensorMap& q_map,                      \
                   const DecodeParams& params) {                                             \
    return launch_tc_head_size<D, TRACE>(num_sms, smem_bytes, stream, kv_map, q_map, params); \
  }                                                                                          \
  }
