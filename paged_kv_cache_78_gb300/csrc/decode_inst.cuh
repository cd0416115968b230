// Instantiation helpers for the decode kernels: one translation unit per
// (element type, head size) keeps the build parallel.
#pragma once

#include <atomic>

#include "decode_kernel.cuh"
#include "pa_launch.h"

namespace pa {

template <typename T, int D, int G>
cudaError_t launch_decode_one(dim3 grid, int smem_bytes, cudaStream_t stream,
                              const CUtensorMap& map, const DecodeParams& params) {
  // The dynamic shared-memory limit is a per-device function attribute; raise
  // it once per device to the largest size seen.
  static std::atomic<int> configured[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (smem_bytes > configured[dev].load(std::memory_order_relaxed)) {
    e = cudaFuncSetAttribute(paged_decode_kernel<T, D, G>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e != cudaSuccess) return e;
    configured[dev].store(smem_bytes, std::memory_order_relaxed);
  }
  void* args[] = {const_cast<CUtensorMap*>(&map), const_cast<DecodeParams*>(&params)};
  return launch_overlapped((const void*)paged_decode_kernel<T, D, G>, grid, dim3(kDecodeThreads),
                           (size_t)smem_bytes, stream, args);
}

template <typename T, int D>
cudaError_t launch_decode_for_head_size(int group, dim3 grid, int smem_bytes,
                                        cudaStream_t stream, const CUtensorMap& map,
                                        const DecodeParams& params, bool* supported) {
  *supported = true;
  switch (group) {
    case 1: return launch_decode_one<T, D, 1>(grid, smem_bytes, stream, map, params);
    case 2: return launch_decode_one<T, D, 2>(grid, smem_bytes, stream, map, params);
    case 3: return launch_decode_one<T, D, 3>(grid, smem_bytes, stream, map, params);
    case 4: return launch_decode_one<T, D, 4>(grid, smem_bytes, stream, map, params);
    case 5: return launch_decode_one<T, D, 5>(grid, smem_bytes, stream, map, params);
    case 6: return launch_decode_one<T, D, 6>(grid, smem_bytes, stream, map, params);
    case 7: return launch_decode_one<T, D, 7>(grid, smem_bytes, stream, map, params);
    case 8: return launch_decode_one<T, D, 8>(grid, smem_bytes, stream, map, params);
    default: *supported = false; return cudaSuccess;
  }
}

template <typename T, int D>
cudaError_t launch_reduce_for_head_size(void* out, const float* part_o, const float* part_lse,
                                        const int32_t* seq_lens, const int32_t* counts,
                                        int group, int num_seqs, int num_heads,
                                        int partition_tokens, int max_parts,
                                        cudaStream_t stream) {
  if (max_parts <= kReduceRowParts) {
    // Few partitions: a warp per row, eight rows per CTA.
    const long long rows = (long long)num_seqs * num_heads;
    void* rargs[] = {&out, &part_o, &part_lse, &seq_lens, &counts, &group, &num_seqs, &num_heads,
                     &partition_tokens, &max_parts};
    return launch_overlapped((const void*)lse_reduce_rows_kernel<T, D>,
                             dim3((unsigned)((rows + 7) / 8)), dim3(256), 0, stream, rargs);
  }
  // Rows of many partitions are shared by several CTAs (32 columns each).
  int cols = max_parts >= 128 ? kReduceMinCols : D;
  dim3 grid((unsigned)num_heads, (unsigned)num_seqs, (unsigned)(D / cols));
  void* args[] = {&out,   &part_o,    &part_lse,         &seq_lens,  &counts, &group,
                  &num_heads, &partition_tokens, &max_parts, &cols};
  return launch_overlapped((const void*)lse_reduce_kernel<T, D>, grid, dim3(kReduceThreads), 0,
                           stream, args);
}

}  // namespace pa

#define PA_DEFINE_DECODE_UNIT(TYPE, TAG, D)                                                    \
  namespace pa {                                                                               \
  cudaError_t launch_decode_##TAG##_d##D(int group, dim3 grid, int smem_bytes,                 \
                                         cudaStream_t stream, const CUtensorMap& map,          \
                                         const DecodeParams& params, bool* supported) {        \
    return launch_decode_for_head_size<TYPE, D>(group, grid, smem_bytes, stream, map, params, \
                                                supported);                                    \
  }                                                                                            \
  cudaError_t launch_reduce_##TAG##_d##D(void* out, const float* part_o,                       \
                                         const float* part_lse, const int32_t* seq_lens,       \
                                         const int32_t* counts, int group, int num_seqs,       \
                                         int num_heads, int partition_tokens, int max_parts,   \
                                         cudaStream_t stream) {                                \
    return launch_reduce_for_head_size<TYPE, D>(out, part_o, part_lse, seq_lens, counts,       \
                                                group, num_seqs, num_heads, partition_tokens,  \
                                                max_parts, stream);                            \
  }                                                                                            \
  }
