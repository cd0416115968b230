// Host-side launchers shared by the C-ABI translation unit and the kernel
// translation units of the library.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pa {

struct DecodeParams;

// Launch `kernel` with programmatic stream serialization: it may begin (and
// run the part before its grid_dependency_wait) while the previous kernel on
// the stream finishes.  `args` points at the kernel's arguments, in order.
inline cudaError_t launch_overlapped(const void* kernel, dim3 grid, dim3 block, size_t smem,
                                     cudaStream_t stream, void** args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, kernel, args);
}

cudaError_t launch_reshape_and_cache(void* cache, const void* key, const void* value,
                                     const int64_t* slot_mapping, int64_t num_tokens,
                                     int64_t num_slots, int row_bytes, int64_t plane_bytes,
                                     unsigned int* err, cudaStream_t stream);

// Block copies from src_cache to dst_cache (the same pool for copy-on-write).
cudaError_t launch_copy_blocks(void* dst_cache, const void* src_cache, const int64_t* pairs,
                               int num_pairs, int64_t dst_blocks, int64_t src_blocks,
                               int64_t block_bytes, unsigned int* err, cudaStream_t stream);

// Byte copy by a kernel (device or page-locked host memory on either side).
cudaError_t launch_copy_bytes(void* dst, const void* src, int64_t bytes, int num_sms,
                              cudaStream_t stream);

// Decode launchers, one per element type.  `supported` is set to false (and
// nothing launched) when no kernel exists for (head_size, group).
cudaError_t launch_decode_bf16(int head_size, int group, dim3 grid, int smem_bytes,
                               cudaStream_t stream, const CUtensorMap& map,
                               const DecodeParams& params, bool* supported);
cudaError_t launch_decode_f32(int head_size, int group, dim3 grid, int smem_bytes,
                              cudaStream_t stream, const CUtensorMap& map,
                              const DecodeParams& params, bool* supported);

// Tensor-core decode (bf16, head size 64 or 128, group <= 16).
cudaError_t launch_decode_tc(int head_size, int num_sms, int smem_bytes, cudaStream_t stream,
                             const CUtensorMap& kv_map, const CUtensorMap& q_map,
                             const DecodeParams& params, bool* supported);

// Shared-prefix decode (bf16, head size 64 or 128): grid = (stage ranges,
// KV heads, chunks).  shared_stage_slots / shared_smem_bytes give its stage
// ring and dynamic shared memory.
struct SharedParams;
int shared_stage_slots(int head_size);
int shared_smem_bytes(int head_size);
cudaError_t launch_decode_shared(int head_size, dim3 grid, int smem_bytes, cudaStream_t stream,
                                 const CUtensorMap& kv_map, const SharedParams& params,
                                 bool* supported);

// Log-sum-exp reduce of split-KV partials.  A row's partial count comes from
// counts[row / group] when counts is given (balanced split), else from its
// sequence length and partition_tokens.
cudaError_t launch_lse_reduce(int dtype, int head_size, void* out, const float* part_o,
                              const float* part_lse, const int32_t* seq_lens,
                              const int32_t* counts, int group, int num_seqs, int num_heads,
                              int partition_tokens, int max_parts, cudaStream_t stream,
                              bool* supported);

}  // namespace pa
