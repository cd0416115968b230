// Dispatch of decode and reduce launches by element type and head size.
#include "decode_kernel.cuh"
#include "pa_launch.h"

namespace pa {

#define PA_DECLARE_UNIT(TAG, D)                                                              \
  cudaError_t launch_decode_##TAG##_d##D(int, dim3, int, cudaStream_t, const CUtensorMap&,   \
                                         const DecodeParams&, bool*);                        \
  cudaError_t launch_reduce_##TAG##_d##D(void*, const float*, const float*, const int32_t*,  \
                                         const int32_t*, int, int, int, int, int, cudaStream_t);
PA_DECLARE_UNIT(bf16, 64)
PA_DECLARE_UNIT(bf16, 128)
PA_DECLARE_UNIT(bf16, 256)
PA_DECLARE_UNIT(f32, 64)
PA_DECLARE_UNIT(f32, 128)
PA_DECLARE_UNIT(f32, 256)
#undef PA_DECLARE_UNIT

cudaError_t launch_decode_bf16(int head_size, int group, dim3 grid, int smem_bytes,
                               cudaStream_t stream, const CUtensorMap& map,
                               const DecodeParams& params, bool* supported) {
  switch (head_size) {
    case 64: return launch_decode_bf16_d64(group, grid, smem_bytes, stream, map, params, supported);
    case 128: return launch_decode_bf16_d128(group, grid, smem_bytes, stream, map, params, supported);
    case 256: return launch_decode_bf16_d256(group, grid, smem_bytes, stream, map, params, supported);
    default: *supported = false; return cudaSuccess;
  }
}

cudaError_t launch_decode_f32(int head_size, int group, dim3 grid, int smem_bytes,
                              cudaStream_t stream, const CUtensorMap& map,
                              const DecodeParams& params, bool* supported) {
  switch (head_size) {
    case 64: return launch_decode_f32_d64(group, grid, smem_bytes, stream, map, params, supported);
    case 128: return launch_decode_f32_d128(group, grid, smem_bytes, stream, map, params, supported);
    case 256: return launch_decode_f32_d256(group, grid, smem_bytes, stream, map, params, supported);
    default: *supported = false; return cudaSuccess;
  }
}

cudaError_t launch_lse_reduce(int dtype, int head_size, void* out, const float* part_o,
                              const float* part_lse, const int32_t* seq_lens,
                              const int32_t* counts, int group, int num_seqs, int num_heads,
                              int partition_tokens, int max_parts, cudaStream_t stream,
                              bool* supported) {
  *supported = true;
#define PA_REDUCE_CASE(TAG, D)                                                                \
  case D:                                                                                     \
    return launch_reduce_##TAG##_d##D(out, part_o, part_lse, seq_lens, counts, group, num_seqs, \
                                      num_heads, partition_tokens, max_parts, stream);
  if (dtype == 0) {
    switch (head_size) { PA_REDUCE_CASE(bf16, 64) PA_REDUCE_CASE(bf16, 128) PA_REDUCE_CASE(bf16, 256) }
  } else {
    switch (head_size) { PA_REDUCE_CASE(f32, 64) PA_REDUCE_CASE(f32, 128) PA_REDUCE_CASE(f32, 256) }
  }
#undef PA_REDUCE_CASE
  *supported = false;
  return cudaSuccess;
}

}  // namespace pa
