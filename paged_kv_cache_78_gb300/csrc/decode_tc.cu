// Tensor-core (tcgen05) decode kernels: bf16, head sizes 64 and 128, query
// groups up to 16; a persistent grid sized by occupancy.  The kernels live
// in one translation unit per (head size, timeline on or off).
#include "decode_tc_kernel.cuh"
#include "pa_launch.h"

namespace pa {

#define PA_DECLARE_TC_UNIT(NAME)                                                       \
  cudaError_t NAME(int, int, cudaStream_t, const CUtensorMap&, const CUtensorMap&, \
                   const DecodeParams&);
PA_DECLARE_TC_UNIT(launch_tc_d64)
PA_DECLARE_TC_UNIT(launch_tc_d64_trace)
PA_DECLARE_TC_UNIT(launch_tc_d128)
PA_DECLARE_TC_UNIT(launch_tc_d128_trace)
#undef PA_DECLARE_TC_UNIT

cudaError_t launch_decode_tc(int head_size, int num_sms, int smem_bytes, cudaStream_t stream,
                             const CUtensorMap& kv_map, const CUtensorMap& q_map,
                             const DecodeParams& params, bool* supported) {
  *supported = true;
  const DecodeParams& prm = params;
  const bool trace = prm.trace != nullptr;  // the timeline kernels run only while one is set
  switch (head_size) {
    case 64:
      return trace ? launch_tc_d64_trace(num_sms, smem_bytes, stream, kv_map, q_map, prm)
                   : launch_tc_d64(num_sms, smem_bytes, stream, kv_map, q_map, prm);
    case 128:
      return trace ? launch_tc_d128_trace(num_sms, smem_bytes, stream, kv_map, q_map, prm)
                   : launch_tc_d128(num_sms, smem_bytes, stream, kv_map, q_map, prm);
    default: *supported = false; return cudaSuccess;
  }
}

}  // namespace pa
