// Tensor-core (tcgen05) decode kernels: bf16, head sizes 64 and 128, query
// groups up to 16.
#include <atomic>

#include "decode_tc_kernel.cuh"
#include "pa_launch.h"

namespace pa {

template <int D>
static cudaError_t launch_tc(dim3 grid, int smem_bytes, cudaStream_t stream,
                             const CUtensorMap& map, const DecodeParams& params) {
  static std::atomic<int> configured[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (smem_bytes > configured[dev].load(std::memory_order_relaxed)) {
    e = cudaFuncSetAttribute(paged_decode_tc_kernel<D>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e != cudaSuccess) return e;
    configured[dev].store(smem_bytes, std::memory_order_relaxed);
  }
  paged_decode_tc_kernel<D><<<grid, kTcThreads, smem_bytes, stream>>>(map, params);
  return cudaGetLastError();
}

cudaError_t launch_decode_tc(int head_size, dim3 grid, int smem_bytes, cudaStream_t stream,
                             const CUtensorMap& map, const DecodeParams& params,
                             bool* supported) {
  *supported = true;
  switch (head_size) {
    case 64: return launch_tc<64>(grid, smem_bytes, stream, map, params);
    case 128: return launch_tc<128>(grid, smem_bytes, stream, map, params);
    default: *supported = false; return cudaSuccess;
  }
}

}  // namespace pa
