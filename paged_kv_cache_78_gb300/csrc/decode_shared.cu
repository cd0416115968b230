// Shared-prefix decode kernels (head sizes 64 and 128) and their launcher.
#include <atomic>

#include "decode_shared_kernel.cuh"
#include "pa_launch.h"

namespace pa {

template <int D, bool kTrace>
static cudaError_t launch_shared(dim3 grid, int smem_bytes, cudaStream_t stream,
                                 const CUtensorMap& kv_map, const SharedParams& params) {
  static std::atomic<int> configured[64];
  auto kernel = paged_decode_shared_kernel<D, kTrace>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (smem_bytes > configured[dev].load(std::memory_order_relaxed)) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e != cudaSuccess) return e;
    configured[dev].store(smem_bytes, std::memory_order_relaxed);
  }
  SharedParams prm = params;
  const size_t ctas = (size_t)prm.trace_cta_base + (size_t)grid.x * grid.y * grid.z;
  if (kTrace && ctas * kTcTraceRoles * (size_t)prm.trace_per_role * 16 > prm.trace_bytes)
    prm.trace = nullptr;  // the buffer cannot hold this launch's timeline: record nothing
  void* args[] = {const_cast<CUtensorMap*>(&kv_map), &prm};
  return launch_overlapped((const void*)kernel, grid, dim3(kShThreads), (size_t)smem_bytes, stream,
                           args);
}

int shared_stage_slots(int head_size) { return head_size == 128 ? 3 : 5; }

int shared_smem_bytes(int head_size) {
  return sh_smem_layout(head_size, shared_stage_slots(head_size)).total;
}

cudaError_t launch_decode_shared(int head_size, dim3 grid, int smem_bytes, cudaStream_t stream,
                                 const CUtensorMap& kv_map, const SharedParams& params,
                                 bool* supported) {
  *supported = true;
  const bool trace = params.trace != nullptr;  // the timeline variant runs only while one is set
  switch (head_size) {
    case 64:
      return trace ? launch_shared<64, true>(grid, smem_bytes, stream, kv_map, params)
                   : launch_shared<64, false>(grid, smem_bytes, stream, kv_map, params);
    case 128:
      return trace ? launch_shared<128, true>(grid, smem_bytes, stream, kv_map, params)
                   : launch_shared<128, false>(grid, smem_bytes, stream, kv_map, params);
    default: *supported = false; return cudaSuccess;
  }
}

}  // namespace pa
