// pa_decode_no_alloc: paged decode whose split-KV scratch lives in a
// workspace the library owns, for callers that cannot allocate device memory.
//
// Who needs it: an engine that reserves all device memory for its block pool
// at start-up and forbids any later allocation, and plain C callers without a
// caching allocator, for whom a cudaMalloc/cudaFree around every decode step
// would synchronise the device.  The caller still passes every input and the
// output; only the partials of split-KV go to the library's array.
#include <cuda_runtime.h>

#include <mutex>

#include "pa.h"

namespace {

// The scratch array: every device that loads the library holds it until the
// process exits.  In host code this name is only a stand-in for the device
// variable; its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_no_alloc_workspace[PA_NO_ALLOC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_lock;
void* g_workspace_addr[kMaxDevices] = {};

// Device address of the array on the current device, looked up once per
// device (the first call on each device does this lookup).
pa_status workspace_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PA_ERR_CUDA;
  std::lock_guard<std::mutex> guard(g_lock);
  if (!g_workspace_addr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_no_alloc_workspace) != cudaSuccess || !ptr)
      return PA_ERR_CUDA;
    g_workspace_addr[dev] = ptr;
  }
  *out = g_workspace_addr[dev];
  return PA_OK;
}

}  // namespace

extern "C" pa_status pa_decode_no_alloc(void* out, const void* query, const void* cache,
                                        const pa_cache_desc* desc, const int32_t* block_tables,
                                        int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                        int32_t num_seqs, int32_t num_heads, float scale,
                                        int32_t max_seq_len, int32_t partition_size,
                                        void* stream) {
  size_t need = 0;
  pa_status st = pa_decode_workspace_size(desc, num_seqs, num_heads, max_seq_len, partition_size,
                                          &need);
  if (st != PA_OK) return st;
  if (need > (size_t)PA_NO_ALLOC_WORKSPACE_BYTES) return PA_ERR_INVALID_ARG;
  // Every call passes the array: even without a split, the tensor-core
  // kernel keeps its work counters in the array's first 256 bytes.
  void* ws = nullptr;
  if ((st = workspace_address(&ws)) != PA_OK) return st;
  // Those 256 bytes must be zero before a call: static storage starts at
  // zero and every call leaves them zero.  The partials after them need no
  // initialisation; under the balanced split the piece counts are written
  // for every (sequence, KV head) pair before the reduce reads them.
  return pa_decode(out, query, cache, desc, block_tables, max_blocks_per_seq, seq_lens, num_seqs,
                   num_heads, scale, max_seq_len, partition_size, ws,
                   (size_t)PA_NO_ALLOC_WORKSPACE_BYTES, stream);
}
