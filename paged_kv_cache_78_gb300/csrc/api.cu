// C ABI of the library: argument checks, TMA descriptor encoding, launch
// geometry and kernel dispatch.  See include/pa.h for the contract.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "decode_kernel.cuh"
#include "decode_shared_kernel.cuh"
#include "decode_tc_kernel.cuh"
#include "pa.h"
#include "pa_launch.h"

// Per-device error word written by the kernels (PA_DEVERR_* bits); static
// storage, so it starts at zero on every device that loads the library.
__device__ unsigned int g_pa_error_word;

namespace {

constexpr int kMaxDevices = 64;
// Shared memory for the CUDA-core kernel's K/V stage ring.  Three or more
// stages in 48 KB leave room for four CTAs per SM, and four rings of three
// stages beat three rings of four (the same bytes in flight, more independent
// pipelines; OPT-13B shape 104.5 -> 102.3 us); rows too wide for that get the
// wider ring.
constexpr int kStageBudgetBytes = 48 * 1024;
constexpr int kStageBudgetWideBytes = 96 * 1024;
constexpr int kMaxSmemPerCta = 227 * 1024;
// Block copies launch two CTAs per pair along grid x, whose limit is 2^31 - 1.
constexpr int32_t kMaxCopyPairs = (1 << 30) - 1;

std::mutex g_mutex;
unsigned int* g_error_word[kMaxDevices] = {};
int g_num_sms[kMaxDevices] = {};

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

// Timeline buffer of the tensor-core decode (pa_set_decode_trace).
std::atomic<void*> g_trace_buf{nullptr};
std::atomic<size_t> g_trace_bytes{0};
std::atomic<int> g_trace_per_role{0};

// Limit of the tensor-core decode's pipeline waits (pa_set_decode_wait_limit);
// 0 = the default, kWaitLimitCycles.
std::atomic<long long> g_wait_limit{0};

bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }
int ilog2(int x) {
  int r = 0;
  while ((1 << r) < x) ++r;
  return r;
}
int elem_bytes(int dtype) { return dtype == PA_BF16 ? 2 : 4; }
bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

pa_status cuda_status(cudaError_t e) { return e == cudaSuccess ? PA_OK : PA_ERR_CUDA; }

// Device-side state of the current device: the error word's address and the SM count.
pa_status device_state(unsigned int** err, int* num_sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_error_word[dev]) {
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_pa_error_word) != cudaSuccess) return PA_ERR_CUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return PA_ERR_CUDA;
    g_num_sms[dev] = sms;
    g_error_word[dev] = static_cast<unsigned int*>(addr);
  }
  if (err) *err = g_error_word[dev];
  if (num_sms) *num_sms = g_num_sms[dev];
  return PA_OK;
}

pa_status encode_fn(EncodeTiledFn* fn) {
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_encode) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !p)
      return PA_ERR_CUDA;
    g_encode = reinterpret_cast<EncodeTiledFn>(p);
  }
  *fn = g_encode;
  return PA_OK;
}

pa_status check_desc(const pa_cache_desc* d) {
  if (!d) return PA_ERR_INVALID_ARG;
  if (d->num_blocks < 1 || d->num_kv_heads < 1 || d->head_size < 1) return PA_ERR_INVALID_ARG;
  if (!is_pow2(d->block_size) || d->block_size > 256) return PA_ERR_INVALID_ARG;
  if (d->dtype != PA_BF16 && d->dtype != PA_FP32) return PA_ERR_INVALID_ARG;
  if ((d->head_size * elem_bytes(d->dtype)) % 16 != 0) return PA_ERR_INVALID_ARG;
  return PA_OK;
}

bool head_size_supported(int d) { return d == 64 || d == 128 || d == 256; }

// Partition policy.  An explicit size is checked.  -1 on the CUDA-core
// kernel picks the largest of 512, 256, 128, 64 tokens (not below the block
// size) that still gives six CTAs per SM; on the tensor-core kernel it picks
// no split when (sequence, KV head) pairs alone fill the grid, else the
// balanced split (1024-token partitions and down for batches of more than
// 256 sequences).  A size that covers max_seq_len means no split (0).
pa_status select_kernel(const pa_cache_desc* desc, int32_t num_seqs, int32_t num_heads,
                        const void* query, int32_t kernel, int32_t* selected);

// The automatic partition size depends only on the shapes and on the kernel
// family PA_KERNEL_AUTO picks for a 16-byte aligned query, so the size
// queries and the decode call always agree.
// Stage ranges of the balanced split: one per resident CTA of the
// tensor-core kernel (two per SM for head size 64, one for 128).
int balanced_ranges(const pa_cache_desc* d, int num_sms) {
  return num_sms * (d->head_size == 64 ? 2 : 1);
}

// Partials per row of the balanced split.  A pair of n stages meets at most
// ceil((n - 1) / Q) + 1 ranges of Q stages; every sequence has num_kv_heads
// pairs, so n <= Q * ranges / num_kv_heads, and n <= ceil(max_seq_len / 128).
int balanced_max_parts(const pa_cache_desc* d, int max_seq_len, int num_sms) {
  const long long by_len = ((long long)max_seq_len + pa::kTcTokens - 1) / pa::kTcTokens;
  const long long by_ranges =
      ((long long)balanced_ranges(d, num_sms) + d->num_kv_heads - 1) / d->num_kv_heads + 1;
  const long long m = by_len < by_ranges ? by_len : by_ranges;
  return m < 1 ? 1 : (int)m;
}

pa_status resolve_partition(const pa_cache_desc* d, int num_seqs, int num_heads, int max_seq_len,
                            int requested, int num_sms, int* out) {
  int p = requested;
  if (p == PA_PARTITION_BALANCED) {
    // The balanced split runs on the tensor-core kernel, for batches whose
    // lengths it keeps in shared memory; elsewhere the automatic rule.
    int32_t family = PA_KERNEL_SIMT;
    if (select_kernel(d, num_seqs, num_heads, reinterpret_cast<const void*>(256), PA_KERNEL_AUTO,
                      &family) != PA_OK)
      family = PA_KERNEL_SIMT;
    if (family == PA_KERNEL_TENSOR && num_seqs <= pa::kTcLensCache) {
      *out = PA_PARTITION_BALANCED;
      return PA_OK;
    }
    p = -1;
  }
  if (p == -1) {
    const long long heads = (long long)num_seqs * d->num_kv_heads;
    int32_t family = PA_KERNEL_SIMT;
    if (select_kernel(d, num_seqs, num_heads, reinterpret_cast<const void*>(256), PA_KERNEL_AUTO,
                      &family) != PA_OK)
      family = PA_KERNEL_SIMT;
    if (family == PA_KERNEL_TENSOR) {
      // Persistent tensor-core kernel: each work item pays a fixed cost to
      // start and finish, so items are long (1024 tokens) unless that leaves
      // fewer items than half the resident CTAs (two per SM for head size 64,
      // one for 128).
      const long long ctas = (long long)num_sms * (d->head_size == 64 ? 2 : 1);
      p = 1024;
      while (p > 128 && p > d->block_size && 2 * heads * ((max_seq_len + p - 1) / p) < ctas)
        p >>= 1;
      // Enough (sequence, KV head) pairs for four items per resident CTA,
      // and no sequence long enough to leave one CTA a long tail: no split
      // (no partials, no reduce, no short tail partitions).
      if (heads >= 4 * ctas && max_seq_len <= 4096) p = 0;
      // Where that splits, the balanced split instead (batches whose lengths
      // the kernel keeps in shared memory): every CTA gets the same number of
      // stages, so no long item leaves a tail.
      if (p > 0 && p < max_seq_len && num_seqs <= pa::kTcLensCache) {
        *out = PA_PARTITION_BALANCED;
        return PA_OK;
      }
    } else {
      // One CTA per (partition, KV head, sequence): enough CTAs for six per SM.
      p = 512;
      while (p > 64 && p > d->block_size && heads * ((max_seq_len + p - 1) / p) < 6LL * num_sms)
        p >>= 1;
      // Batches the kernel takes longest first, with (sequence, KV head)
      // pairs for four CTAs per SM and no sequence past 2048 tokens: no
      // split.  The long sequences start first and the short ones fill the
      // tail, with no partials and no reduce.
      if (num_seqs <= pa::kLongestFirstMaxSeqs && heads >= 4LL * num_sms && max_seq_len <= 2048)
        p = 0;
    }
    if (p > 0 && p < d->block_size) p = d->block_size;
  } else if (p < PA_PARTITION_BALANCED) {
    return PA_ERR_INVALID_ARG;
  } else if (p > 0 && p % d->block_size != 0) {
    return PA_ERR_INVALID_ARG;
  }
  if (p > 0 && max_seq_len <= p) p = 0;
  *out = p;
  return PA_OK;
}

// Workspace: a 256-byte header (the tensor-core kernel's work counter), then,
// when splitting, the fp32 partial outputs and their log-sum-exp values.
constexpr size_t kWorkspaceHeader = 256;

size_t partial_o_bytes(int num_seqs, int num_heads, int head_size, int max_parts) {
  const size_t rows = (size_t)num_seqs * num_heads * max_parts;
  return (rows * head_size * 4 + 255) / 256 * 256;
}

// pairs: (sequence, KV head) pairs whose piece counts follow the partials
// (balanced split), else 0.
size_t workspace_bytes_for(int num_seqs, int num_heads, int head_size, int max_parts,
                           size_t pairs = 0) {
  if (max_parts == 0) return kWorkspaceHeader;
  const size_t rows = (size_t)num_seqs * num_heads * max_parts;
  return kWorkspaceHeader + partial_o_bytes(num_seqs, num_heads, head_size, max_parts) +
         (rows * 4 + 255) / 256 * 256 + (pairs * 4 + 255) / 256 * 256;
}

// The tensor-core kernels' map of the pool: one block's K and V rows, every
// 128-byte column group, in one box, laid out per 8-token chunk as
// [column group][K rows][V rows] (each 8 rows one 1024-byte swizzle atom).
// Dimensions, innermost first: 64 elements; token within an 8-token chunk;
// K or V; (KV head, column group); 8-token chunk of the plane
// (block * block_size / 8 + chunk within the block).  R = rows of a box.
CUresult encode_tc_kv_map(EncodeTiledFn encode, const pa_cache_desc* desc, const void* cache,
                          int R, CUtensorMap* map) {
  const int D = desc->head_size;
  const int BS = desc->block_size;
  const cuuint64_t row = (cuuint64_t)desc->num_kv_heads * D * 2;
  const cuuint64_t tdim[5] = {64ull, 8ull, 2ull, (cuuint64_t)desc->num_kv_heads * (D / 64),
                              (cuuint64_t)desc->num_blocks * (cuuint64_t)(BS / 8)};
  const cuuint64_t tstride[4] = {row, (cuuint64_t)desc->num_blocks * BS * row, 128ull, 8 * row};
  const cuuint32_t tbox[5] = {64u, 8u, 2u, (cuuint32_t)(D / 64), (cuuint32_t)(R / 8)};
  const cuuint32_t estride[5] = {1u, 1u, 1u, 1u, 1u};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(cache), tdim, tstride,
                tbox, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

// The tensor-core decode next to a shared-prefix decode's group kernel: it
// skips the groups' members (seq_start > 0) and decodes the other sequences
// (the balanced split for batches of up to 256 sequences), recording their
// partial counts next to the members' in the same array.
struct CascadeArgs {
  const int32_t* seq_start;
  int32_t* counts;
  float* part_o;
  float* part_lse;
  int max_parts;
};

// Stage ranges per (chunk, KV head) of the group kernel: enough CTAs to fill
// the SMs, no more ranges than the shortest chunk has stages, at most 16 (the
// reduce then takes rows of up to 16 partials).
int shared_ranges(const pa_cache_desc* d, const pa_shared_plan_info* info, int num_sms) {
  const long long units = (long long)info->num_chunks * d->num_kv_heads;
  long long r = units > 0 ? num_sms / units : 1;
  if (r > info->min_chunk_stages) r = info->min_chunk_stages;
  if (r > 16) r = 16;
  return r < 1 ? 1 : (int)r;
}

// Partials per row of a shared-prefix decode: the group kernel's ranges for
// member rows, the balanced split's pieces for the others.
int shared_max_parts(const pa_cache_desc* d, const pa_shared_plan_info* info, int num_seqs,
                     int max_seq_len, int num_sms) {
  const int r = shared_ranges(d, info, num_sms);
  const int others = info->num_members < num_seqs && num_seqs <= pa::kTcLensCache
                         ? balanced_max_parts(d, max_seq_len, num_sms)
                         : 1;
  return r > others ? r : others;
}

// Workspace of pa_decode_shared: the 256-byte header, fp32 partials and
// log-sum-exp values of max_parts per row, then a partial count per pair.
size_t shared_workspace_bytes(int num_seqs, int num_heads, int num_kv_heads, int head_size,
                              int max_parts) {
  const size_t rows = (size_t)num_seqs * num_heads * max_parts;
  const size_t pairs = (size_t)num_seqs * num_kv_heads;
  return 256 + (rows * head_size * 4 + 255) / 256 * 256 + (rows * 4 + 255) / 256 * 256 +
         (pairs * 4 + 255) / 256 * 256;
}

// The kernel family for a decode call (desc already checked).
pa_status select_kernel(const pa_cache_desc* desc, int32_t num_seqs, int32_t num_heads,
                        const void* query, int32_t kernel, int32_t* selected) {
  const int group = num_heads / desc->num_kv_heads;
  const int D = desc->head_size;
  if (!head_size_supported(D) || desc->num_kv_heads > 65535) return PA_ERR_UNSUPPORTED;
  // Tensor cores: bf16, head size 64 or 128, query group up to 16, blocks of
  // at least 8 tokens (a TMA box then fills whole 1024-byte swizzle atoms).
  const bool tc_ok = desc->dtype == PA_BF16 && (D == 64 || D == 128) && group <= pa::kTcHeads &&
                     desc->block_size >= 8 && aligned(query, 16) &&
                     (long long)num_seqs * num_heads < (1ll << 31) &&
                     (long long)desc->num_blocks * (desc->block_size / 8) < (1ll << 31);
  bool use_tc;
  if (kernel == PA_KERNEL_TENSOR) {
    if (!tc_ok) return PA_ERR_UNSUPPORTED;
    use_tc = true;
  } else if (kernel == PA_KERNEL_SIMT) {
    use_tc = false;
  } else {
    // Automatic choice: the tensor-core kernel for grouped queries (G >= 2),
    // whose CUDA-core cost grows with G; the CUDA-core kernel for G = 1,
    // where it measures faster.
    use_tc = tc_ok && group >= 2;
  }
  if (!use_tc && group > 8) return PA_ERR_UNSUPPORTED;
  *selected = use_tc ? PA_KERNEL_TENSOR : PA_KERNEL_SIMT;
  return PA_OK;
}

}  // namespace

extern "C" {

const char* pa_version(void) { return "0.1.0"; }

pa_status pa_set_decode_trace(void* device_buffer, size_t bytes, int32_t events_per_role) {
  if (device_buffer && (events_per_role < 1 || bytes < 16 || !aligned(device_buffer, 8)))
    return PA_ERR_INVALID_ARG;
  g_trace_per_role.store(device_buffer ? events_per_role : 0);
  g_trace_bytes.store(device_buffer ? bytes : 0);
  g_trace_buf.store(device_buffer);
  return PA_OK;
}

pa_status pa_set_decode_wait_limit(int64_t cycles) {
  if (cycles < 0) return PA_ERR_INVALID_ARG;
  g_wait_limit.store(cycles);
  return PA_OK;
}

const char* pa_status_string(pa_status s) {
  switch (s) {
    case PA_OK: return "ok";
    case PA_ERR_INVALID_ARG: return "invalid argument";
    case PA_ERR_UNSUPPORTED: return "unsupported shape";
    case PA_ERR_CUDA: return "CUDA error";
    case PA_ERR_OUT_OF_BLOCKS: return "out of blocks";
    case PA_ERR_BAD_STATE: return "bad state";
    case PA_ERR_DEVICE_CHECK: return "device-side check failed";
    case PA_ERR_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

pa_status pa_get_device_error(uint32_t* flags, void* stream) {
  if (!flags) return PA_ERR_INVALID_ARG;
  unsigned int* err = nullptr;
  pa_status st = device_state(&err, nullptr);
  if (st != PA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned int v = 0;
  if (cudaStreamSynchronize(s) != cudaSuccess) return PA_ERR_CUDA;
  if (cudaMemcpy(&v, err, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return PA_ERR_CUDA;
  unsigned int zero = 0;
  if (cudaMemcpy(err, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
    return PA_ERR_CUDA;
  *flags = v;
  if (v & PA_DEVERR_TIMEOUT) return PA_ERR_TIMEOUT;
  return v ? PA_ERR_DEVICE_CHECK : PA_OK;
}

pa_status pa_reshape_and_cache(void* cache, const pa_cache_desc* desc, const void* key,
                               const void* value, const int64_t* slot_mapping,
                               int32_t num_tokens, void* stream) {
  pa_status st = check_desc(desc);
  if (st != PA_OK) return st;
  if (num_tokens < 0) return PA_ERR_INVALID_ARG;
  if (num_tokens == 0) return PA_OK;
  if (!cache || !key || !value || !slot_mapping) return PA_ERR_INVALID_ARG;
  if (!aligned(cache, 16) || !aligned(key, 16) || !aligned(value, 16) || !aligned(slot_mapping, 8))
    return PA_ERR_INVALID_ARG;
  unsigned int* err = nullptr;
  if ((st = device_state(&err, nullptr)) != PA_OK) return st;
  const int row_bytes = desc->num_kv_heads * desc->head_size * elem_bytes(desc->dtype);
  const int64_t num_slots = (int64_t)desc->num_blocks * desc->block_size;
  const int64_t plane_bytes = num_slots * row_bytes;
  return cuda_status(pa::launch_reshape_and_cache(cache, key, value, slot_mapping, num_tokens,
                                                  num_slots, row_bytes, plane_bytes, err,
                                                  static_cast<cudaStream_t>(stream)));
}

pa_status pa_copy_blocks(void* cache, const pa_cache_desc* desc, const int64_t* pairs,
                         int32_t num_pairs, void* stream) {
  pa_status st = check_desc(desc);
  if (st != PA_OK) return st;
  if (num_pairs < 0 || num_pairs > kMaxCopyPairs) return PA_ERR_INVALID_ARG;
  if (num_pairs == 0) return PA_OK;
  if (!cache || !pairs || !aligned(cache, 16) || !aligned(pairs, 8)) return PA_ERR_INVALID_ARG;
  unsigned int* err = nullptr;
  if ((st = device_state(&err, nullptr)) != PA_OK) return st;
  const int64_t block_bytes = (int64_t)desc->block_size * desc->num_kv_heads * desc->head_size *
                              elem_bytes(desc->dtype);
  return cuda_status(pa::launch_copy_blocks(cache, cache, pairs, num_pairs, desc->num_blocks,
                                            desc->num_blocks, block_bytes, err,
                                            static_cast<cudaStream_t>(stream)));
}

// The address a kernel uses for `p`: device memory as is, page-locked host
// memory through its device mapping; anything else (pageable host memory)
// is refused.
static pa_status kernel_address(const void* p, const void** out) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return PA_ERR_INVALID_ARG;
  }
  if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) {
    *out = p;
    return PA_OK;
  }
  if (a.type == cudaMemoryTypeHost && a.devicePointer != nullptr) {
    *out = a.devicePointer;
    return PA_OK;
  }
  return PA_ERR_INVALID_ARG;
}

pa_status pa_swap_blocks(void* dst_cache, const pa_cache_desc* dst_desc, const void* src_cache,
                         const pa_cache_desc* src_desc, const int64_t* pairs, int32_t num_pairs,
                         void* stream) {
  pa_status st = check_desc(dst_desc);
  if (st != PA_OK) return st;
  if ((st = check_desc(src_desc)) != PA_OK) return st;
  if (dst_desc->block_size != src_desc->block_size ||
      dst_desc->num_kv_heads != src_desc->num_kv_heads ||
      dst_desc->head_size != src_desc->head_size || dst_desc->dtype != src_desc->dtype)
    return PA_ERR_INVALID_ARG;
  if (num_pairs < 0 || num_pairs > kMaxCopyPairs) return PA_ERR_INVALID_ARG;
  if (num_pairs == 0) return PA_OK;
  if (!dst_cache || !src_cache || !pairs || !aligned(dst_cache, 16) || !aligned(src_cache, 16) ||
      !aligned(pairs, 8))
    return PA_ERR_INVALID_ARG;
  const void* d = nullptr;
  const void* s = nullptr;
  const void* pr = nullptr;
  if ((st = kernel_address(dst_cache, &d)) != PA_OK) return st;
  if ((st = kernel_address(src_cache, &s)) != PA_OK) return st;
  if ((st = kernel_address(pairs, &pr)) != PA_OK) return st;
  unsigned int* err = nullptr;
  if ((st = device_state(&err, nullptr)) != PA_OK) return st;
  const int64_t block_bytes = (int64_t)dst_desc->block_size * dst_desc->num_kv_heads *
                              dst_desc->head_size * elem_bytes(dst_desc->dtype);
  return cuda_status(pa::launch_copy_blocks(const_cast<void*>(d), s,
                                            static_cast<const int64_t*>(pr), num_pairs,
                                            dst_desc->num_blocks, src_desc->num_blocks,
                                            block_bytes, err, static_cast<cudaStream_t>(stream)));
}

pa_status pa_copy_bytes(void* dst, const void* src, size_t bytes, void* stream) {
  if (bytes == 0) return PA_OK;
  if (!dst || !src || bytes > ((size_t)1 << 40)) return PA_ERR_INVALID_ARG;
  const void* d = nullptr;
  const void* s = nullptr;
  pa_status st = kernel_address(dst, &d);
  if (st != PA_OK) return st;
  if ((st = kernel_address(src, &s)) != PA_OK) return st;
  const uintptr_t d0 = reinterpret_cast<uintptr_t>(d), s0 = reinterpret_cast<uintptr_t>(s);
  if (d0 < s0 + bytes && s0 < d0 + bytes) return PA_ERR_INVALID_ARG;  // overlapping ranges
  int sms = 0;
  if ((st = device_state(nullptr, &sms)) != PA_OK) return st;
  return cuda_status(pa::launch_copy_bytes(const_cast<void*>(d), s, (int64_t)bytes, sms,
                                           static_cast<cudaStream_t>(stream)));
}

pa_status pa_decode_partition_size(const pa_cache_desc* desc, int32_t num_seqs,
                                   int32_t num_heads, int32_t max_seq_len,
                                   int32_t partition_size, int32_t* resolved) {
  pa_status st = check_desc(desc);
  if (st != PA_OK) return st;
  if (!resolved || num_seqs < 0 || max_seq_len < 0 || num_heads < 1 ||
      num_heads % desc->num_kv_heads != 0)
    return PA_ERR_INVALID_ARG;
  int sms = 0;
  if (partition_size < 0 && (st = device_state(nullptr, &sms)) != PA_OK) return st;
  int p = 0;
  if ((st = resolve_partition(desc, num_seqs, num_heads, max_seq_len, partition_size, sms, &p)) !=
      PA_OK)
    return st;
  *resolved = p;
  return PA_OK;
}

pa_status pa_decode_workspace_size(const pa_cache_desc* desc, int32_t num_seqs,
                                   int32_t num_heads, int32_t max_seq_len,
                                   int32_t partition_size, size_t* bytes) {
  if (!bytes) return PA_ERR_INVALID_ARG;
  int32_t p = 0;
  pa_status st = pa_decode_partition_size(desc, num_seqs, num_heads, max_seq_len,
                                          partition_size, &p);
  if (st != PA_OK) return st;
  if (p == PA_PARTITION_BALANCED) {
    int sms = 0;
    if ((st = device_state(nullptr, &sms)) != PA_OK) return st;
    *bytes = workspace_bytes_for(num_seqs, num_heads, desc->head_size,
                                 balanced_max_parts(desc, max_seq_len, sms),
                                 (size_t)num_seqs * desc->num_kv_heads);
    return PA_OK;
  }
  *bytes = workspace_bytes_for(num_seqs, num_heads, desc->head_size,
                               p == 0 ? 0 : (max_seq_len + p - 1) / p);
  return PA_OK;
}

pa_status pa_decode_select_kernel(const pa_cache_desc* desc, int32_t num_seqs, int32_t num_heads,
                                  const void* query, int32_t kernel, int32_t* selected) {
  pa_status st = check_desc(desc);
  if (st != PA_OK) return st;
  if (!selected || num_seqs < 0 || num_heads < 1 || num_heads % desc->num_kv_heads != 0)
    return PA_ERR_INVALID_ARG;
  if (kernel != PA_KERNEL_AUTO && kernel != PA_KERNEL_SIMT && kernel != PA_KERNEL_TENSOR)
    return PA_ERR_INVALID_ARG;
  return select_kernel(desc, num_seqs, num_heads, query, kernel, selected);
}

pa_status pa_decode(void* out, const void* query, const void* cache, const pa_cache_desc* desc,
                    const int32_t* block_tables, int32_t max_blocks_per_seq,
                    const int32_t* seq_lens, int32_t num_seqs, int32_t num_heads, float scale,
                    int32_t max_seq_len, int32_t partition_size, void* workspace,
                    size_t workspace_bytes, void* stream) {
  return pa_decode_ex(out, query, cache, desc, block_tables, max_blocks_per_seq, seq_lens,
                      num_seqs, num_heads, scale, max_seq_len, partition_size, workspace,
                      workspace_bytes, PA_KERNEL_AUTO, stream);
}

// pa_decode_ex, with the step's newest tokens written into the cache first
// when new_k / new_v are given (pa_decode_append).
static pa_status decode_impl(void* out, const void* query, const void* cache,
                             const pa_cache_desc* desc, const int32_t* block_tables,
                             int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t num_seqs,
                             int32_t num_heads, float scale, int32_t max_seq_len,
                             int32_t partition_size, void* workspace, size_t workspace_bytes,
                             int32_t kernel, const void* new_k, const void* new_v, void* stream,
                             const CascadeArgs* cas = nullptr) {
  pa_status st = check_desc(desc);
  if (st != PA_OK) return st;
  if (num_seqs < 0 || num_seqs > 65535 || num_heads < 1 || max_seq_len < 0 ||
      max_blocks_per_seq < 1 || !std::isfinite(scale))
    return PA_ERR_INVALID_ARG;
  if (kernel != PA_KERNEL_AUTO && kernel != PA_KERNEL_SIMT && kernel != PA_KERNEL_TENSOR)
    return PA_ERR_INVALID_ARG;
  if (num_heads % desc->num_kv_heads != 0) return PA_ERR_INVALID_ARG;
  if (num_seqs == 0) return PA_OK;
  if (!out || !query || !cache || !block_tables || !seq_lens) return PA_ERR_INVALID_ARG;
  const int es = elem_bytes(desc->dtype);
  if (!aligned(cache, 16) || !aligned(query, es) || !aligned(out, es) ||
      !aligned(block_tables, 4) || !aligned(seq_lens, 4))
    return PA_ERR_INVALID_ARG;
  const int group = num_heads / desc->num_kv_heads;
  const int D = desc->head_size;
  const int BS = desc->block_size;
  int32_t family = 0;
  if ((st = select_kernel(desc, num_seqs, num_heads, query, kernel, &family)) != PA_OK) return st;
  const bool use_tc = family == PA_KERNEL_TENSOR;

  unsigned int* err = nullptr;
  int sms = 0;
  if ((st = device_state(&err, &sms)) != PA_OK) return st;
  int part = 0;
  if ((st = resolve_partition(desc, num_seqs, num_heads, max_seq_len, partition_size, sms,
                              &part)) != PA_OK)
    return st;
  if (cas) {
    if (!use_tc) return PA_ERR_UNSUPPORTED;
    part = num_seqs <= pa::kTcLensCache ? PA_PARTITION_BALANCED : 0;
  }
  bool balanced = part == PA_PARTITION_BALANCED;
  if (balanced && !use_tc) {
    // The CUDA-core kernel (a query the tensor-core kernel cannot load, or
    // an explicit family) splits into equal partitions instead, no more of
    // them than the balanced split's partials, so its workspace suffices.
    const int mp = balanced_max_parts(desc, max_seq_len, sms);
    part = (max_seq_len + mp - 1) / mp;
    part = (part + BS - 1) / BS * BS;
    if (part >= max_seq_len) part = 0;
    balanced = false;
  }
  const int max_parts = cas        ? cas->max_parts
                        : balanced ? balanced_max_parts(desc, max_seq_len, sms)
                        : part > 0 ? (max_seq_len + part - 1) / part
                                   : 1;
  const size_t pairs = balanced ? (size_t)num_seqs * desc->num_kv_heads : 0;
  float* part_o = nullptr;
  float* part_lse = nullptr;
  int32_t* part_counts = nullptr;
  unsigned int* sched = nullptr;
  if (cas) {
    // pa_decode_shared checked the workspace and laid out its parts.
    sched = static_cast<unsigned int*>(workspace);
    part_o = cas->part_o;
    part_lse = cas->part_lse;
    part_counts = cas->counts;
  } else if (part > 0 || balanced || use_tc) {
    const size_t need =
        workspace_bytes_for(num_seqs, num_heads, D, part > 0 || balanced ? max_parts : 0, pairs);
    if (!workspace || workspace_bytes < need || !aligned(workspace, 256))
      return PA_ERR_INVALID_ARG;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    sched = reinterpret_cast<unsigned int*>(ws);
    if (part > 0 || balanced) {
      const size_t o_bytes = partial_o_bytes(num_seqs, num_heads, D, max_parts);
      const size_t rows = (size_t)num_seqs * num_heads * max_parts;
      part_o = reinterpret_cast<float*>(ws + kWorkspaceHeader);
      part_lse = reinterpret_cast<float*>(ws + kWorkspaceHeader + o_bytes);
      if (balanced)
        part_counts = reinterpret_cast<int32_t*>(ws + kWorkspaceHeader + o_bytes +
                                                 (rows * 4 + 255) / 256 * 256);
    }
  }

  pa::DecodeParams prm;
  std::memset(&prm, 0, sizeof(prm));
  int R, smem;
  if (use_tc) {
    // 128-token stages; a box is min(block_size, 128) rows of one 128-byte
    // column group.  Three stages.
    R = BS < pa::kTcTokens ? BS : pa::kTcTokens;
    prm.num_stages = 3;
    prm.num_consumers = 1;
    smem = pa::tc_smem_layout(D, prm.num_stages, cas != nullptr).total;
    prm.sched = sched;
    prm.trace = static_cast<unsigned long long*>(g_trace_buf.load());
    prm.trace_per_role = g_trace_per_role.load();
    prm.trace_bytes = g_trace_bytes.load();
    const long long limit = g_wait_limit.load();
    prm.wait_limit = limit > 0 ? limit : pa::kWaitLimitCycles;
    prm.total_items = (int)std::min<long long>((long long)num_seqs * desc->num_kv_heads * max_parts,
                                               (1ll << 31) - 1);
    // With many partitions per sequence most (partition, sequence, head)
    // slots of a mixed-length batch are past a sequence's end; the kernel
    // then numbers only the real items (batches it caches in shared memory).
    prm.dense_items = !balanced && max_parts > 4 && num_seqs <= pa::kTcLensCache;
    if (cas) {
      prm.seq_start = cas->seq_start;
      prm.part_counts = cas->counts;
      prm.dense_items = 0;
      if (!balanced) prm.total_items = num_seqs * desc->num_kv_heads;  // one item per pair
    }
    if (balanced) {
      prm.balanced = 1;
      prm.total_items = balanced_ranges(desc, sms);
      prm.part_counts = part_counts;
    }
  } else {
    // 32-token stages, TMA boxes of min(block_size, 32) rows, one box per
    // 128-byte column group, each box at a 1024-byte aligned slot so the
    // 128-byte swizzle pattern starts on an atom.
    R = BS < pa::kStageTokens ? BS : pa::kStageTokens;
    const int groups = D * es / 128;
    const int gslot = R * 128 > 1024 ? R * 128 : 1024;
    const int region = (pa::kStageTokens / R) * groups * gslot;
    const int stage_bytes = 2 * region;
    // As many stages as the budget holds (at most 64); at least two when two
    // fit in a CTA's shared memory, else one.  Every ring slot belongs to one
    // consumer warp, so the stage count is a multiple of the consumer count:
    // 4 consumers with 4, 8, ... stages, or 1-3 consumers with as many stages.
    const int merge = pa::decode_merge_bytes(group, D);
    auto area_for = [&](int n) {
      const int a = n * stage_bytes;
      return a < merge ? (merge + 15) / 16 * 16 : a;
    };
    int ns = kStageBudgetBytes / stage_bytes;
    if (ns < 3) ns = kStageBudgetWideBytes / stage_bytes;
    if (ns > 64) ns = 64;
    if (ns < 2) ns = pa::decode_smem_bytes(area_for(2), group, D) <= kMaxSmemPerCta ? 2 : 1;
    if (ns >= pa::kConsumerWarps) ns -= ns % pa::kConsumerWarps;
    prm.num_stages = ns;
    prm.num_consumers = ns < pa::kConsumerWarps ? ns : pa::kConsumerWarps;
    prm.kv_boxes = R >= 8;
    if (prm.kv_boxes) {
      // One box per block: [column group][K or V][R rows of 128 bytes].
      prm.group_slot = 2 * R * 128;
      prm.region_bytes = R * 128;
      prm.box_stride = groups * 2 * R * 128;
    } else {
      prm.group_slot = gslot;
      prm.region_bytes = region;
      prm.box_stride = groups * gslot;
    }
    prm.stage_bytes = stage_bytes;
    prm.stage_area = area_for(ns);
    // Unsplit batches are taken longest first (with a split the partitions
    // are of equal length but for the last, and the CTAs past a sequence's
    // end would pay for the ranking).  The lengths to rank fit in one stage
    // (at least 2 KB).
    prm.longest_first = num_seqs <= pa::kLongestFirstMaxSeqs && part == 0;
    smem = pa::decode_smem_bytes(prm.stage_area, group, D);
  }
  if (smem > kMaxSmemPerCta) return PA_ERR_UNSUPPORTED;

  EncodeTiledFn encode = nullptr;
  if ((st = encode_fn(&encode)) != PA_OK) return st;
  CUtensorMap map;
  std::memset(&map, 0, sizeof(map));
  // The pool as a 5-D tensor (innermost first): 128-byte column chunk,
  // column group, KV head, token within block, (K or V) * num_blocks + block.
  const int inner = 128 / es;
  const int groups = D * es / 128;
  const cuuint64_t gdim[5] = {(cuuint64_t)inner, (cuuint64_t)groups,
                              (cuuint64_t)desc->num_kv_heads, (cuuint64_t)BS,
                              2ull * (cuuint64_t)desc->num_blocks};
  const cuuint64_t gstride[4] = {128ull, (cuuint64_t)D * es,
                                 (cuuint64_t)desc->num_kv_heads * D * es,
                                 (cuuint64_t)BS * desc->num_kv_heads * D * es};
  const cuuint32_t box[5] = {(cuuint32_t)inner, 1u, 1u, (cuuint32_t)R, 1u};
  const cuuint32_t estride[5] = {1u, 1u, 1u, 1u, 1u};
  CUresult cr;
  if (use_tc) {
    cr = encode_tc_kv_map(encode, desc, cache, R, &map);
  } else if (prm.kv_boxes) {
    // CUDA-core kernel, blocks of 8 tokens or more: one box per block holds
    // its R rows of K and V for every column group, laid out
    // [column group][K or V][rows].  Dimensions, innermost first: one
    // 128-byte chunk; token within the block; K or V; (KV head, column
    // group); block.
    const cuuint64_t row = (cuuint64_t)desc->num_kv_heads * D * es;
    const cuuint64_t kdim[5] = {(cuuint64_t)inner, (cuuint64_t)BS, 2ull,
                                (cuuint64_t)desc->num_kv_heads * groups,
                                (cuuint64_t)desc->num_blocks};
    const cuuint64_t kstride[4] = {row, (cuuint64_t)desc->num_blocks * BS * row, 128ull,
                                   (cuuint64_t)BS * row};
    const cuuint32_t kbox[5] = {(cuuint32_t)inner, (cuuint32_t)R, 2u, (cuuint32_t)groups, 1u};
    cr = encode(&map,
                desc->dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                       : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                5, const_cast<void*>(cache), kdim, kstride, kbox, estride,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    cr = encode(&map,
                desc->dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                       : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                5, const_cast<void*>(cache), gdim, gstride, box, estride,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  if (cr != CUDA_SUCCESS) return PA_ERR_CUDA;
  // The tensor-core kernel loads each work item's 16 query rows by TMA: the
  // queries as [rows = num_seqs * num_heads][column group][64 elements].
  CUtensorMap qmap;
  std::memset(&qmap, 0, sizeof(qmap));
  if (use_tc) {
    const cuuint64_t qdim[3] = {64ull, (cuuint64_t)(D / 64),
                                (cuuint64_t)num_seqs * (cuuint64_t)num_heads};
    const cuuint64_t qstride[2] = {128ull, (cuuint64_t)D * 2};
    const cuuint32_t qbox[3] = {64u, 1u, (cuuint32_t)pa::kTcHeads};
    const cuuint32_t qes[3] = {1u, 1u, 1u};
    cr = encode(&qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(query), qdim,
                qstride, qbox, qes, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (cr != CUDA_SUCCESS) return PA_ERR_CUDA;
  }

  prm.out = out;
  prm.cache_w = static_cast<uint8_t*>(const_cast<void*>(cache));
  prm.new_k = new_k;
  prm.new_v = new_v;
  prm.query = query;
  prm.block_tables = block_tables;
  prm.seq_lens = seq_lens;
  prm.part_o = part_o;
  prm.part_lse = part_lse;
  prm.err = err;
  prm.num_blocks = desc->num_blocks;
  prm.block_size = BS;
  prm.log2_block_size = ilog2(BS);
  prm.num_kv_heads = desc->num_kv_heads;
  prm.num_heads = num_heads;
  prm.num_seqs = num_seqs;
  prm.group = group;
  prm.max_blocks_per_seq = max_blocks_per_seq;
  prm.partition_tokens = balanced ? 0 : part;
  prm.max_parts = max_parts;
  prm.scale_log2 = (float)((double)scale * 1.4426950408889634);
  prm.box_rows = R;
  prm.log2_box_rows = ilog2(R);

  const dim3 grid((unsigned)max_parts, (unsigned)desc->num_kv_heads, (unsigned)num_seqs);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  bool supported = true;
  cudaError_t e;
  if (use_tc)
    e = pa::launch_decode_tc(D, sms, smem, s, map, qmap, prm, &supported);
  else if (desc->dtype == PA_BF16)
    e = pa::launch_decode_bf16(D, group, grid, smem, s, map, prm, &supported);
  else
    e = pa::launch_decode_f32(D, group, grid, smem, s, map, prm, &supported);
  if (!supported) return PA_ERR_UNSUPPORTED;
  if (e != cudaSuccess) return PA_ERR_CUDA;
  if (!cas && (part > 0 || (balanced && max_parts > 1))) {
    e = pa::launch_lse_reduce(desc->dtype, D, out, part_o, part_lse, seq_lens, part_counts, group,
                              num_seqs, num_heads, balanced ? 0 : part, max_parts, s, &supported);
    if (!supported) return PA_ERR_UNSUPPORTED;
    if (e != cudaSuccess) return PA_ERR_CUDA;
  }
  return PA_OK;
}

pa_status pa_decode_ex(void* out, const void* query, const void* cache, const pa_cache_desc* desc,
                       const int32_t* block_tables, int32_t max_blocks_per_seq,
                       const int32_t* seq_lens, int32_t num_seqs, int32_t num_heads, float scale,
                       int32_t max_seq_len, int32_t partition_size, void* workspace,
                       size_t workspace_bytes, int32_t kernel, void* stream) {
  return decode_impl(out, query, cache, desc, block_tables, max_blocks_per_seq, seq_lens, num_seqs,
                     num_heads, scale, max_seq_len, partition_size, workspace, workspace_bytes,
                     kernel, nullptr, nullptr, stream);
}

pa_status pa_decode_append(void* out, const void* query, void* cache, const pa_cache_desc* desc,
                           const int32_t* block_tables, int32_t max_blocks_per_seq,
                           const int32_t* seq_lens, int32_t num_seqs, int32_t num_heads,
                           float scale, int32_t max_seq_len, int32_t partition_size,
                           const void* key_new, const void* value_new, void* workspace,
                           size_t workspace_bytes, int32_t kernel, void* stream) {
  if (num_seqs > 0 && (!key_new || !value_new || !aligned(key_new, 16) || !aligned(value_new, 16)))
    return PA_ERR_INVALID_ARG;
  return decode_impl(out, query, cache, desc, block_tables, max_blocks_per_seq, seq_lens, num_seqs,
                     num_heads, scale, max_seq_len, partition_size, workspace, workspace_bytes,
                     kernel, key_new, value_new, stream);
}

pa_status pa_decode_shared_workspace_size(const pa_cache_desc* desc, int32_t num_seqs,
                                          int32_t num_heads, int32_t max_seq_len,
                                          const pa_shared_plan_info* info, size_t* bytes) {
  pa_status st = check_desc(desc);
  if (st != PA_OK) return st;
  if (!bytes || !info || num_seqs < 0 || num_heads < 1 || num_heads % desc->num_kv_heads != 0 ||
      info->num_chunks < 0 || max_seq_len < 0)
    return PA_ERR_INVALID_ARG;
  if (info->num_chunks == 0) {
    *bytes = workspace_bytes_for(num_seqs, num_heads, desc->head_size, 0);
    return PA_OK;
  }
  int sms = 0;
  if ((st = device_state(nullptr, &sms)) != PA_OK) return st;
  *bytes = shared_workspace_bytes(num_seqs, num_heads, desc->num_kv_heads, desc->head_size,
                                  shared_max_parts(desc, info, num_seqs, max_seq_len, sms));
  return PA_OK;
}

pa_status pa_decode_shared(void* out, const void* query, void* cache, const pa_cache_desc* desc,
                           const int32_t* block_tables, int32_t max_blocks_per_seq,
                           const int32_t* seq_lens, int32_t num_seqs, int32_t num_heads,
                           float scale, int32_t max_seq_len, const int32_t* plan,
                           const pa_shared_plan_info* info, const void* key_new,
                           const void* value_new, void* workspace, size_t workspace_bytes,
                           void* stream) {
  pa_status st = check_desc(desc);
  if (st != PA_OK) return st;
  if (!info || (key_new == nullptr) != (value_new == nullptr)) return PA_ERR_INVALID_ARG;
  if (key_new && (!aligned(key_new, 16) || !aligned(value_new, 16))) return PA_ERR_INVALID_ARG;
  if (num_seqs < 0 || num_seqs > 65535 || num_heads < 1 || max_seq_len < 0 ||
      max_blocks_per_seq < 1 || !std::isfinite(scale) || num_heads % desc->num_kv_heads != 0)
    return PA_ERR_INVALID_ARG;
  if (num_seqs == 0) return PA_OK;
  if (!out || !query || !cache || !block_tables || !seq_lens) return PA_ERR_INVALID_ARG;
  int32_t family = 0;
  if ((st = select_kernel(desc, num_seqs, num_heads, query, PA_KERNEL_TENSOR, &family)) != PA_OK)
    return st;
  const int nc = info->num_chunks;
  if (nc == 0)  // nothing shared: the unsplit tensor-core decode
    return decode_impl(out, query, cache, desc, block_tables, max_blocks_per_seq, seq_lens,
                       num_seqs, num_heads, scale, max_seq_len, 0, workspace, workspace_bytes,
                       PA_KERNEL_TENSOR, key_new, value_new, stream);
  const int group = num_heads / desc->num_kv_heads;
  if (nc < 0 || info->num_members < nc || info->num_members > num_seqs ||
      info->group_size != group || info->min_shared_tokens < desc->block_size ||
      info->min_chunk_stages < 1 ||
      info->plan_ints != 4 + 4 * nc + num_seqs + info->num_members || !plan || !aligned(plan, 4))
    return PA_ERR_INVALID_ARG;
  unsigned int* err = nullptr;
  int sms = 0;
  if ((st = device_state(&err, &sms)) != PA_OK) return st;
  const int D = desc->head_size;
  const int ranges = shared_ranges(desc, info, sms);
  const int max_parts = shared_max_parts(desc, info, num_seqs, max_seq_len, sms);
  const size_t need =
      shared_workspace_bytes(num_seqs, num_heads, desc->num_kv_heads, D, max_parts);
  if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return PA_ERR_INVALID_ARG;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const size_t rows = (size_t)num_seqs * num_heads * max_parts;
  float* part_o = reinterpret_cast<float*>(ws + 256);
  float* part_lse = reinterpret_cast<float*>(ws + 256 + (rows * D * 4 + 255) / 256 * 256);
  int32_t* counts = reinterpret_cast<int32_t*>(ws + 256 + (rows * D * 4 + 255) / 256 * 256 +
                                               (rows * 4 + 255) / 256 * 256);

  EncodeTiledFn encode = nullptr;
  if ((st = encode_fn(&encode)) != PA_OK) return st;
  const int R = desc->block_size < pa::kTcTokens ? desc->block_size : pa::kTcTokens;
  CUtensorMap map;
  std::memset(&map, 0, sizeof(map));
  if (encode_tc_kv_map(encode, desc, cache, R, &map) != CUDA_SUCCESS) return PA_ERR_CUDA;
  pa::SharedParams sp;
  std::memset(&sp, 0, sizeof(sp));
  sp.query = query;
  sp.block_tables = block_tables;
  sp.seq_lens = seq_lens;
  sp.chunks = plan + 4;
  sp.members = plan + 4 + 4 * (size_t)nc + num_seqs;
  sp.out = out;
  sp.part_o = part_o;
  sp.part_lse = part_lse;
  sp.part_counts = counts;
  sp.cache_w = static_cast<uint8_t*>(cache);
  sp.new_k = key_new;
  sp.new_v = value_new;
  sp.err = err;
  sp.num_chunks = nc;
  sp.num_members = info->num_members;
  sp.num_seqs = num_seqs;
  sp.num_heads = num_heads;
  sp.num_kv_heads = desc->num_kv_heads;
  sp.group = group;
  sp.num_blocks = desc->num_blocks;
  sp.block_size = desc->block_size;
  sp.log2_block_size = ilog2(desc->block_size);
  sp.max_blocks_per_seq = max_blocks_per_seq;
  sp.max_parts = max_parts;
  sp.ranges = ranges;
  sp.box_rows = R;
  sp.log2_box_rows = ilog2(R);
  sp.num_stages = pa::shared_stage_slots(D);
  sp.scale_log2 = (float)((double)scale * 1.4426950408889634);
  const long long limit = g_wait_limit.load();
  sp.wait_limit = limit > 0 ? limit : pa::kWaitLimitCycles;
  sp.trace = static_cast<unsigned long long*>(g_trace_buf.load());
  sp.trace_per_role = g_trace_per_role.load();
  sp.trace_bytes = g_trace_bytes.load();
  // The decode launch after it records CTAs from 0 (at most two per SM).
  sp.trace_cta_base = 2 * sms;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  bool supported = true;
  const dim3 grid((unsigned)ranges, (unsigned)desc->num_kv_heads, (unsigned)nc);
  cudaError_t e =
      pa::launch_decode_shared(D, grid, pa::shared_smem_bytes(D), s, map, sp, &supported);
  if (!supported) return PA_ERR_UNSUPPORTED;
  if (e != cudaSuccess) return PA_ERR_CUDA;
  const bool others = info->num_members < num_seqs;
  if (others) {
    // The sequences outside every group.
    const CascadeArgs cas{plan + 4 + 4 * (size_t)nc, counts, part_o, part_lse, max_parts};
    st = decode_impl(out, query, cache, desc, block_tables, max_blocks_per_seq, seq_lens,
                     num_seqs, num_heads, scale, max_seq_len, 0, workspace, workspace_bytes,
                     PA_KERNEL_TENSOR, key_new, value_new, stream, &cas);
    if (st != PA_OK) return st;
  }
  if (ranges > 1 || others) {
    e = pa::launch_lse_reduce(desc->dtype, D, out, part_o, part_lse, seq_lens, counts, group,
                              num_seqs, num_heads, 0, max_parts, s, &supported);
    if (!supported) return PA_ERR_UNSUPPORTED;
    if (e != cudaSuccess) return PA_ERR_CUDA;
  }
  return PA_OK;
}

}  // extern "C"
