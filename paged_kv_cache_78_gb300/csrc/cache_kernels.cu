// Cache write (reshape_and_cache) and copy-on-write block copy for sm_103a.
//
// Both are byte moves in 16-byte vectors.  In the pool layout
// [2][num_blocks][block_size][num_kv_heads][head_size] the slot
// b * block_size + t of plane kv starts at element
// ((kv * num_blocks + b) * block_size + t) * Hkv * D = (kv * NB * BS + slot) * Hkv * D,
// so one token's heads form one contiguous row of Hkv * D elements, and one
// physical block of one plane is block_size such rows.
#include "pa_device.cuh"
#include "pa_launch.h"

namespace pa {

// One thread per (token, K or V, 16-byte chunk of the token's row).
// The new token's key and value go to the slot slot_mapping names
// (itan.pw "vLLMにおけるKVCacheマネージャーの詳細解説", section
// "ブロックアロケーションの基本概念"); slot < 0 is padding.
__global__ void reshape_and_cache_kernel(uint8_t* __restrict__ cache,
                                         const uint8_t* __restrict__ key,
                                         const uint8_t* __restrict__ value,
                                         const int64_t* __restrict__ slot_mapping,
                                         int64_t num_tokens, int64_t num_slots, int row_chunks,
                                         int64_t plane_bytes, unsigned int* err) {
  grid_dependents_launch();
  grid_dependency_wait();
  const int64_t per_token = 2 * (int64_t)row_chunks;
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= num_tokens * per_token) return;
  const int64_t t = i / per_token;
  const int r = (int)(i - t * per_token);
  const int kv = r >= row_chunks;
  const int c = kv ? r - row_chunks : r;
  const int64_t slot = __ldg(slot_mapping + t);
  if (slot < 0) return;
  if (slot >= num_slots) {
    if (r == 0) record_error(err, PA_DEVERR_SLOT);
    return;
  }
  const int64_t row_bytes = (int64_t)row_chunks * 16;
  const uint8_t* src = (kv ? value : key) + t * row_bytes + (int64_t)c * 16;
  uint8_t* dst = cache + kv * plane_bytes + slot * row_bytes + (int64_t)c * 16;
  stg_v4(dst, ldg_nc_v4(src));
}

// One CTA per (pair, K or V, slice of the block): block src of the source
// pool -> block dst of the destination pool, copied whole.  Copy-on-write
// copies within one pool (studying-code.tistory.com/16, section "생성 단계에서의
// Copy-on-Write": the writer of a shared block copies its content to a new
// block); swapping copies between the GPU pool and a CPU pool of the same
// block geometry (same page, section "스와핑(Swapping)").
__global__ void copy_blocks_kernel(uint8_t* __restrict__ dst_cache,
                                   const uint8_t* __restrict__ src_cache,
                                   const int64_t* __restrict__ pairs, int64_t dst_blocks,
                                   int64_t src_blocks, int64_t block_bytes, int64_t dst_plane,
                                   int64_t src_plane, unsigned int* err) {
  grid_dependents_launch();
  grid_dependency_wait();
  const int pair = blockIdx.x >> 1;
  const int kv = blockIdx.x & 1;
  const int64_t src = __ldg(pairs + 2 * pair);
  const int64_t dst = __ldg(pairs + 2 * pair + 1);
  if (src < 0 || dst < 0 || src >= src_blocks || dst >= dst_blocks) {
    if (kv == 0 && blockIdx.y == 0 && threadIdx.x == 0) record_error(err, PA_DEVERR_BLOCK_ID);
    return;
  }
  const uint8_t* s = src_cache + kv * src_plane + src * block_bytes;
  uint8_t* d = dst_cache + kv * dst_plane + dst * block_bytes;
  const int64_t n16 = block_bytes / 16;
  const int64_t step = (int64_t)gridDim.y * blockDim.x;
  int64_t i = (int64_t)blockIdx.y * blockDim.x + threadIdx.x;
  // Four independent 16-byte loads in flight per thread.
  for (; i + 3 * step < n16; i += 4 * step) {
    const uint4 a = ldg_nc_v4(s + i * 16);
    const uint4 b = ldg_nc_v4(s + (i + step) * 16);
    const uint4 c = ldg_nc_v4(s + (i + 2 * step) * 16);
    const uint4 e = ldg_nc_v4(s + (i + 3 * step) * 16);
    stg_v4(d + i * 16, a);
    stg_v4(d + (i + step) * 16, b);
    stg_v4(d + (i + 2 * step) * 16, c);
    stg_v4(d + (i + 3 * step) * 16, e);
  }
  for (; i < n16; i += step) stg_v4(d + i * 16, ldg_nc_v4(s + i * 16));
}

// Plain byte copy between any two addresses the GPU reaches (device memory,
// page-locked host memory through its mapping).  A kernel rather than a copy
// engine so that it chains with the neighbouring launches by programmatic
// dependent launch: the step's host-side inputs come in and its output goes
// out without the copy engine's own start-up on the stream.  Both sides
// 16-byte aligned: 16-byte vectors, four in flight per thread, then the
// ragged tail byte by byte; otherwise byte by byte throughout.
__global__ void copy_bytes_kernel(uint8_t* __restrict__ dst, const uint8_t* src,
                                  int64_t bytes, int vec) {
  grid_dependents_launch();
  grid_dependency_wait();
  const int64_t step = (int64_t)gridDim.x * blockDim.x;
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  int64_t done = 0;
  if (vec) {
    const int64_t n16 = bytes / 16;
    int64_t i = t;
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    for (; i + 3 * step < n16; i += 4 * step) {
      const uint4 a = __ldcg(s4 + i);
      const uint4 b = __ldcg(s4 + i + step);
      const uint4 c = __ldcg(s4 + i + 2 * step);
      const uint4 e = __ldcg(s4 + i + 3 * step);
      stg_v4(dst + i * 16, a);
      stg_v4(dst + (i + step) * 16, b);
      stg_v4(dst + (i + 2 * step) * 16, c);
      stg_v4(dst + (i + 3 * step) * 16, e);
    }
    for (; i < n16; i += step) stg_v4(dst + i * 16, __ldcg(s4 + i));
    done = n16 * 16;
  }
  for (int64_t i = done + t; i < bytes; i += step) dst[i] = __ldcg(src + i);
}

cudaError_t launch_reshape_and_cache(void* cache, const void* key, const void* value,
                                     const int64_t* slot_mapping, int64_t num_tokens,
                                     int64_t num_slots, int row_bytes, int64_t plane_bytes,
                                     unsigned int* err, cudaStream_t stream) {
  const int row_chunks = row_bytes / 16;
  const int64_t threads = num_tokens * 2 * row_chunks;
  const int block = 256;
  const int64_t grid = (threads + block - 1) / block;
  uint8_t* c = static_cast<uint8_t*>(cache);
  const uint8_t* k = static_cast<const uint8_t*>(key);
  const uint8_t* v = static_cast<const uint8_t*>(value);
  void* args[] = {&c, &k, &v, &slot_mapping, &num_tokens, &num_slots,
                  const_cast<int*>(&row_chunks), &plane_bytes, &err};
  return launch_overlapped((const void*)reshape_and_cache_kernel, dim3((unsigned)grid),
                           dim3(block), 0, stream, args);
}

cudaError_t launch_copy_blocks(void* dst_cache, const void* src_cache, const int64_t* pairs,
                               int num_pairs, int64_t dst_blocks, int64_t src_blocks,
                               int64_t block_bytes, unsigned int* err, cudaStream_t stream) {
  const int block = 256;
  const int64_t per_cta = (int64_t)block * 16 * 8;  // about 8 vectors per thread
  int slices = (int)((block_bytes + per_cta - 1) / per_cta);
  if (slices < 1) slices = 1;
  if (slices > 1024) slices = 1024;
  dim3 grid((unsigned)num_pairs * 2u, (unsigned)slices);
  uint8_t* d = static_cast<uint8_t*>(dst_cache);
  const uint8_t* s = static_cast<const uint8_t*>(src_cache);
  int64_t dst_plane = dst_blocks * block_bytes, src_plane = src_blocks * block_bytes;
  void* args[] = {&d, &s, &pairs, &dst_blocks, &src_blocks, &block_bytes, &dst_plane, &src_plane,
                  &err};
  return launch_overlapped((const void*)copy_blocks_kernel, grid, dim3(block), 0, stream, args);
}

cudaError_t launch_copy_bytes(void* dst, const void* src, int64_t bytes, int num_sms,
                              cudaStream_t stream) {
  const int block = 256;
  const int vec = ((reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src)) & 15) == 0;
  const int64_t units = vec ? bytes / 16 : bytes;
  int64_t grid = (units + block - 1) / block;
  if (grid > 2 * (int64_t)num_sms) grid = 2 * (int64_t)num_sms;
  if (grid < 1) grid = 1;
  uint8_t* d = static_cast<uint8_t*>(dst);
  const uint8_t* s = static_cast<const uint8_t*>(src);
  void* args[] = {&d, &s, &bytes, const_cast<int*>(&vec)};
  return launch_overlapped((const void*)copy_bytes_kernel, dim3((unsigned)grid), dim3(block), 0,
                           stream, args);
}

}  // namespace pa
