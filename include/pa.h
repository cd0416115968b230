/*
 * pa.h -- C ABI of the GB300 paged KV-cache library (libpa.so).
 *
 * One layer's KV cache is a single device buffer laid out as
 *
 *     cache[2][num_blocks][block_size][num_kv_heads][head_size]
 *
 * with index 0 of the first axis holding keys and 1 values.  This is the
 * per-layer tensor the itan.pw page ("vLLMにおけるKVCacheマネージャーの詳細解説",
 * sections "ブロックアロケーションの基本概念" and "BlockPoolの生成過程")
 * allocates for every attention layer: num_blocks physical blocks of
 * block_size token slots each.  A sequence reaches its tokens through a block
 * table that maps logical block i to a physical block (studying-code.tistory.com/16,
 * section "vLLM 방식: 논리 ↔ 물리 메모리 분리").  Token j of a sequence lives
 * in slot  table[j / block_size] * block_size + j % block_size.
 *
 * Conventions for every call below
 *   - Device pointers are plain CUDA device addresses the caller allocated;
 *     the library never allocates, frees or synchronises device memory except
 *     where a call says so.  Host pointers are ordinary process memory.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Kernel calls are asynchronous on that stream.
 *   - Arguments are checked on the host before any launch; a bad argument
 *     returns PA_ERR_INVALID_ARG (or PA_ERR_UNSUPPORTED for a valid shape this
 *     build has no kernel for) and launches nothing.  A failed launch returns
 *     PA_ERR_CUDA.
 *   - Index errors that only the device can see (a slot, block id or
 *     sequence length outside the pool or table) are recorded in a per-device
 *     error word and the offending access is skipped; nothing traps.  Read
 *     the word with pa_get_device_error().
 *   - dtype (pa_cache_desc.dtype) is the element type of the cache and of
 *     every key, value, query and output tensor of the call.  Arithmetic is
 *     fp32 in both cases.
 */
#ifndef PAGED_KV_CACHE_PA_H_
#define PAGED_KV_CACHE_PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pa_status {
  PA_OK = 0,
  PA_ERR_INVALID_ARG = 1,    /* null pointer, bad size or inconsistent shape */
  PA_ERR_UNSUPPORTED = 2,    /* valid, but the library has no kernel for it (head size, group) */
  PA_ERR_CUDA = 3,           /* a CUDA runtime call or launch failed */
  PA_ERR_OUT_OF_BLOCKS = 4,  /* block pool exhausted; pool state unchanged */
  PA_ERR_BAD_STATE = 5,      /* unknown sequence id, or an operation the state forbids */
  PA_ERR_DEVICE_CHECK = 6,   /* pa_get_device_error found a recorded device-side error */
  PA_ERR_TIMEOUT = 7         /* a bounded device wait gave up (see pa_get_device_error) */
} pa_status;

typedef enum pa_dtype { PA_BF16 = 0, PA_FP32 = 1 } pa_dtype;

/* Bits of the device error word. */
#define PA_DEVERR_SLOT 0x1u        /* reshape_and_cache: slot >= num_blocks * block_size */
#define PA_DEVERR_BLOCK_ID 0x2u    /* decode / copy_blocks: block id outside [0, num_blocks) */
#define PA_DEVERR_SEQ_LEN 0x4u     /* decode: seq_len > max_seq_len or > table capacity */
#define PA_DEVERR_TIMEOUT 0x8u     /* a pipeline wait exceeded its limit (about 2 s by default) */

/* partition_size of pa_decode: the stage-balanced split (see pa_decode). */
#define PA_PARTITION_BALANCED (-2)

/* Geometry of one layer's cache. */
typedef struct pa_cache_desc {
  int32_t num_blocks;    /* physical blocks in the pool, >= 1 */
  int32_t block_size;    /* token slots per block: a power of two in [1, 256] */
  int32_t num_kv_heads;  /* KV heads, >= 1 */
  int32_t head_size;     /* elements per head: 64, 128 or 256 */
  int32_t dtype;         /* pa_dtype */
} pa_cache_desc;

/* ---------------------------------------------------------------------------
 * Cache write.  Each new token's key and value go to the physical slot that
 * slot_mapping names (itan.pw page, section "ブロックアロケーションの基本概念":
 * slot_mapping records, for every new token, its slot in the physical KV cache;
 * studying-code.tistory.com/16, section "디코딩 과정": new KV is stored into
 * physical blocks during each iteration):
 *     cache[0][slot / block_size][slot % block_size][h][:] = key[t][h][:]
 *     cache[1][slot / block_size][slot % block_size][h][:] = value[t][h][:]
 *   cache         device, in/out, the layer's pool.
 *   key, value    device, [num_tokens][num_kv_heads][head_size], contiguous.
 *   slot_mapping  device int64 [num_tokens]; slot < 0 marks a padding token
 *                 that is skipped.  Slots must be distinct (two tokens writing
 *                 one slot leave either value).  A slot past the pool is
 *                 skipped and recorded as PA_DEVERR_SLOT.
 * Result is bit-exact: a byte copy.  num_tokens == 0 is a no-op.
 * ------------------------------------------------------------------------- */
pa_status pa_reshape_and_cache(void* cache, const pa_cache_desc* desc, const void* key,
                               const void* value, const int64_t* slot_mapping,
                               int32_t num_tokens, void* stream);

/* ---------------------------------------------------------------------------
 * Copy-on-write block copies.  For each pair i, physical block
 * pairs[2i] (source) is copied to block pairs[2i+1] (destination), keys and
 * values, bit-exactly (studying-code.tistory.com/16, section "생성 단계에서의
 * Copy-on-Write": the writer of a shared block takes a new block and copies
 * the old block's content into it; section "메모리 복사 오버헤드의 최적화":
 * only that one block is copied).
 *   pairs   device int64 [num_pairs][2].  Destinations must be distinct and
 *           no destination may also be a source in the same call (the pool
 *           only emits fresh destinations).  An id outside the pool skips the
 *           pair and records PA_DEVERR_BLOCK_ID.
 * num_pairs == 0 is a no-op; num_pairs above 2^30 - 1 returns
 * PA_ERR_INVALID_ARG.
 * ------------------------------------------------------------------------- */
pa_status pa_copy_blocks(void* cache, const pa_cache_desc* desc, const int64_t* pairs,
                         int32_t num_pairs, void* stream);

/* ---------------------------------------------------------------------------
 * Swap block copies between two pools of the same block geometry (block
 * size, KV heads, head size, dtype; the block counts may differ): for each
 * pair i, block pairs[2i] of src_cache is copied to block pairs[2i+1] of
 * dst_cache, keys and values, bit-exactly.  The pages' swapping moves a
 * preempted sequence's blocks to CPU memory and back
 * (studying-code.tistory.com/16, section "스와핑(Swapping)").  One of the
 * pools is normally the GPU pool and the other a CPU pool in page-locked
 * host memory, which the kernel reads or writes directly (over NVLink-C2C on
 * GB300).  Each of dst_cache, src_cache and pairs must be device memory or
 * page-locked host memory; pageable host memory returns PA_ERR_INVALID_ARG
 * and launches nothing.  pairs: int64 [num_pairs][2] (pa_pool_swap_out /
 * pa_pool_swap_in give them).  An id outside its pool skips the pair and
 * records PA_DEVERR_BLOCK_ID.  num_pairs above 2^30 - 1 returns
 * PA_ERR_INVALID_ARG.  Asynchronous on `stream`: the host pool may
 * be reused only after the stream has passed the copy.
 * ------------------------------------------------------------------------- */
pa_status pa_swap_blocks(void* dst_cache, const pa_cache_desc* dst_desc, const void* src_cache,
                         const pa_cache_desc* src_desc, const int64_t* pairs, int32_t num_pairs,
                         void* stream);

/* ---------------------------------------------------------------------------
 * Copy `bytes` bytes from src to dst with a kernel on `stream`.  Each of dst
 * and src is device memory or page-locked host memory (read or written
 * through its device mapping, over NVLink-C2C on GB300); pageable host
 * memory returns PA_ERR_INVALID_ARG and launches nothing, and so do
 * overlapping ranges.  This is how a serving step's host-side inputs (the
 * new tokens' query, K and V, slot mapping, block tables and lengths) come
 * in and its attention output goes out: as a kernel, the copy chains with
 * pa_reshape_and_cache and pa_decode by programmatic dependent launch, where
 * a copy-engine transfer would stop the chain on both sides.  Any size and
 * alignment; 16-byte aligned pointers on both sides move 16 bytes per load.
 * bytes == 0 is a no-op.  Asynchronous on `stream`: the host side may be
 * reused (src) or read (dst) only after the stream has passed the copy.
 * ------------------------------------------------------------------------- */
pa_status pa_copy_bytes(void* dst, const void* src, size_t bytes, void* stream);

/* ---------------------------------------------------------------------------
 * Paged decode attention: one query token per sequence against the
 * sequence's cached tokens, block by block through its block table
 * (studying-code.tistory.com/16, section "PagedAttention: 운영체제의 페이징
 * 개념에서 영감을 받은 새로운 어텐션 알고리즘": the query is multiplied with each
 * block's keys and values and the per-block results are combined into o_i;
 * garden.houmin.site/infra/paged-attention, section "KV Cache 管理器").  The
 * pages print no softmax or scale; the operation is the standard one:
 *
 *   out[s][hq][:] = sum_j softmax_j(scale * q[s][hq] . k_j) v_j,  j < seq_lens[s],
 *   k_j = cache[0][table[s][j / bs]][j % bs][hq / G][:],  v_j likewise at index 1,
 *   G = num_heads / num_kv_heads (query heads hq = h*G .. h*G+G-1 share KV head h).
 *
 *   out          device [num_seqs][num_heads][head_size], dtype.
 *   query        device [num_seqs][num_heads][head_size], dtype.
 *   block_tables device int32 [num_seqs][max_blocks_per_seq]; only the first
 *                ceil(seq_lens[s] / block_size) entries of row s are read.
 *   seq_lens     device int32 [num_seqs]; the count includes the token just
 *                written.  0 gives a zero output row.
 *   max_seq_len  host bound on every seq_lens[s] (sizes the split grid).
 *   partition_size  0: one CTA per (sequence, KV head) walks the whole
 *                sequence.  > 0: split-KV, tokens cut into partitions of this
 *                many tokens (a multiple of block_size), each reduced to a
 *                partial (max, sum, weighted values) in workspace, then
 *                combined by a log-sum-exp reduce kernel.  -1: the library
 *                picks (pa_decode_partition_size reports the choice).
 *                PA_PARTITION_BALANCED (-2): the tensor-core kernel's
 *                persistent CTAs get equal shares of the batch's work.  The
 *                128-token stages of every (sequence, KV head) pair are laid
 *                end to end and cut into one range of ceil(stages / ranges)
 *                stages per resident CTA; a pair cut by range ends becomes
 *                several partials, combined as above.  It applies to the
 *                tensor-core kernel and batches of up to 256 sequences; for
 *                other shapes -2 is treated as -1.  If the CUDA-core kernel
 *                runs the call instead (a query that is not 16-byte aligned,
 *                or PA_KERNEL_SIMT), it splits into equal partitions that fit
 *                the same workspace.
 *   workspace    device scratch of at least pa_decode_workspace_size() bytes,
 *                256-byte aligned.  Its first 256 bytes hold the tensor-core
 *                kernel's work counter: they must be zero when the workspace
 *                is first used (allocate it zeroed), and every call leaves
 *                them zero.  The rest (split-KV partials) needs no
 *                initialisation.  It may be NULL for a CUDA-core call that
 *                does not split.  Calls that overlap on the GPU need separate
 *                workspaces.
 * G = num_heads / num_kv_heads must be at most 16 for bf16 caches whose
 * head size is 64 or 128 and whose blocks hold 8 tokens or more (tensor-core
 * kernel), at most 8 otherwise (CUDA-core kernel).  Grouped heads share each
 * K/V block load.  Arithmetic: fp32 scores and an online fp32 softmax; bf16
 * output is rounded to nearest even.  A sequence longer than max_seq_len or than its
 * table row is recorded as PA_DEVERR_SEQ_LEN and its row is left undefined.
 * ------------------------------------------------------------------------- */
pa_status pa_decode(void* out, const void* query, const void* cache, const pa_cache_desc* desc,
                    const int32_t* block_tables, int32_t max_blocks_per_seq,
                    const int32_t* seq_lens, int32_t num_seqs, int32_t num_heads, float scale,
                    int32_t max_seq_len, int32_t partition_size, void* workspace,
                    size_t workspace_bytes, void* stream);

/* Kernel families for pa_decode_ex. */
typedef enum pa_decode_kernel {
  PA_KERNEL_AUTO = 0,   /* tensor cores where supported and G >= 2, else CUDA cores */
  PA_KERNEL_SIMT = 1,   /* CUDA cores: fp32 dot products and accumulation; group <= 8 */
  PA_KERNEL_TENSOR = 2  /* 5th-generation tensor cores: bf16 only, head size 64 or 128,
                           group <= 16, block_size >= 8; scores and P.V accumulate in fp32,
                           the softmax weights P enter the P.V product rounded to bf16 */
} pa_decode_kernel;

/* pa_decode with an explicit kernel family (PA_ERR_UNSUPPORTED when the
 * requested family has no kernel for the arguments).  pa_decode is
 * pa_decode_ex with PA_KERNEL_AUTO. */
pa_status pa_decode_ex(void* out, const void* query, const void* cache, const pa_cache_desc* desc,
                       const int32_t* block_tables, int32_t max_blocks_per_seq,
                       const int32_t* seq_lens, int32_t num_seqs, int32_t num_heads, float scale,
                       int32_t max_seq_len, int32_t partition_size, void* workspace,
                       size_t workspace_bytes, int32_t kernel, void* stream);

/* ---------------------------------------------------------------------------
 * pa_decode_ex with the step's cache write fused in: each sequence's newest
 * token (position seq_lens[s] - 1, the token the decode step appends) has
 * its keys and values in key_new / value_new, device, cache dtype,
 * [num_seqs][num_kv_heads][head_size], 16-byte aligned.  Before reading that
 * token, the decode writes it into the slot its block table gives
 * (block_tables[s][(L-1) / block_size] * block_size + (L-1) % block_size),
 * exactly what pa_reshape_and_cache with that slot mapping writes; the
 * write and the read are one launch instead of two (the pages' decode step
 * stores the new token's KV in its block, then attends:
 * studying-code.tistory.com/16, section "디코딩 과정").  Copy-on-write copies
 * (pa_copy_blocks) must run before.  A sequence of length 0 writes nothing;
 * a block id outside the pool skips the write and records
 * PA_DEVERR_BLOCK_ID.  Other arguments and results as pa_decode_ex.
 * ------------------------------------------------------------------------- */
pa_status pa_decode_append(void* out, const void* query, void* cache, const pa_cache_desc* desc,
                           const int32_t* block_tables, int32_t max_blocks_per_seq,
                           const int32_t* seq_lens, int32_t num_seqs, int32_t num_heads,
                           float scale, int32_t max_seq_len, int32_t partition_size,
                           const void* key_new, const void* value_new, void* workspace,
                           size_t workspace_bytes, int32_t kernel, void* stream);

/* ---------------------------------------------------------------------------
 * Shared-prefix decode.  Sequences that share leading physical blocks
 * (parallel samples forked from one prompt, studying-code.tistory.com/16,
 * section "생성 단계에서의 Copy-on-Write", tech.blogsailing.com/?p=100,
 * section 3; requests whose prompts hit the same cached prefix, itan.pw page,
 * section "プレイフィックスキャッシュの詳細") hold the same K/V rows for those
 * tokens.  The pages share the memory; these calls also share the work: a
 * group's query rows (up to 128 per tile) attend the shared blocks together,
 * each block read once, and then their members' own blocks, packed several
 * members to a 128-token stage with every row masked to its own member's
 * tokens; the result is the same as pa_decode's.  Sequences outside every
 * group go to the tensor-core decode in the same call.
 *
 * pa_decode_shared_plan (host only) finds the sharing from the host copy of
 * the block tables: sequences with the same first block id form a group;
 * its shared length is the longest run of leading block ids all members
 * have in common, capped for every member at floor((seq_len - 1) /
 * block_size) blocks (each member's newest token stays its own).  Groups of
 * one member or of fewer than min_shared_blocks shared blocks are dropped.
 * A group is cut into chunks of 4 * floor(32 / G) members (G = num_heads /
 * num_kv_heads; at most PA_SHARED_TILE_ROWS query rows, a member's G rows in
 * one of four 32-row warps).  The plan is written to `plan` (host,
 * PA_SHARED_PLAN_INTS(num_seqs) int32 at least), its sizes to *info:
 *   plan[0..3]   chunks, sequences, members, G
 *   then per chunk {first member index, members, shared tokens, group},
 *   per sequence the first token of its own part (0 outside a group), and
 *   the members' sequence ids.
 * Returns PA_ERR_INVALID_ARG for bad sizes, a table too short for a length,
 * or G > 32.
 * ------------------------------------------------------------------------- */
#define PA_SHARED_TILE_ROWS 128
#define PA_SHARED_PLAN_INTS(num_seqs) (4 + 6 * (int64_t)(num_seqs))
typedef struct pa_shared_plan_info {
  int32_t num_chunks;         /* chunks of query rows (0: nothing is shared) */
  int32_t num_members;        /* sequences in a group */
  int32_t min_shared_tokens;  /* fewest shared tokens of any chunk */
  int32_t min_chunk_stages;   /* fewest 128-token stages of any chunk (shared and own tokens) */
  int32_t group_size;         /* G the plan was built for */
  int32_t plan_ints;          /* int32 of the plan in use (the bytes to upload) */
} pa_shared_plan_info;
pa_status pa_decode_shared_plan(const int32_t* block_tables, int32_t max_blocks_per_seq,
                                const int32_t* seq_lens, int32_t num_seqs, int32_t block_size,
                                int32_t num_heads, int32_t num_kv_heads,
                                int32_t min_shared_blocks, int32_t* plan, size_t plan_ints,
                                pa_shared_plan_info* info);

/* Workspace bytes of pa_decode_shared for this batch (max_seq_len bounds
 * its lengths, as in pa_decode) and plan (256-byte aligned; zero it once at
 * allocation, every call leaves its header zero). */
pa_status pa_decode_shared_workspace_size(const pa_cache_desc* desc, int32_t num_seqs,
                                          int32_t num_heads, int32_t max_seq_len,
                                          const pa_shared_plan_info* info, size_t* bytes);

/* pa_decode over the same arguments, with the shared blocks of the plan's
 * groups attended once per group.  `plan` is a device copy of the first
 * info->plan_ints int32 that pa_decode_shared_plan wrote for exactly these
 * block tables and lengths (a plan for other tables gives wrong rows; it
 * cannot make the kernels touch memory outside the pool, the tables, the
 * queries, the workspace or the output: member ids, shared lengths and
 * ranges are checked on the device, and a violation records
 * PA_DEVERR_SEQ_LEN and leaves those rows undefined).  key_new / value_new:
 * both NULL, or the step's newest tokens as in pa_decode_append (written into
 * the cache by the decode).  The tensor-core decode must support the shape
 * (bf16, head size 64 or 128, G <= 16, blocks of 8 tokens or more, a
 * 16-byte aligned query), else PA_ERR_UNSUPPORTED.  A plan without chunks
 * runs pa_decode_ex's unsplit tensor-core decode.  Asynchronous on `stream`.
 * Launches: the group kernel (grid: stage ranges x KV heads x chunks, the
 * ranges chosen to fill the SMs; with one range it writes final rows); the
 * tensor-core decode of the sequences outside every group, if any (the
 * balanced split for batches of up to 256 sequences); the log-sum-exp reduce
 * when some row has several partials. */
pa_status pa_decode_shared(void* out, const void* query, void* cache, const pa_cache_desc* desc,
                           const int32_t* block_tables, int32_t max_blocks_per_seq,
                           const int32_t* seq_lens, int32_t num_seqs, int32_t num_heads,
                           float scale, int32_t max_seq_len, const int32_t* plan,
                           const pa_shared_plan_info* info, const void* key_new,
                           const void* value_new, void* workspace, size_t workspace_bytes,
                           void* stream);

/* The kernel family pa_decode_ex(..., kernel, ...) runs for a cache `desc`,
 * num_seqs sequences of num_heads query heads and a query buffer at `query`
 * (its address only decides the 16-byte alignment the tensor-core kernel
 * needs; it is not read): PA_KERNEL_SIMT or PA_KERNEL_TENSOR in *selected.
 * PA_ERR_UNSUPPORTED when the requested family has no kernel for these
 * arguments, PA_ERR_INVALID_ARG for arguments pa_decode_ex rejects.  Host
 * only: touches no device. */
pa_status pa_decode_select_kernel(const pa_cache_desc* desc, int32_t num_seqs, int32_t num_heads,
                                  const void* query, int32_t kernel, int32_t* selected);

/* The partition size pa_decode uses for these arguments (0 = no split,
 * PA_PARTITION_BALANCED for the balanced split). */
pa_status pa_decode_partition_size(const pa_cache_desc* desc, int32_t num_seqs,
                                   int32_t num_heads, int32_t max_seq_len,
                                   int32_t partition_size, int32_t* resolved);

/* Workspace bytes pa_decode needs for these arguments: a 256-byte header,
 * plus num_seqs * num_heads * max_partitions * (head_size + 1) * 4 (each part
 * rounded up to 256) when it splits.  The balanced split adds
 * num_seqs * num_kv_heads * 4 bytes (rounded up to 256) of piece counts;
 * its max_partitions is min(ceil(max_seq_len / 128),
 * ceil(ranges / num_kv_heads) + 1), where ranges is the number of SMs times
 * two for head size 64, times one for 128. */
pa_status pa_decode_workspace_size(const pa_cache_desc* desc, int32_t num_seqs,
                                   int32_t num_heads, int32_t max_seq_len,
                                   int32_t partition_size, size_t* bytes);

/* ---------------------------------------------------------------------------
 * pa_decode without a caller-provided workspace.  The pages have no
 * counterpart to this call: it exists for callers that cannot allocate
 * device memory — an engine that reserves all device memory for its block
 * pool at start-up and forbids later allocations, or a plain C caller with no
 * caching allocator, for whom cudaMalloc/cudaFree around each decode step
 * would synchronise the device.
 *
 * Same arguments and result as pa_decode with the workspace left out: the
 * split-KV partials go to an array the library keeps in device memory, of
 * PA_NO_ALLOC_WORKSPACE_BYTES (16 MiB) per device, held until the process
 * exits.  A call whose partials need more (pa_decode_workspace_size) returns
 * PA_ERR_INVALID_ARG and launches nothing; so does every argument pa_decode
 * rejects.  The call allocates nothing.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.
 *   - Every call on a device shares the one array, which keeps the previous
 *     call's contents; its work-counter header starts at zero and every call
 *     leaves it zero, so nothing needs clearing between calls.  Calls whose
 *     work overlaps on the GPU (two streams, or two threads) race on it:
 *     order them on one stream, or use pa_decode with separate workspaces.
 * ------------------------------------------------------------------------- */
#define PA_NO_ALLOC_WORKSPACE_BYTES (16u << 20)
pa_status pa_decode_no_alloc(void* out, const void* query, const void* cache,
                             const pa_cache_desc* desc, const int32_t* block_tables,
                             int32_t max_blocks_per_seq, const int32_t* seq_lens,
                             int32_t num_seqs, int32_t num_heads, float scale,
                             int32_t max_seq_len, int32_t partition_size, void* stream);

/* ---------------------------------------------------------------------------
 * Slot mapping from block tables (host).  slots[i] is the physical slot of
 * token positions[i] of sequence seq_idx[i]:
 *   table[seq][pos / block_size] * block_size + pos % block_size
 * (tech.blogsailing.com/?p=100, section 2: a token index splits into the
 * logical block token_idx // BLOCK_SIZE and the offset token_idx % BLOCK_SIZE;
 * the block table maps the logical block to a physical one).
 * All arrays are host memory; block_tables is [num_seqs][max_blocks_per_seq].
 * Returns PA_ERR_INVALID_ARG if a sequence index falls outside [0, num_seqs),
 * a position outside its table row or a table entry outside [0, num_blocks).
 * ------------------------------------------------------------------------- */
pa_status pa_slot_mapping(const int32_t* block_tables, int32_t num_seqs,
                          int32_t max_blocks_per_seq, int32_t block_size, int32_t num_blocks,
                          const int32_t* seq_idx, const int32_t* positions, int32_t n,
                          int64_t* slots);

/* ---------------------------------------------------------------------------
 * Host block pool: the block bookkeeping that produces block tables, slot
 * mappings and copy-on-write pairs.  Host memory only; not thread-safe (one
 * pool per scheduler thread).  Rules (studying-code.tistory.com/16, sections
 * "물리적 블록 할당", "요청 완료 후 메모리 관리", the two-sample example and
 * "생성 단계에서의 Copy-on-Write"; tech.blogsailing.com/?p=100, section 3;
 * itan.pw page, section "ブロック割当のロジック"):
 *   - a prompt of n tokens takes ceil(n / block_size) blocks from the front of
 *     a FIFO free list; later tokens fill the last block and a new block is
 *     taken only when it is full;
 *   - fork shares every block of the parent and raises its reference count;
 *   - a token written into a block whose count is above 1 first moves the
 *     sequence to a new block: the old block's count drops by one and a
 *     (src, dst) pair is reported for pa_copy_blocks; a holder that finds the
 *     count at 1 writes in place;
 *   - freeing a sequence lowers the count of each block, last block first,
 *     and blocks at 0 go to the tail of the free list;
 *   - a call that runs out of free blocks returns PA_ERR_OUT_OF_BLOCKS and
 *     leaves the pool exactly as it was.
 * Sequence ids count up from 0 in creation order and are never reused.
 * ------------------------------------------------------------------------- */
typedef struct pa_pool pa_pool;

/* free_order: NULL for 0..num_blocks-1, else a permutation of the block ids
 * giving the initial order of the free list (front first). */
pa_status pa_pool_create(int32_t num_blocks, int32_t block_size, const int32_t* free_order,
                         pa_pool** out);
void pa_pool_destroy(pa_pool* pool);
/* New sequence holding num_tokens (>= 0) prompt tokens. */
pa_status pa_pool_add_seq(pa_pool* pool, int64_t num_tokens, int64_t* seq_id);
/* New sequence sharing all of parent's blocks and its length. */
pa_status pa_pool_fork(pa_pool* pool, int64_t parent, int64_t* child);
/* Reserve the slot of the sequence's next token.  cow_pair receives the
 * (src, dst) copy to run before the write, or (-1, -1). */
pa_status pa_pool_append_token(pa_pool* pool, int64_t seq, int64_t* slot, int64_t cow_pair[2]);
/* append_token for n sequences in order, all or nothing.  slots: [n];
 * cow_pairs: room for [n][2]; *num_pairs receives how many pairs were written. */
pa_status pa_pool_append_tokens(pa_pool* pool, const int64_t* seqs, int32_t n, int64_t* slots,
                                int64_t* cow_pairs, int32_t* num_pairs);
pa_status pa_pool_free_seq(pa_pool* pool, int64_t seq);
/* Block table of seq: up to cap entries into out; *num_table_blocks and
 * *seq_len receive the table length and the token count. */
pa_status pa_pool_block_table(const pa_pool* pool, int64_t seq, int32_t* out, int32_t cap,
                              int32_t* num_table_blocks, int64_t* seq_len);
/* Dense [n][max_blocks_per_seq] tables and lengths for n sequences (unused
 * entries 0), ready to copy to the device for pa_decode. */
pa_status pa_pool_fill_tables(const pa_pool* pool, const int64_t* seqs, int32_t n,
                              int32_t* block_tables, int32_t max_blocks_per_seq,
                              int32_t* seq_lens);
/* Slot of token pos (< seq_len) of seq. */
pa_status pa_pool_slot(const pa_pool* pool, int64_t seq, int64_t pos, int64_t* slot);
pa_status pa_pool_ref_count(const pa_pool* pool, int32_t block, int32_t* ref);
int32_t pa_pool_num_free(const pa_pool* pool);
/* Memory use: *tokens = sum of the GPU-resident sequences' lengths,
 * *blocks_in_use = physical blocks with a reference.  Without sharing, the KV slots allocated
 * but unused are blocks_in_use * block_size - tokens, all of them in
 * sequences' last blocks (studying-code.tistory.com/16, section "물리적 블록
 * 할당": the waste of a request stays within one block; tech.blogsailing.com/
 * ?p=100, section 2: on average BLOCK_SIZE / 2 per sequence).  Shared blocks
 * count once in blocks_in_use and once per sequence in tokens. */
pa_status pa_pool_usage(const pa_pool* pool, int64_t* tokens, int64_t* blocks_in_use);

/* ---------------------------------------------------------------------------
 * Swapping (studying-code.tistory.com/16, sections "All-or-Nothing Eviction"
 * and "스와핑(Swapping)": a preempted sequence group leaves the GPU whole, its
 * blocks go to a CPU block allocator whose size never exceeds the GPU's
 * block count, and come back when the GPU has room).
 *   pa_pool_set_cpu_blocks: size the CPU region (0 <= n <= num_blocks; only
 *     while no sequence is swapped out); its free list starts as 0..n-1.
 *   pa_pool_swap_out: move every block of the n sequences to CPU blocks,
 *     taken from the front of the CPU free list in first-use order (sequences
 *     in the given order, blocks in table order; a block shared inside the
 *     group moves once and keeps its count).  pairs (room for [blocks][2])
 *     receive (GPU block, CPU block) for pa_swap_blocks(cpu pool <- gpu
 *     pool), *num_pairs their number.  The GPU blocks are then released like
 *     pa_pool_free_seq (each sequence's last block first, to the tail of the
 *     free queue; cached prefix blocks stay cached).  PA_ERR_BAD_STATE if a
 *     sequence is unknown or already swapped, or a block is also held by a
 *     sequence outside the group; PA_ERR_OUT_OF_BLOCKS if the CPU region is
 *     too small; either way nothing changes.
 *   pa_pool_swap_in: the reverse, GPU blocks from the front of the free
 *     queue, pairs (CPU block, GPU block) for pa_swap_blocks(gpu pool <- cpu
 *     pool).
 *   A swapped-out sequence has no slots and no GPU table: append, fork,
 *   fill_tables and slot return PA_ERR_BAD_STATE; pa_pool_block_table gives
 *   its CPU block ids; pa_pool_free_seq releases its CPU blocks.
 * ------------------------------------------------------------------------- */
pa_status pa_pool_set_cpu_blocks(pa_pool* pool, int32_t num_cpu_blocks);
pa_status pa_pool_swap_out(pa_pool* pool, const int64_t* seqs, int32_t n, int64_t* pairs,
                           int32_t* num_pairs);
pa_status pa_pool_swap_in(pa_pool* pool, const int64_t* seqs, int32_t n, int64_t* pairs,
                          int32_t* num_pairs);
pa_status pa_pool_is_swapped(const pa_pool* pool, int64_t seq, int32_t* swapped);
int32_t pa_pool_num_free_cpu(const pa_pool* pool);

/* ---------------------------------------------------------------------------
 * Prefix caching on the pool (itan.pw "vLLMにおけるKVCacheマネージャーの詳細
 * 解説", sections "KVCacheManagerの処理詳細" and "プレイフィックスキャッシュの
 * 詳細": requests that begin with the same tokens share the KV blocks of that
 * prefix; only whole blocks are shared, and only a prefix that matches from
 * the first token).
 *   - A sequence created by pa_pool_add_seq_tokens knows its token ids.  Each
 *     of its full blocks gets a chained hash (the previous block's hash and
 *     the block's block_size token ids; 128 bits) and is registered under it
 *     unless another block already is.  A partly filled block has no hash.
 *   - pa_pool_add_seq_tokens shares the longest run of leading blocks whose
 *     hashes are registered, at most (num_tokens - 1) / block_size of them
 *     (the last prompt token is always computed); a shared block gains a
 *     reference and, if it was free, leaves the free queue before the
 *     request's other blocks are taken from the front of the queue.
 *     *num_cached_tokens = shared blocks * block_size: the caller writes the
 *     KV of tokens [*num_cached_tokens, num_tokens) (pa_reshape_and_cache)
 *     before any sequence reads them.  Out of blocks: nothing changes.
 *   - pa_pool_append_token_id appends like pa_pool_append_token and records
 *     the token id; a block it fills is registered.  pa_pool_append_token(s)
 *     on such a sequence drops it from prefix caching (no token id).
 *   - A freed block keeps its hash (it can still be shared) until the free
 *     queue hands it out for new content.  pa_pool_fork copies the token ids.
 *   - pa_pool_is_cached: whether the block is registered.  pa_pool_free_queue:
 *     the free queue front to back (cap entries into out; *n = its length).
 *     pa_pool_reset_prefix_cache: forget every registration (blocks, counts
 *     and tables unchanged).
 * ------------------------------------------------------------------------- */
pa_status pa_pool_add_seq_tokens(pa_pool* pool, const int32_t* tokens, int64_t num_tokens,
                                 int64_t* seq_id, int64_t* num_cached_tokens);
pa_status pa_pool_append_token_id(pa_pool* pool, int64_t seq, int32_t token, int64_t* slot,
                                  int64_t cow_pair[2]);
pa_status pa_pool_is_cached(const pa_pool* pool, int32_t block, int32_t* cached);
pa_status pa_pool_free_queue(const pa_pool* pool, int32_t* out, int32_t cap, int32_t* n);
pa_status pa_pool_reset_prefix_cache(pa_pool* pool);

/* ---------------------------------------------------------------------------
 * Diagnostics.
 * pa_get_device_error synchronises `stream`, returns the current device's
 * error word (PA_DEVERR_* bits) in *flags and clears it.  Returns
 * PA_ERR_DEVICE_CHECK when a bit was set, PA_OK otherwise.
 * ------------------------------------------------------------------------- */
pa_status pa_get_device_error(uint32_t* flags, void* stream);
const char* pa_status_string(pa_status status);

/* Timeline of the tensor-core decode, for performance work.  After a call
 * with a non-NULL device buffer, every tensor-core pa_decode of this process
 * records, per CTA and per warp (0 producer, 1 MMA issuer, 2..5 softmax
 * warpgroup), the warp's first events_per_role events as two 64-bit words
 *     buf[((cta * 6 + warp) * events_per_role + i) * 2 + 0] = SM clock (clock64)
 *     buf[((cta * 6 + warp) * events_per_role + i) * 2 + 1] = tag << 32 | argument
 * Tags (argument), producer: 9 CTA start (low 32 bits of the global timer,
 * ns), 10 work item classified (item index), 1 item published (item
 * number), 11 query tile issued (count), 12 block-table window loaded,
 * 20 stage's boxes about to be issued (stage), 2 stage's boxes issued
 * (stage), 8 producer done (items).  MMA issuer: 13 item taken (item
 * number), 3 QK issued (stage), 17 P.V inputs ready (stage), 4 PV issued
 * (stage).  Softmax warp 2: 14 item taken (item number), 15 scores ready
 * (stage), 5 scores read (stage), 24 maximum check done (stage), 25 P
 * stored to shared memory (stage), 6 P published (stage), 16 item's O read
 * from tensor memory (last stage), 7 item output written (item number);
 * warps 3..5: 19 P written
 * (warp << 16 | stage), 22 item output written (warp << 16 | item number);
 * warps 2..5: 21 item entry read (warp << 16 | item number).  The group
 * kernel of pa_decode_shared records its CTAs (flattened grid index) from
 * record 2 * SMs on: producer 30 start (global timer, ns), 31 prologue done
 * (its stages), 32 stage slot free (stage), 33 stage's boxes issued, 34 next
 * stage's blocks resolved; MMA issuer 35 QK issued (stage), 36 PV issued
 * (stage); softmax warps 2..5: 37 query rows stored, 38 stage's data
 * landed (stage), 43 masks built and scores ready (stage), 39 stage's
 * weights written to
 * tensor memory (stage), 46 O rescale stores issued (stage), 47 O rescale
 * stores done (stage), 40 P published (stage), 42 last P.V done, 41 rows or
 * partials written.
 * Entries beyond a warp's events are left as they were.  A launch whose grid
 * needs more than `bytes` records nothing.  NULL turns tracing off (the
 * default).  Host-side setting shared by all threads of the process. */
pa_status pa_set_decode_trace(void* device_buffer, size_t bytes, int32_t events_per_role);

/* Limit, in SM clock cycles, of every pipeline wait of the tensor-core decode
 * (a wait for a K/V stage, a score or output tile, a work-item slot or a free
 * buffer; the MMA issuer's wait for any of its inputs).  A wait that runs
 * out records PA_DEVERR_TIMEOUT; the CTA then stops taking work, waits for
 * its own TMA loads and MMAs in flight (those waits keep the default limit,
 * so nothing is left writing into memory the CTA gives back), frees its
 * tensor memory and returns, and the rows of the call's output are
 * undefined.  The work counters in the workspace header are left at zero,
 * so the next call with the same workspace runs normally.  0 restores the
 * default (4e9 cycles, about 2 s at 2 GHz; far beyond any healthy wait), a
 * negative value returns PA_ERR_INVALID_ARG.  The pages have no counterpart:
 * this is a test hook, which makes the timeout path run on purpose with a
 * limit of a few cycles.  Host-side setting shared by all threads of the
 * process; the CUDA-core kernel always keeps the default. */
pa_status pa_set_decode_wait_limit(int64_t cycles);
/* Library version, e.g. "0.1.0". */
const char* pa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGED_KV_CACHE_PA_H_ */
