/*
 * pa_oracle.c -- plain CPU oracle for the paged KV-cache hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  The tests, the smoke check and the benchmark's
 * CPU-baseline leg call this file; the library under paged_kv_cache_78_gb300/
 * never does, and this file shares no code, header, table or helper with it.
 *
 * Every floating-point value is widened to binary64 before any arithmetic
 * (bf16 and fp32 both convert to double exactly), and every formula is the
 * plain definition written out, with no blocking, fusion or reordering:
 *
 *   cache layout, one layer:  [2, num_blocks, block_size, num_kv_heads, head_size]
 *       index 0 of the first axis holds keys, index 1 values
 *       (itan.pw "vLLMにおけるKVCacheマネージャーの詳細解説", sections
 *        "ブロックアロケーションの基本概念" and "BlockPoolの生成過程": the tensor
 *        shape and "2 = key and value respectively").
 *   slot of a token:          physical_block * block_size + offset_in_block
 *       (same page, "ブロックアロケーションの基本概念": slot_mapping names the
 *        physical slot of every new token; the formula follows the block table
 *        sketch of tech.blogsailing.com/?p=100 section 2, where a token index
 *        splits into token_idx // BLOCK_SIZE and token_idx % BLOCK_SIZE).
 *   decode attention:         o = sum_j softmax_j(scale * q.k_j) v_j over the
 *       sequence's tokens j < seq_len, k_j / v_j fetched through the block table
 *       (studying-code.tistory.com/16, section "PagedAttention: 운영체제의 페이징
 *        개념에서 영감을 받은 새로운 어텐션 알고리즘"; garden.houmin.site/infra/
 *        paged-attention, section "KV Cache 管理器": q_i times the key block K_j
 *        gives scores A_ij, which then weight the value block V_j).  The pages
 *        print no softmax or scale; this is the standard scaled softmax with
 *        scale passed in.  Query head hq reads KV head hq / (Hq / Hkv).
 *   copy-on-write copy:       the whole block src is copied to dst, K and V
 *       (studying-code.tistory.com/16, section "생성 단계에서의 Copy-on-Write").
 *
 * Numbers are stored little-endian; bf16 is the upper 16 bits of an IEEE
 * binary32.  dtype code 0 = bf16 (2 bytes), 1 = fp32 (4 bytes).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

static size_t elem_size(int dtype) { return dtype == 0 ? 2 : 4; }

/* Read element idx of an array of dtype as double (exact). */
static double read_elem(const void* base, size_t idx, int dtype) {
  if (dtype == 0) {
    uint16_t h;
    memcpy(&h, (const uint8_t*)base + idx * 2, 2);
    uint32_t w = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &w, 4);
    return (double)f;
  } else {
    float f;
    memcpy(&f, (const uint8_t*)base + idx * 4, 4);
    return (double)f;
  }
}

/* Element offset of cache[kv][b][t][h][d]. */
static size_t cache_index(int kv, int64_t b, int64_t t, int h, int d, int64_t nb,
                          int bs, int hkv, int dh) {
  return ((((size_t)kv * (size_t)nb + (size_t)b) * (size_t)bs + (size_t)t) *
              (size_t)hkv + (size_t)h) * (size_t)dh + (size_t)d;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Threads of the calling thread's later parallel loops (n >= 1); timing
 * only, the results do not depend on it. */
void oracle_set_num_threads(int n) {
#ifdef _OPENMP
  if (n >= 1) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

/*
 * Write the new tokens' keys and values into the cache through slot_mapping:
 * cache[0][slot / bs][slot % bs][h][:] = key[t][h][:] and the same for value
 * at index 1.  A negative slot marks a padding token and is skipped.  Byte
 * copy: the result is bit-exact by definition.
 * Returns 0, or -1 if a slot lies beyond the pool.
 */
int oracle_reshape_and_cache(void* cache, int64_t num_blocks, int block_size,
                             int num_kv_heads, int head_size, int dtype,
                             const void* key, const void* value,
                             const int64_t* slot_mapping, int64_t num_tokens) {
  size_t es = elem_size(dtype);
  size_t row = (size_t)head_size * es;
  for (int64_t t = 0; t < num_tokens; ++t) {
    int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    if (slot >= num_blocks * (int64_t)block_size) return -1;
    int64_t b = slot / block_size;
    int64_t off = slot % block_size;
    for (int h = 0; h < num_kv_heads; ++h) {
      size_t src = ((size_t)t * (size_t)num_kv_heads + (size_t)h) * row;
      size_t dk = cache_index(0, b, off, h, 0, num_blocks, block_size,
                              num_kv_heads, head_size) * es;
      size_t dv = cache_index(1, b, off, h, 0, num_blocks, block_size,
                              num_kv_heads, head_size) * es;
      memcpy((uint8_t*)cache + dk, (const uint8_t*)key + src, row);
      memcpy((uint8_t*)cache + dv, (const uint8_t*)value + src, row);
    }
  }
  return 0;
}

/*
 * Copy-on-write block copies, in list order: for pair i, block pairs[2i]
 * (source) is copied to block pairs[2i+1] (destination), keys and values.
 * Returns 0, or -1 if an index lies beyond the pool.
 */
int oracle_copy_blocks(void* cache, int64_t num_blocks, int block_size,
                       int num_kv_heads, int head_size, int dtype,
                       const int64_t* pairs, int64_t num_pairs) {
  size_t es = elem_size(dtype);
  size_t blk = (size_t)block_size * (size_t)num_kv_heads * (size_t)head_size * es;
  for (int64_t i = 0; i < num_pairs; ++i) {
    int64_t src = pairs[2 * i], dst = pairs[2 * i + 1];
    if (src < 0 || dst < 0 || src >= num_blocks || dst >= num_blocks) return -1;
    for (int kv = 0; kv < 2; ++kv) {
      size_t s = cache_index(kv, src, 0, 0, 0, num_blocks, block_size,
                             num_kv_heads, head_size) * es;
      size_t d = cache_index(kv, dst, 0, 0, 0, num_blocks, block_size,
                             num_kv_heads, head_size) * es;
      memmove((uint8_t*)cache + d, (const uint8_t*)cache + s, blk);
    }
  }
  return 0;
}

/*
 * Scores of one (sequence, query head) over tokens [j0, j1):
 * x[j - j0] = scale * sum_d q[d] * k_j[d], k_j gathered through the block
 * table.  Returns 0, or -1 on a block id outside the pool.
 */
static int head_scores(double* x, const void* query, const void* cache,
                       int64_t num_blocks, int block_size, int num_kv_heads,
                       int head_size, int dtype, const int32_t* table_row,
                       int s, int hq, int h, int num_heads, double scale,
                       int64_t j0, int64_t j1) {
  for (int64_t j = j0; j < j1; ++j) {
    int64_t b = table_row[j / block_size];
    int64_t t = j % block_size;
    if (b < 0 || b >= num_blocks) return -1;
    double dot = 0.0;
    for (int d = 0; d < head_size; ++d) {
      double qd = read_elem(query, ((size_t)s * num_heads + hq) * head_size + d, dtype);
      double kd = read_elem(cache, cache_index(0, b, t, h, d, num_blocks, block_size,
                                               num_kv_heads, head_size), dtype);
      dot += qd * kd;
    }
    x[j - j0] = scale * dot;
  }
  return 0;
}

/*
 * Paged decode attention, two-pass softmax in binary64.
 *   out[s][hq][d] = sum_j w_j v_j[d] / sum_j w_j,
 *   w_j = exp(x_j - max_i x_i),  x_j = scale * q[s][hq] . k_j,
 * for j < seq_lens[s]; query head hq reads KV head hq / (num_heads /
 * num_kv_heads).  A sequence of length 0 gives a zero row.
 * query: [num_seqs, num_heads, head_size] of dtype; out: the same shape in
 * double.  block_tables: [num_seqs, max_blocks_per_seq].
 * Returns 0, or -1 on an index outside the pool or table.
 */
int oracle_decode(double* out, const void* query, const void* cache,
                  int64_t num_blocks, int block_size, int num_kv_heads,
                  int head_size, int dtype, const int32_t* block_tables,
                  int max_blocks_per_seq, const int32_t* seq_lens, int num_seqs,
                  int num_heads, double scale) {
  if (num_kv_heads <= 0 || num_heads % num_kv_heads != 0) return -1;
  int group = num_heads / num_kv_heads;
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (int64_t task = 0; task < (int64_t)num_seqs * num_heads; ++task) {
    int s = (int)(task / num_heads);
    int hq = (int)(task % num_heads);
    int h = hq / group;
    double* o = out + ((size_t)s * num_heads + hq) * head_size;
    int64_t len = seq_lens[s];
    for (int d = 0; d < head_size; ++d) o[d] = 0.0;
    if (len <= 0) continue;
    if ((len + block_size - 1) / block_size > max_blocks_per_seq) { bad = 1; continue; }
    const int32_t* row = block_tables + (size_t)s * max_blocks_per_seq;
    double* x = (double*)malloc(sizeof(double) * (size_t)len);
    if (!x) { bad = 1; continue; }
    if (head_scores(x, query, cache, num_blocks, block_size, num_kv_heads, head_size,
                    dtype, row, s, hq, h, num_heads, scale, 0, len) != 0) {
      bad = 1;
      free(x);
      continue;
    }
    double m = x[0];
    for (int64_t j = 1; j < len; ++j) if (x[j] > m) m = x[j];
    double den = 0.0;
    for (int64_t j = 0; j < len; ++j) {
      x[j] = exp(x[j] - m);
      den += x[j];
    }
    for (int64_t j = 0; j < len; ++j) {
      int64_t b = row[j / block_size];
      int64_t t = j % block_size;
      for (int d = 0; d < head_size; ++d) {
        double vd = read_elem(cache, cache_index(1, b, t, h, d, num_blocks, block_size,
                                                 num_kv_heads, head_size), dtype);
        o[d] += x[j] * vd;
      }
    }
    for (int d = 0; d < head_size; ++d) o[d] /= den;
    free(x);
  }
  return bad ? -1 : 0;
}

/*
 * Split-KV partials in binary64.  Tokens of sequence s are cut into
 * partitions of partition_size tokens; for partition p (tokens
 * [p*P, min(L, (p+1)*P))) and query head hq:
 *   m_p = max_j x_j,  l_p = sum_j exp(x_j - m_p),  acc_p[d] = sum_j exp(x_j - m_p) v_j[d].
 * Outputs: part_m/part_l [num_seqs, num_heads, max_parts],
 * part_acc [num_seqs, num_heads, max_parts, head_size].  Entries of
 * partitions that do not exist (p >= ceil(L/P)) are set to m = -inf, l = 0,
 * acc = 0.  Returns 0, or -1 on a bad index or if a sequence needs more than
 * max_parts partitions.
 */
int oracle_decode_partials(double* part_m, double* part_l, double* part_acc,
                           const void* query, const void* cache, int64_t num_blocks,
                           int block_size, int num_kv_heads, int head_size, int dtype,
                           const int32_t* block_tables, int max_blocks_per_seq,
                           const int32_t* seq_lens, int num_seqs, int num_heads,
                           double scale, int partition_size, int max_parts) {
  if (partition_size <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads != 0) return -1;
  int group = num_heads / num_kv_heads;
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (int64_t task = 0; task < (int64_t)num_seqs * num_heads; ++task) {
    int s = (int)(task / num_heads);
    int hq = (int)(task % num_heads);
    int h = hq / group;
    int64_t len = seq_lens[s];
    size_t base = ((size_t)s * num_heads + hq) * (size_t)max_parts;
    for (int p = 0; p < max_parts; ++p) {
      part_m[base + p] = -INFINITY;
      part_l[base + p] = 0.0;
      for (int d = 0; d < head_size; ++d) part_acc[(base + p) * head_size + d] = 0.0;
    }
    if (len <= 0) continue;
    int64_t nparts = (len + partition_size - 1) / partition_size;
    if (nparts > max_parts ||
        (len + block_size - 1) / block_size > max_blocks_per_seq) { bad = 1; continue; }
    const int32_t* row = block_tables + (size_t)s * max_blocks_per_seq;
    double* x = (double*)malloc(sizeof(double) * (size_t)partition_size);
    if (!x) { bad = 1; continue; }
    for (int64_t p = 0; p < nparts; ++p) {
      int64_t j0 = p * partition_size;
      int64_t j1 = j0 + partition_size < len ? j0 + partition_size : len;
      if (head_scores(x, query, cache, num_blocks, block_size, num_kv_heads, head_size,
                      dtype, row, s, hq, h, num_heads, scale, j0, j1) != 0) {
        bad = 1;
        break;
      }
      double m = x[0];
      for (int64_t j = j0 + 1; j < j1; ++j) if (x[j - j0] > m) m = x[j - j0];
      double l = 0.0;
      double* acc = part_acc + (base + p) * head_size;
      for (int64_t j = j0; j < j1; ++j) {
        double w = exp(x[j - j0] - m);
        l += w;
        int64_t b = row[j / block_size];
        int64_t t = j % block_size;
        for (int d = 0; d < head_size; ++d)
          acc[d] += w * read_elem(cache, cache_index(1, b, t, h, d, num_blocks, block_size,
                                                     num_kv_heads, head_size), dtype);
      }
      part_m[base + p] = m;
      part_l[base + p] = l;
    }
    free(x);
  }
  return bad ? -1 : 0;
}

/*
 * Log-sum-exp combination of split-KV partials (binary64):
 *   M = max_p m_p,  o[d] = sum_p exp(m_p - M) acc_p[d] / sum_p exp(m_p - M) l_p.
 * Partitions with m_p = -inf contribute nothing; a row with no partition
 * gives zeros.
 */
void oracle_combine_partials(double* out, const double* part_m, const double* part_l,
                             const double* part_acc, int num_seqs, int num_heads,
                             int head_size, int max_parts) {
  for (int64_t task = 0; task < (int64_t)num_seqs * num_heads; ++task) {
    size_t base = (size_t)task * (size_t)max_parts;
    double* o = out + (size_t)task * head_size;
    double mx = -INFINITY;
    for (int p = 0; p < max_parts; ++p) if (part_m[base + p] > mx) mx = part_m[base + p];
    for (int d = 0; d < head_size; ++d) o[d] = 0.0;
    if (mx == -INFINITY) continue;
    double den = 0.0;
    for (int p = 0; p < max_parts; ++p) {
      if (part_m[base + p] == -INFINITY) continue;
      double w = exp(part_m[base + p] - mx);
      den += w * part_l[base + p];
      for (int d = 0; d < head_size; ++d) o[d] += w * part_acc[(base + p) * head_size + d];
    }
    for (int d = 0; d < head_size; ++d) o[d] /= den;
  }
}
