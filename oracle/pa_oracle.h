/*
 * pa_oracle.h -- plain, slow CPU oracle for paged decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link or
 * call this code; only the test suite, the smoke check and the CPU-baseline leg
 * of the benchmark use it.  It shares no code, header or table with the CUDA
 * library.
 *
 * What it computes (sources are the pages on the PagedAttention paper):
 *   - "PagedAttention 论文精读笔记", §2.1, attention equation:
 *       a_ij = exp(q_i.k_j / sqrt(d)) / sum_t exp(q_i.k_t / sqrt(d)),
 *       o_i  = sum_j a_ij v_j
 *     evaluated in fp64 over each sequence's logical KV, gathered from the
 *     physical blocks through the block table (same page, §4.2 and §5.2).
 *   - "paged-attention은 도대체 뭘 최적화 하는 것일까", §5 and §17: a token
 *     at logical position t lives in logical block t / B at offset t % B; the
 *     block table maps the logical block to a physical block.  The slot number
 *     of a new token is physical_block * B + offset.
 *   - "PagedAttention 论文精读笔记", §6.1 (copy-on-write): a shared block is
 *     duplicated by copying the whole physical block to a fresh one.
 *
 * Memory layout read here (the pages fix none; this is the library's):
 *   k_pool, v_pool : [num_blocks][num_kv_heads][block_size][head_dim]
 *   query          : [num_seqs][num_heads][head_dim]
 *   block_tables   : int32 [num_seqs][max_blocks_per_seq]
 *   context_lens   : int32 [num_seqs]
 *   slot_mapping   : int64 [num_tokens]   (slot < 0 means "skip this token")
 *   pairs          : int64 [num_pairs][2] (src, dst)
 * Element types: 0 = IEEE binary32, 1 = IEEE binary16, 2 = bfloat16.
 *
 * Every function returns 0 on success and a negative value on a bad argument
 * (ORC_EBADARG) or a reference outside the pool (ORC_ERANGE); on error the
 * outputs are left partially written.
 */
#ifndef PA_ORACLE_H
#define PA_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_F32 = 0, ORC_F16 = 1, ORC_BF16 = 2 };
enum { ORC_OK = 0, ORC_EBADARG = -1, ORC_ERANGE = -2, ORC_ENOMEM = -3 };

/* Exact value of element `index` of an array of `dtype`, as a double. */
double orc_elem_to_double(const void *base, int64_t index, int dtype);

/* Cache write: for every token t with slot_mapping[t] >= 0, copy the raw bits
 * of key[t][h][:] to k_pool[slot / B][h][slot % B][:] and value[t][h][:] to
 * v_pool likewise, for every KV head h.  key/value are [num_tokens][Hkv][d]. */
int orc_reshape_and_cache(const void *key, const void *value,
                          void *k_pool, void *v_pool,
                          const int64_t *slot_mapping, int64_t num_tokens,
                          int64_t num_blocks, int num_kv_heads, int block_size,
                          int head_dim, int elem_bytes);

/* Copy-on-write block copy: for each pair in list order and each layer,
 * copy the K block and the V block (Hkv * B * d elements each) from physical
 * block src to physical block dst.  k_pools/v_pools hold one pool per layer. */
int orc_copy_blocks(void *const *k_pools, void *const *v_pools, int num_layers,
                    const int64_t *pairs, int64_t num_pairs, int64_t num_blocks,
                    int64_t block_bytes);

/* Swap: for each pair in list order and each layer, copy the K block and the
 * V block (block_bytes each) from block src of the source pools to block dst
 * of the destination pools (a GPU pool and a host pool of the same block
 * shape, in either direction).  "PagedAttention 论文精读笔记", §7.4: evicted
 * blocks are copied to CPU memory and copied back when the sequence resumes. */
int orc_swap_blocks(void *const *src_k, void *const *src_v, int64_t src_num_blocks,
                    void *const *dst_k, void *const *dst_v, int64_t dst_num_blocks,
                    int num_layers, const int64_t *pairs, int64_t num_pairs, int64_t block_bytes);

/* Decode attention in fp64.  out is [num_seqs][num_heads][head_dim] doubles.
 * weight_sum (may be NULL) is [num_seqs][num_heads]: sum over attended tokens
 * of the normalised weights, which is 1 up to rounding (0 when ctx = 0).
 * Query head h reads KV head h / (num_heads / num_kv_heads).
 * A sequence with context length 0 gets an all-zero output.
 * num_threads <= 1 runs serially; otherwise OpenMP over (sequence, KV head). */
int orc_decode(double *out, double *weight_sum,
               const void *query, const void *k_pool, const void *v_pool, int dtype,
               const int32_t *block_tables, int max_blocks_per_seq,
               const int32_t *context_lens, int num_seqs,
               int num_heads, int num_kv_heads, int block_size, int head_dim,
               int64_t num_blocks, double scale, int num_threads);

/* The same attention, evaluated partition by partition: tokens
 * [p*P, min((p+1)*P, ctx)) form partition p.  Each partition yields its own
 * (m_p, l_p, o_p) -- running max, sum of exp(z - m_p), normalised output --
 * and the partitions are merged with
 *     M = max_p m_p,  L = sum_p l_p exp(m_p - M),
 *     o = sum_p (l_p exp(m_p - M) / L) o_p.
 * The merge is the library's reading of "combine the partial results"
 * ("PagedAttention paper review", section "How does this work?"); it is
 * mathematically equal to orc_decode, which is what the tests check. */
int orc_decode_partitioned(double *out,
                           const void *query, const void *k_pool, const void *v_pool,
                           int dtype, const int32_t *block_tables, int max_blocks_per_seq,
                           const int32_t *context_lens, int num_seqs,
                           int num_heads, int num_kv_heads, int block_size,
                           int head_dim, int64_t num_blocks, double scale,
                           int partition_size);

/* Prefill over a cached prefix ("PagedAttention 论文精读笔记", §6.3: with a
 * shared prefix cached, the prompt phase computes only the user's part; §2.1
 * attention equation).  Sequence s has n_s = query_start[s+1] - query_start[s]
 * new tokens, the last n_s of its context_lens[s] cached tokens (their K/V are
 * already in the pools).  Query row query_start[s] + i (i < n_s) sits at
 * position p = context_lens[s] - n_s + i and attends to positions 0..p.
 * out is [num_query_rows][num_heads][head_dim] doubles, num_query_rows =
 * query_start[num_seqs]; query is [num_query_rows][num_heads][head_dim]. */
int orc_prefill(double *out, const void *query, const int32_t *query_start,
                const void *k_pool, const void *v_pool, int dtype,
                const int32_t *block_tables, int max_blocks_per_seq,
                const int32_t *context_lens, int num_seqs,
                int num_heads, int num_kv_heads, int block_size, int head_dim,
                int64_t num_blocks, double scale, int num_threads);

/* Number of OpenMP threads the oracle would use for num_threads = 0 (all). */
int orc_max_threads(void);

#ifdef __cplusplus
}
#endif

#endif /* PA_ORACLE_H */
