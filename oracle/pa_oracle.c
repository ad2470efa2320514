/*
 * pa_oracle.c -- plain, slow CPU oracle for paged decode attention.
 *
 * TEST INFRASTRUCTURE ONLY (see pa_oracle.h).  Written for a reader who checks
 * it against the pages by eye: no blocking, no fusion, no reordering beyond
 * the definitions it cites.  All floating point is fp64; every stored element
 * converts to fp64 exactly.
 */
#include "pa_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------------------
 * Element decoding, from the definitions of the formats.
 *   binary32: the C float type.
 *   binary16 (IEEE 754-2008): 1 sign bit, 5 exponent bits (bias 15), 10
 *     fraction bits; exponent 0 = zero/subnormal (fraction * 2^-24),
 *     exponent 31 = infinity (fraction 0) or NaN.
 *   bfloat16: the upper 16 bits of a binary32.
 * ------------------------------------------------------------------------- */
static double half_bits_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int exponent = (h >> 10) & 0x1f;
    int fraction = h & 0x3ff;
    double magnitude;
    if (exponent == 0) {
        magnitude = ldexp((double)fraction, -24);
    } else if (exponent == 31) {
        magnitude = fraction == 0 ? INFINITY : NAN;
    } else {
        magnitude = ldexp((double)(1024 + fraction), exponent - 25);
    }
    return sign ? -magnitude : magnitude;
}

static double bf16_bits_to_double(uint16_t b)
{
    uint32_t word = (uint32_t)b << 16;
    float f;
    memcpy(&f, &word, sizeof f);
    return (double)f;
}

double orc_elem_to_double(const void *base, int64_t index, int dtype)
{
    if (dtype == ORC_F32) {
        float f;
        memcpy(&f, (const char *)base + index * 4, 4);
        return (double)f;
    }
    uint16_t bits;
    memcpy(&bits, (const char *)base + index * 2, 2);
    return dtype == ORC_F16 ? half_bits_to_double(bits) : bf16_bits_to_double(bits);
}

static int dtype_bytes(int dtype)
{
    return dtype == ORC_F32 ? 4 : (dtype == ORC_F16 || dtype == ORC_BF16) ? 2 : 0;
}

/* Element offset of (physical block, KV head, offset in block, dim 0) in a
 * pool laid out [num_blocks][num_kv_heads][block_size][head_dim]. */
static int64_t pool_offset(int64_t block, int kv_head, int offset_in_block,
                           int num_kv_heads, int block_size, int head_dim)
{
    return ((block * num_kv_heads + kv_head) * block_size + offset_in_block) * (int64_t)head_dim;
}

/* ---------------------------------------------------------------------------
 * Cache write.  "paged-attention은 도대체 뭘 최적화 하는 것일까", §17 (write_kv):
 * the token's logical position becomes (logical block, offset); the block
 * table gives the physical block; the KV goes to that block at that offset.
 * The slot number carries the result of that lookup: slot = block * B + offset.
 * ------------------------------------------------------------------------- */
int orc_reshape_and_cache(const void *key, const void *value,
                          void *k_pool, void *v_pool,
                          const int64_t *slot_mapping, int64_t num_tokens,
                          int64_t num_blocks, int num_kv_heads, int block_size,
                          int head_dim, int elem_bytes)
{
    if (num_tokens < 0 || num_blocks <= 0 || num_kv_heads <= 0 || block_size <= 0 ||
        head_dim <= 0 || elem_bytes <= 0)
        return ORC_EBADARG;
    size_t row_bytes = (size_t)head_dim * (size_t)elem_bytes;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0)
            continue;
        int64_t block = slot / block_size;
        int offset = (int)(slot % block_size);
        if (block >= num_blocks)
            return ORC_ERANGE;
        for (int h = 0; h < num_kv_heads; ++h) {
            int64_t src = ((int64_t)t * num_kv_heads + h) * head_dim;
            int64_t dst = pool_offset(block, h, offset, num_kv_heads, block_size, head_dim);
            memcpy((char *)k_pool + dst * elem_bytes, (const char *)key + src * elem_bytes, row_bytes);
            memcpy((char *)v_pool + dst * elem_bytes, (const char *)value + src * elem_bytes, row_bytes);
        }
    }
    return ORC_OK;
}

/* ---------------------------------------------------------------------------
 * Copy-on-write.  "PagedAttention 论文精读笔记", §6.1: when a writer finds the
 * reference count of its last block above one, a new physical block is
 * allocated and the old block's contents are copied into it.  One pair is one
 * such copy; it applies to the K and the V block of every layer.
 * ------------------------------------------------------------------------- */
int orc_copy_blocks(void *const *k_pools, void *const *v_pools, int num_layers,
                    const int64_t *pairs, int64_t num_pairs, int64_t num_blocks,
                    int64_t block_bytes)
{
    if (num_layers < 0 || num_pairs < 0 || num_blocks <= 0 || block_bytes <= 0)
        return ORC_EBADARG;
    for (int64_t i = 0; i < num_pairs; ++i) {
        int64_t src = pairs[2 * i];
        int64_t dst = pairs[2 * i + 1];
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks)
            return ORC_ERANGE;
        for (int layer = 0; layer < num_layers; ++layer) {
            memmove((char *)k_pools[layer] + dst * block_bytes,
                    (const char *)k_pools[layer] + src * block_bytes, (size_t)block_bytes);
            memmove((char *)v_pools[layer] + dst * block_bytes,
                    (const char *)v_pools[layer] + src * block_bytes, (size_t)block_bytes);
        }
    }
    return ORC_OK;
}

/* ---------------------------------------------------------------------------
 * Swapping.  "PagedAttention 论文精读笔记", §7.4: the blocks of an evicted
 * sequence are copied to CPU memory, and back to (possibly different) GPU
 * blocks when it is scheduled again.  Source and destination are two pools.
 * ------------------------------------------------------------------------- */
int orc_swap_blocks(void *const *src_k, void *const *src_v, int64_t src_num_blocks,
                    void *const *dst_k, void *const *dst_v, int64_t dst_num_blocks,
                    int num_layers, const int64_t *pairs, int64_t num_pairs, int64_t block_bytes)
{
    if (num_layers < 0 || num_pairs < 0 || src_num_blocks <= 0 || dst_num_blocks <= 0 || block_bytes <= 0)
        return ORC_EBADARG;
    for (int64_t i = 0; i < num_pairs; ++i) {
        int64_t src = pairs[2 * i];
        int64_t dst = pairs[2 * i + 1];
        if (src < 0 || src >= src_num_blocks || dst < 0 || dst >= dst_num_blocks)
            return ORC_ERANGE;
        for (int layer = 0; layer < num_layers; ++layer) {
            memcpy((char *)dst_k[layer] + dst * block_bytes,
                   (const char *)src_k[layer] + src * block_bytes, (size_t)block_bytes);
            memcpy((char *)dst_v[layer] + dst * block_bytes,
                   (const char *)src_v[layer] + src * block_bytes, (size_t)block_bytes);
        }
    }
    return ORC_OK;
}

/* ---------------------------------------------------------------------------
 * Gather one sequence's logical K and V for one KV head into contiguous fp64
 * rows: row j (j < ctx) comes from physical block table[j / B], offset j % B.
 * ("PagedAttention 论文精读笔记", §4.2: K_j = (k_{(j-1)B+1} .. k_{jB}) is the
 * j-th block of keys; §5.2: the block table maps logical to physical blocks.)
 * ------------------------------------------------------------------------- */
static int gather_sequence(double *Kc, double *Vc, const void *k_pool, const void *v_pool,
                           int dtype, const int32_t *table_row, int ctx, int kv_head,
                           int num_kv_heads, int block_size, int head_dim, int64_t num_blocks)
{
    for (int j = 0; j < ctx; ++j) {
        int64_t block = table_row[j / block_size];
        if (block < 0 || block >= num_blocks)
            return ORC_ERANGE;
        int64_t base = pool_offset(block, kv_head, j % block_size, num_kv_heads, block_size, head_dim);
        for (int i = 0; i < head_dim; ++i) {
            Kc[(int64_t)j * head_dim + i] = orc_elem_to_double(k_pool, base + i, dtype);
            Vc[(int64_t)j * head_dim + i] = orc_elem_to_double(v_pool, base + i, dtype);
        }
    }
    return ORC_OK;
}

/* Attention of one query vector q (head_dim doubles) over n contiguous rows.
 * "PagedAttention 论文精读笔记", §2.1:
 *   z_j = scale * q.k_j,  a_j = exp(z_j) / sum_t exp(z_t),  o = sum_j a_j v_j.
 * Subtracting M = max_j z_j from every z_j before exp leaves a_j unchanged and
 * keeps exp in range.  Outputs o (head_dim), and optionally the running max
 * M, the sum L = sum_j exp(z_j - M) and the sum of the weights a_j. */
static void attend(double *o, double *M_out, double *L_out, double *wsum_out,
                   const double *q, const double *K, const double *V, int n, int head_dim,
                   double scale, double *z)
{
    for (int i = 0; i < head_dim; ++i)
        o[i] = 0.0;
    if (n == 0) {
        if (M_out) *M_out = -INFINITY;
        if (L_out) *L_out = 0.0;
        if (wsum_out) *wsum_out = 0.0;
        return;
    }
    double M = -INFINITY;
    for (int j = 0; j < n; ++j) {
        double dot = 0.0;
        for (int i = 0; i < head_dim; ++i)
            dot += q[i] * K[(int64_t)j * head_dim + i];
        z[j] = scale * dot;
        if (z[j] > M)
            M = z[j];
    }
    double L = 0.0;
    for (int j = 0; j < n; ++j) {
        z[j] = exp(z[j] - M); /* z now holds the unnormalised weights w_j */
        L += z[j];
    }
    double wsum = 0.0;
    for (int j = 0; j < n; ++j) {
        double a = z[j] / L;
        wsum += a;
        for (int i = 0; i < head_dim; ++i)
            o[i] += a * V[(int64_t)j * head_dim + i];
    }
    if (M_out) *M_out = M;
    if (L_out) *L_out = L;
    if (wsum_out) *wsum_out = wsum;
}

static int check_decode_args(const int32_t *context_lens, int num_seqs, int max_blocks_per_seq,
                             int num_heads, int num_kv_heads, int block_size, int head_dim,
                             int64_t num_blocks, int dtype)
{
    if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || block_size <= 0 ||
        head_dim <= 0 || num_blocks <= 0 || max_blocks_per_seq < 0 || dtype_bytes(dtype) == 0)
        return ORC_EBADARG;
    if (num_heads % num_kv_heads != 0)
        return ORC_EBADARG;
    for (int s = 0; s < num_seqs; ++s) {
        if (context_lens[s] < 0 || (int64_t)context_lens[s] > (int64_t)max_blocks_per_seq * block_size)
            return ORC_EBADARG;
    }
    return ORC_OK;
}

static int max_context(const int32_t *context_lens, int num_seqs)
{
    int m = 0;
    for (int s = 0; s < num_seqs; ++s)
        if (context_lens[s] > m)
            m = context_lens[s];
    return m;
}

int orc_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* One (sequence, KV head) task of orc_decode: gather, then attend for each of
 * the G query heads that read this KV head. */
static int decode_task(double *out, double *weight_sum, const void *query,
                       const void *k_pool, const void *v_pool, int dtype,
                       const int32_t *block_tables, int max_blocks_per_seq,
                       const int32_t *context_lens, int s, int kv_head,
                       int num_heads, int num_kv_heads, int block_size, int head_dim,
                       int64_t num_blocks, double scale,
                       double *Kc, double *Vc, double *z, double *q)
{
    int group = num_heads / num_kv_heads;
    int ctx = context_lens[s];
    int rc = gather_sequence(Kc, Vc, k_pool, v_pool, dtype,
                             block_tables + (int64_t)s * max_blocks_per_seq, ctx, kv_head,
                             num_kv_heads, block_size, head_dim, num_blocks);
    if (rc != ORC_OK)
        return rc;
    for (int g = 0; g < group; ++g) {
        int h = kv_head * group + g; /* so that h / group == kv_head */
        int64_t row = (int64_t)s * num_heads + h;
        for (int i = 0; i < head_dim; ++i)
            q[i] = orc_elem_to_double(query, row * head_dim + i, dtype);
        double wsum;
        attend(out + row * head_dim, NULL, NULL, &wsum, q, Kc, Vc, ctx, head_dim, scale, z);
        if (weight_sum)
            weight_sum[row] = wsum;
    }
    return ORC_OK;
}

int orc_decode(double *out, double *weight_sum,
               const void *query, const void *k_pool, const void *v_pool, int dtype,
               const int32_t *block_tables, int max_blocks_per_seq,
               const int32_t *context_lens, int num_seqs,
               int num_heads, int num_kv_heads, int block_size, int head_dim,
               int64_t num_blocks, double scale, int num_threads)
{
    int rc = check_decode_args(context_lens, num_seqs, max_blocks_per_seq, num_heads,
                               num_kv_heads, block_size, head_dim, num_blocks, dtype);
    if (rc != ORC_OK)
        return rc;
    int max_ctx = max_context(context_lens, num_seqs);
    int64_t tasks = (int64_t)num_seqs * num_kv_heads;
    int status = ORC_OK;
#ifdef _OPENMP
    if (num_threads <= 0)
        num_threads = omp_get_max_threads();
#else
    num_threads = 1;
#endif
#pragma omp parallel num_threads(num_threads > 1 ? num_threads : 1)
    {
        size_t rows = (size_t)(max_ctx > 0 ? max_ctx : 1);
        double *Kc = malloc(rows * head_dim * sizeof(double));
        double *Vc = malloc(rows * head_dim * sizeof(double));
        double *z = malloc(rows * sizeof(double));
        double *q = malloc((size_t)head_dim * sizeof(double));
        int local = (Kc && Vc && z && q) ? ORC_OK : ORC_ENOMEM;
#pragma omp for schedule(dynamic, 1)
        for (int64_t task = 0; task < tasks; ++task) {
            if (local != ORC_OK)
                continue;
            int s = (int)(task / num_kv_heads);
            int kv_head = (int)(task % num_kv_heads);
            local = decode_task(out, weight_sum, query, k_pool, v_pool, dtype, block_tables,
                                max_blocks_per_seq, context_lens, s, kv_head, num_heads,
                                num_kv_heads, block_size, head_dim, num_blocks, scale,
                                Kc, Vc, z, q);
        }
        if (local != ORC_OK) {
#pragma omp critical
            status = local;
        }
        free(Kc);
        free(Vc);
        free(z);
        free(q);
    }
    return status;
}

int orc_decode_partitioned(double *out,
                           const void *query, const void *k_pool, const void *v_pool,
                           int dtype, const int32_t *block_tables, int max_blocks_per_seq,
                           const int32_t *context_lens, int num_seqs,
                           int num_heads, int num_kv_heads, int block_size,
                           int head_dim, int64_t num_blocks, double scale,
                           int partition_size)
{
    int rc = check_decode_args(context_lens, num_seqs, max_blocks_per_seq, num_heads,
                               num_kv_heads, block_size, head_dim, num_blocks, dtype);
    if (rc != ORC_OK)
        return rc;
    if (partition_size <= 0)
        return ORC_EBADARG;
    int group = num_heads / num_kv_heads;
    int max_ctx = max_context(context_lens, num_seqs);
    int max_parts = (max_ctx + partition_size - 1) / partition_size;
    size_t rows = (size_t)(max_ctx > 0 ? max_ctx : 1);
    double *Kc = malloc(rows * head_dim * sizeof(double));
    double *Vc = malloc(rows * head_dim * sizeof(double));
    double *z = malloc(rows * sizeof(double));
    double *q = malloc((size_t)head_dim * sizeof(double));
    double *m_p = malloc((size_t)(max_parts + 1) * sizeof(double));
    double *l_p = malloc((size_t)(max_parts + 1) * sizeof(double));
    double *o_p = malloc((size_t)(max_parts + 1) * head_dim * sizeof(double));
    int status = (Kc && Vc && z && q && m_p && l_p && o_p) ? ORC_OK : ORC_ENOMEM;
    for (int s = 0; s < num_seqs && status == ORC_OK; ++s) {
        int ctx = context_lens[s];
        int parts = (ctx + partition_size - 1) / partition_size;
        for (int kv_head = 0; kv_head < num_kv_heads && status == ORC_OK; ++kv_head) {
            status = gather_sequence(Kc, Vc, k_pool, v_pool, dtype,
                                     block_tables + (int64_t)s * max_blocks_per_seq, ctx,
                                     kv_head, num_kv_heads, block_size, head_dim, num_blocks);
            if (status != ORC_OK)
                break;
            for (int g = 0; g < group; ++g) {
                int h = kv_head * group + g;
                int64_t row = (int64_t)s * num_heads + h;
                double *o = out + row * head_dim;
                for (int i = 0; i < head_dim; ++i) {
                    q[i] = orc_elem_to_double(query, row * head_dim + i, dtype);
                    o[i] = 0.0;
                }
                /* Each partition on its own. */
                for (int p = 0; p < parts; ++p) {
                    int begin = p * partition_size;
                    int end = begin + partition_size < ctx ? begin + partition_size : ctx;
                    attend(o_p + (int64_t)p * head_dim, &m_p[p], &l_p[p], NULL, q,
                           Kc + (int64_t)begin * head_dim, Vc + (int64_t)begin * head_dim,
                           end - begin, head_dim, scale, z);
                }
                /* Merge: M = max m_p, L = sum l_p e^(m_p - M),
                 * o = sum (l_p e^(m_p - M) / L) o_p.  Empty partitions (l_p = 0)
                 * contribute nothing; no partitions (ctx = 0) leave o = 0. */
                double M = -INFINITY;
                for (int p = 0; p < parts; ++p)
                    if (l_p[p] > 0.0 && m_p[p] > M)
                        M = m_p[p];
                double L = 0.0;
                for (int p = 0; p < parts; ++p)
                    if (l_p[p] > 0.0)
                        L += l_p[p] * exp(m_p[p] - M);
                for (int p = 0; p < parts; ++p) {
                    if (l_p[p] <= 0.0)
                        continue;
                    double weight = l_p[p] * exp(m_p[p] - M) / L;
                    for (int i = 0; i < head_dim; ++i)
                        o[i] += weight * o_p[(int64_t)p * head_dim + i];
                }
            }
        }
    }
    free(Kc);
    free(Vc);
    free(z);
    free(q);
    free(m_p);
    free(l_p);
    free(o_p);
    return status;
}

/* ---------------------------------------------------------------------------
 * Prefill over a cached prefix: the same attention as orc_decode, for every
 * new token of a sequence, each over the positions up to its own.
 * ------------------------------------------------------------------------- */
int orc_prefill(double *out, const void *query, const int32_t *query_start,
                const void *k_pool, const void *v_pool, int dtype,
                const int32_t *block_tables, int max_blocks_per_seq,
                const int32_t *context_lens, int num_seqs,
                int num_heads, int num_kv_heads, int block_size, int head_dim,
                int64_t num_blocks, double scale, int num_threads)
{
    int rc = check_decode_args(context_lens, num_seqs, max_blocks_per_seq, num_heads,
                               num_kv_heads, block_size, head_dim, num_blocks, dtype);
    if (rc != ORC_OK)
        return rc;
    for (int s = 0; s < num_seqs; ++s) {
        int n = query_start[s + 1] - query_start[s];
        if (n < 0 || n > context_lens[s])
            return ORC_EBADARG;
    }
    int group = num_heads / num_kv_heads;
    int max_ctx = max_context(context_lens, num_seqs);
    int64_t tasks = (int64_t)num_seqs * num_kv_heads;
    int status = ORC_OK;
#ifdef _OPENMP
    if (num_threads <= 0)
        num_threads = omp_get_max_threads();
#else
    num_threads = 1;
#endif
#pragma omp parallel num_threads(num_threads > 1 ? num_threads : 1)
    {
        size_t rows = (size_t)(max_ctx > 0 ? max_ctx : 1);
        double *Kc = malloc(rows * head_dim * sizeof(double));
        double *Vc = malloc(rows * head_dim * sizeof(double));
        double *z = malloc(rows * sizeof(double));
        double *q = malloc((size_t)head_dim * sizeof(double));
        int local = (Kc && Vc && z && q) ? ORC_OK : ORC_ENOMEM;
#pragma omp for schedule(dynamic, 1)
        for (int64_t task = 0; task < tasks; ++task) {
            if (local != ORC_OK)
                continue;
            int s = (int)(task / num_kv_heads);
            int kv_head = (int)(task % num_kv_heads);
            int ctx = context_lens[s];
            int first = query_start[s];
            int n = query_start[s + 1] - first;
            local = gather_sequence(Kc, Vc, k_pool, v_pool, dtype,
                                    block_tables + (int64_t)s * max_blocks_per_seq, ctx, kv_head,
                                    num_kv_heads, block_size, head_dim, num_blocks);
            if (local != ORC_OK)
                continue;
            for (int i = 0; i < n; ++i) {
                int position = ctx - n + i;
                for (int g = 0; g < group; ++g) {
                    int h = kv_head * group + g;
                    int64_t row = (int64_t)(first + i) * num_heads + h;
                    for (int k = 0; k < head_dim; ++k)
                        q[k] = orc_elem_to_double(query, row * head_dim + k, dtype);
                    attend(out + row * head_dim, NULL, NULL, NULL, q, Kc, Vc, position + 1, head_dim,
                           scale, z);
                }
            }
        }
        if (local != ORC_OK) {
#pragma omp critical
            status = local;
        }
        free(Kc);
        free(Vc);
        free(z);
        free(q);
    }
    return status;
}
