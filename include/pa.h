/*
 * pa.h -- C ABI of the paged KV-cache decode library for GB300 (sm_103a).
 *
 * Three operations on a KV cache stored in fixed-size physical blocks, as the
 * pages on the PagedAttention paper describe it:
 *   - pa_reshape_and_cache : write new tokens' K/V into their slots
 *       ("Efficient Memory Management ... PagedAttention Review", §3-2,
 *        "fused reshape and block write"; "paged-attention은 도대체 뭘
 *        최적화 하는 것일까", §17 write_kv)
 *   - pa_decode            : exact decode attention through the block tables
 *       ("PagedAttention 论文精读笔记", §2.1 attention equation and §4.2
 *        block-wise form; Review §3-2 "fused block read and attention")
 *   - pa_copy_blocks       : copy whole blocks for copy-on-write
 *       ("PagedAttention 论文精读笔记", §6.1; Review §3-2 "fused block copy")
 *   - pa_swap_blocks       : move whole blocks between GPU and host memory
 *       ("PagedAttention 论文精读笔记", §7.4)
 *   - pa_prefill           : prompt-phase attention of new tokens over a
 *       cached prefix, causal within the new tokens
 *       ("PagedAttention 论文精读笔记", §6.3 and §5.3)
 *
 * Conventions shared by every call
 *   - Pointers named "device" are CUDA device pointers of the current device;
 *     the caller owns every buffer.  The library allocates no memory per call
 *     (its only device memory: one error word per device, and the fixed
 *     array of pa_decode_noalloc).
 *   - Device data arrays (K/V, pools, queries, outputs) must be 16-byte
 *     aligned, index arrays aligned to their element size, and the decode
 *     workspace 256-byte aligned; anything else is PA_ERR_INVALID_ARG
 *     (PA_ERR_WORKSPACE for the workspace).
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls are
 *     asynchronous on it; the caller keeps every buffer alive until the
 *     stream reaches the call.
 *   - KV pool layout: [num_blocks][num_kv_heads][block_size][head_dim], the
 *     head_dim elements of one token contiguous.  K and V are separate pools.
 *   - A slot number is physical_block * block_size + offset_in_block.
 *   - Return value: PA_OK, or a negative pa_status.  Argument errors are
 *     detected on the host before anything is launched.  Faults found by the
 *     kernels (an id outside the pool, a bounded wait that ran out) are never
 *     trapped: they set a per-device error word, read and cleared by
 *     pa_get_device_error().
 */
#ifndef PA_H
#define PA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PA_ABI_VERSION 2

typedef enum { PA_F32 = 0, PA_F16 = 1, PA_BF16 = 2 } pa_dtype;

typedef enum {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = -1,    /* bad pointer, size, alignment or shape            */
    PA_ERR_UNSUPPORTED = -2,    /* valid, but no kernel for this shape/dtype        */
    PA_ERR_WORKSPACE = -3,      /* workspace missing or smaller than required       */
    PA_ERR_CUDA = -4,           /* a CUDA runtime call or launch failed             */
    PA_ERR_DEVICE_FAULT = -5,   /* a kernel found an out-of-range id or length      */
    PA_ERR_DEVICE_TIMEOUT = -6  /* a kernel's bounded wait ran out                  */
} pa_status;

/* Bits of the device error word (pa_get_device_error). */
#define PA_DEVERR_BLOCK_ID     0x1  /* block table entry outside [0, num_blocks)           */
#define PA_DEVERR_SLOT         0x2  /* slot_mapping entry >= num_blocks * block_size       */
#define PA_DEVERR_CONTEXT_LEN  0x4  /* context_len < 0, > max_blocks_per_seq * block_size,
                                       or > the max_context_len the call was sized for    */
#define PA_DEVERR_COPY_PAIR    0x8  /* copy or swap pair id outside its pool                */
#define PA_DEVERR_TIMEOUT      0x10 /* a bounded wait inside a kernel ran out              */
/* Reported only in checked mode (PA_OPT_DEBUG_CHECKS, below): */
#define PA_DEVERR_DUP_SLOT     0x20 /* two tokens of one cache write share a slot          */
#define PA_DEVERR_PAIR_CONFLICT 0x40 /* copy/swap pairs: a destination repeated, or (same
                                        pool) a destination equal to its own or another
                                        pair's source                                      */

/*
 * Library options, process-wide (every device, every thread).  Each starts
 * from its environment variable, read once at the library's first call, and
 * can be changed between calls with pa_set_option.  Calls read the options
 * with plain atomic loads: no lock, no environment lookup per call.
 *
 *   PA_OPT_DEBUG_CHECKS (env PA_DEBUG_CHECKS=1): checked mode.  Before its
 *     main kernel, each call below also launches a pre-pass that verifies the
 *     preconditions the caller normally guarantees and reports violations
 *     through the device error word -- never by trapping:
 *       pa_reshape_and_cache  slot_mapping entries >= 0 distinct
 *                             (PA_DEVERR_DUP_SLOT)
 *       pa_copy_blocks        destinations distinct, no destination equal to
 *                             any pair's source, its own included
 *                             (PA_DEVERR_PAIR_CONFLICT)
 *       pa_swap_blocks        destinations distinct; when the source and
 *                             destination pools are the same memory, also as
 *                             pa_copy_blocks (PA_DEVERR_PAIR_CONFLICT)
 *       pa_decode(_noalloc)   0 <= context_lens[s] <= max_context_len and
 *                             <= max_blocks_per_seq * block_size
 *                             (PA_DEVERR_CONTEXT_LEN), every block id the
 *                             sequence reads in [0, num_blocks)
 *                             (PA_DEVERR_BLOCK_ID)
 *     The main kernel then runs as usual: its result is unspecified where a
 *     precondition is broken, but no access leaves the caller's buffers.
 *     The pair and slot checks compare all pairs of entries: O(n^2) work,
 *     meant for debugging, not for production batches.
 *   PA_OPT_DECODE_KERNEL (env PA_DECODE_KERNEL=simt -> 1): decode kernel for
 *     16-bit pools: 0 = tensor-core consumer (default), 1 = CUDA-core one.
 *   PA_OPT_DROP_FIRST_FILL (env PA_DEBUG_DROP_FIRST_FILL=1): test hook of the
 *     bounded waits -- every decode CTA leaves its first pipeline stage
 *     unfilled, its wait runs out and the call reports PA_DEVERR_TIMEOUT.
 */
typedef enum { PA_OPT_DEBUG_CHECKS = 0, PA_OPT_DECODE_KERNEL = 1, PA_OPT_DROP_FIRST_FILL = 2 } pa_option;

/* Sets `option` to `value` (0 or 1); returns its previous value, or
 * PA_ERR_INVALID_ARG for an unknown option or value. */
int pa_set_option(int option, int value);

/* Current value of `option`, or PA_ERR_INVALID_ARG for an unknown one. */
int pa_get_option(int option);

/* Shape of one layer's KV pool (K and V pools have the same shape). */
typedef struct {
    int64_t num_blocks;    /* physical blocks in the pool, > 0                          */
    int32_t num_kv_heads;  /* > 0                                                       */
    int32_t block_size;    /* tokens per block, > 0 (pa_decode: 8, 16 or 32)           */
    int32_t head_dim;      /* head_dim * element size must be a multiple of 16 bytes   */
    int32_t dtype;         /* pa_dtype of every element                                */
} pa_cache_desc;

/*
 * Cache write.  For every token t in [0, num_tokens) whose slot_mapping[t] is
 * >= 0, and every KV head h, copies the raw bits of key[t][h][0..d) to
 * k_cache[slot / B][h][slot % B][0..d) and value[t][h][0..d) to v_cache at
 * the same place.  Tokens with a negative slot are skipped.
 *   key, value    device, [num_tokens][num_kv_heads][head_dim], cache dtype
 *   k_cache, ...  device pools described by `cache`
 *   slot_mapping  device, int64 [num_tokens]; entries must be distinct
 * A slot >= num_blocks * B sets PA_DEVERR_SLOT and that token is skipped.
 * num_tokens = 0 is a no-op.
 */
int pa_reshape_and_cache(const void *key, const void *value, void *k_cache, void *v_cache,
                         const int64_t *slot_mapping, int64_t num_tokens,
                         const pa_cache_desc *cache, void *stream);

/*
 * Bytes of device workspace pa_decode needs for a batch of at most num_seqs
 * sequences, num_heads query heads and contexts of at most max_context_len
 * tokens, at the given partition_size (0 = automatic choice).  The workspace
 * holds the work list, the list of sequences split into several partitions,
 * and the per-partition partial results (running max, sum, normalised
 * output, fp32) that the cross-partition merge reads.
 * pa_decode resets what it needs at the start of every call, so the workspace
 * needs no initialisation; two calls in flight at once must not share one.
 * Returns 0 for invalid arguments.
 */
size_t pa_decode_workspace_size(int32_t num_seqs, int32_t num_heads, int32_t max_context_len,
                                int32_t partition_size, int32_t head_dim);

/*
 * Decode attention.  For every sequence s and query head h (KV head
 * hk = h / (num_heads / num_kv_heads)):
 *     out[s][h] = sum_j softmax_j(scale * q[s][h] . k_j) v_j,
 * over the first context_lens[s] tokens of the sequence, token j being read
 * from physical block block_tables[s][j / B] at offset j % B.  Slots past
 * context_lens[s] in the last block are never read into the sums (they may
 * hold anything, NaN included).  context_lens[s] = 0 gives out[s] = 0.
 *   out            device, [num_seqs][num_heads][head_dim], element type out_dtype
 *   query          device, [num_seqs][num_heads][head_dim], cache dtype
 *   block_tables   device, int32 [num_seqs][max_blocks_per_seq]; entries past
 *                  ceil(context_lens[s] / B) are not read
 *   context_lens   device, int32 [num_seqs]
 *   max_context_len  host, an upper bound of context_lens (sizes the work split)
 *   partition_size   0 = automatic; else the split-KV partition length, a
 *                  multiple of 64 tokens: contexts longer than it are split
 *                  into partitions computed in parallel and merged
 *   workspace      device, at least pa_decode_workspace_size(num_seqs, num_heads,
 *                  max_context_len, partition_size, head_dim) bytes
 * Supported: num_heads / num_kv_heads in {1, 2, 4, 8}, head_dim in {64, 128},
 * block_size in {8, 16, 32}, any cache dtype; else PA_ERR_UNSUPPORTED.
 */
int pa_decode(void *out, int32_t out_dtype, const void *query,
              const void *k_cache, const void *v_cache, const pa_cache_desc *cache,
              const int32_t *block_tables, int32_t max_blocks_per_seq,
              const int32_t *context_lens, int32_t num_seqs, int32_t max_context_len,
              int32_t num_heads, int32_t num_kv_heads, float scale, int32_t partition_size,
              void *workspace, size_t workspace_bytes, void *stream);

/*
 * Size of the device array pa_decode_noalloc uses as its workspace: 32 MiB
 * on every GPU where the library's code is loaded, held until the process
 * exits.  When CUDA loads modules lazily (the default since CUDA 12.2, see
 * CUDA_MODULE_LOADING), the array is committed on a device at the first
 * pa_decode_noalloc call there, not when the library is loaded.
 */
#define PA_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

/*
 * pa_decode without a caller-provided workspace, for callers that cannot
 * allocate device memory: an engine that reserved all of its GPU memory up
 * front and forbids later allocations, code that must not block on an
 * allocator or a device-wide synchronisation, or a plugin whose host owns all
 * device memory.  The paper has no counterpart of this call; it exists for
 * those callers only.  The arguments mean what they mean for pa_decode; the
 * workspace is a fixed array of PA_NOALLOC_SCRATCH_BYTES inside the library.
 *   - Nothing is allocated per call: no cudaMalloc, no cudaFree, no
 *     allocator call.
 *   - Set-up: the first call on a device (with that device current) looks
 *     up the array's device address; with lazy module loading this is also
 *     when CUDA commits the array's 32 MiB on that device.  So a caller that
 *     reserves the rest of the GPU's memory for itself makes this first call
 *     at start-up, before that reservation, and before any stream capture.
 *     A call with num_seqs = 0 (and an otherwise valid `cache`) does only
 *     this set-up and launches nothing.
 *   - A batch whose workspace exceeds the array returns PA_ERR_WORKSPACE
 *     before anything is launched.  The check uses the partition size the
 *     call will actually run (the automatic choice included), so a batch is
 *     refused only if pa_decode itself would need more than the array.
 *   - All calls share the array, which keeps the last call's contents (each
 *     call resets what it needs).  Calls whose work overlaps on the GPU --
 *     other streams or host threads -- race on it; serialise them.
 */
int pa_decode_noalloc(void *out, int32_t out_dtype, const void *query,
                      const void *k_cache, const void *v_cache, const pa_cache_desc *cache,
                      const int32_t *block_tables, int32_t max_blocks_per_seq,
                      const int32_t *context_lens, int32_t num_seqs, int32_t max_context_len,
                      int32_t num_heads, int32_t num_kv_heads, float scale, int32_t partition_size,
                      void *stream);

/*
 * Prefill over a cached prefix ("PagedAttention 论文精读笔记", §6.3: with a
 * shared prefix held in cached physical blocks, the prompt phase computes
 * only the request's own tokens; §2.1 attention equation; §5.3 prompt step).
 * Sequence s has n_s = query_start_loc[s+1] - query_start_loc[s] new tokens,
 * the LAST n_s of its context_lens[s] cached tokens: their K/V must already
 * be in the pools (pa_reshape_and_cache earlier on the stream).  New token i
 * of s sits at position context_lens[s] - n_s + i and attends to positions
 * 0 .. context_lens[s] - n_s + i:
 *   out[q][h][:] = sum_j softmax_j(scale * query[q][h] . k_j) v_j,
 *   q = query_start_loc[s] + i, query head h reading KV head h / G,
 *   G = num_heads / num_kv_heads.
 *   out               device, [num_query_tokens][num_heads][head_dim] of
 *                     out_dtype (any pa_dtype); rows not covered by a
 *                     sequence are not written
 *   query             device, [num_query_tokens][num_heads][head_dim] of
 *                     cache->dtype
 *   query_start_loc   device, int32 [num_seqs + 1], non-decreasing, last
 *                     entry <= num_query_tokens
 *   max_query_len     host, >= every n_s (sizes the launch)
 *   block_tables      device, int32 [num_seqs][max_blocks_per_seq]
 *   context_lens      device, int32 [num_seqs], n_s <= context_lens[s] <=
 *                     max_blocks_per_seq * block_size
 * scale must be > 0.  Computed on the tensor cores with fp32 accumulation;
 * the weights P enter P.V as the pools' 16-bit type (bf16: as the sum of two
 * bf16 halves).  Supported: f16 or bf16 pools, G in
 * {1, 2, 4, 8}, head_dim in {64, 128}, block_size in {8, 16, 32}; else
 * PA_ERR_UNSUPPORTED.  A sequence whose lengths break the rules above sets
 * PA_DEVERR_CONTEXT_LEN and is skipped; a bad block id sets
 * PA_DEVERR_BLOCK_ID.  No workspace.
 */
int pa_prefill(void *out, int32_t out_dtype, const void *query, const int32_t *query_start_loc,
               int32_t num_query_tokens, int32_t max_query_len,
               const void *k_cache, const void *v_cache, const pa_cache_desc *cache,
               const int32_t *block_tables, int32_t max_blocks_per_seq,
               const int32_t *context_lens, int32_t num_seqs, int32_t num_heads,
               int32_t num_kv_heads, float scale, void *stream);

/*
 * Copy-on-write block copy, one launch for all pairs and layers.  For every
 * pair i and layer l, copies the K block (num_kv_heads * B * head_dim
 * elements) of k_caches[l] from physical block pairs[i][0] to pairs[i][1],
 * and the V block of v_caches[l] likewise.
 *   k_caches, v_caches  HOST arrays of num_layers device pool pointers
 *                       (1 <= num_layers <= 256), all shaped by `cache`
 *   src_dst_pairs       device, int64 [num_pairs][2]; destinations distinct,
 *                       no destination is also a source
 * A pair outside [0, num_blocks) sets PA_DEVERR_COPY_PAIR and is skipped.
 */
int pa_copy_blocks(void *const *k_caches, void *const *v_caches, int32_t num_layers,
                   const int64_t *src_dst_pairs, int64_t num_pairs,
                   const pa_cache_desc *cache, void *stream);

/*
 * Swap blocks between two pools of the same block shape -- a GPU pool and a
 * pool in page-locked host memory -- in one launch: swap-out (GPU -> host)
 * when a sequence is preempted, swap-in (host -> GPU, possibly into other
 * blocks) when it resumes ("PagedAttention 论文精读笔记", §7.4 swapping).  For
 * every pair i and layer l, the K block src_k[l][pairs[i][0]] is copied to
 * dst_k[l][pairs[i][1]], and the V block likewise.  The GPU reads and writes
 * the host pool directly (unified addressing over the CPU-GPU link).
 *   src_k, src_v, dst_k, dst_v  HOST arrays of num_layers pool pointers (1 <=
 *                       num_layers <= 256); each pool is device memory,
 *                       page-locked host memory (cudaHostAlloc / registered)
 *                       or managed memory -- pageable host memory is
 *                       PA_ERR_INVALID_ARG
 *   src_num_blocks, dst_num_blocks  blocks in the source / destination pools
 *   src_dst_pairs       int64 [num_pairs][2], device or page-locked host;
 *                       destinations distinct
 *   cache               block shape (num_kv_heads, block_size, head_dim, dtype);
 *                       its num_blocks is not used
 * A pair outside its pool sets PA_DEVERR_COPY_PAIR and is skipped.
 */
int pa_swap_blocks(void *const *src_k, void *const *src_v, int64_t src_num_blocks,
                   void *const *dst_k, void *const *dst_v, int64_t dst_num_blocks,
                   int32_t num_layers, const int64_t *src_dst_pairs, int64_t num_pairs,
                   const pa_cache_desc *cache, void *stream);

/*
 * Synchronises `stream`, then reads and clears the current device's error
 * word into *code (a PA_DEVERR_* mask, 0 if none).  Returns PA_OK when the
 * word was 0, PA_ERR_DEVICE_TIMEOUT when the timeout bit was set,
 * PA_ERR_DEVICE_FAULT for any other bit, PA_ERR_CUDA if the sync failed.
 */
int pa_get_device_error(void *stream, int32_t *code);

/* Static, human-readable name of a pa_status value. */
const char *pa_status_string(int status);

/* PA_ABI_VERSION of the loaded library. */
int pa_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PA_H */
