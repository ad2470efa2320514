// kernels.h -- internal interface between the C ABI (pa_api.cu) and the
// kernel translation units.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

namespace pa {

struct PoolShape {
    int64_t num_blocks;
    int num_kv_heads;
    int block_size;
    int head_dim;
    int elem_bytes;
};

// ---- cache write / block copy (cache_ops.cu) --------------------------------
cudaError_t launch_reshape_and_cache(const void* key, const void* value, void* k_cache, void* v_cache,
                                     const int64_t* slot_mapping, int64_t num_tokens,
                                     const PoolShape& shape, int* err, cudaStream_t stream);

constexpr int kMaxCopyLayers = 256;
cudaError_t launch_copy_blocks(void* const* k_caches, void* const* v_caches, int num_layers,
                               const int64_t* pairs, int64_t num_pairs, const PoolShape& shape,
                               int* err, cudaStream_t stream);
cudaError_t launch_swap_blocks(void* const* src_k, void* const* src_v, int64_t src_num_blocks, void* const* dst_k,
                               void* const* dst_v, int64_t dst_num_blocks, int num_layers, const int64_t* pairs,
                               int64_t num_pairs, const PoolShape& shape, int* err, cudaStream_t stream);

// ---- checked mode (checks.cu): precondition pre-passes -----------------------
// Each reports violations through the error word and never traps; see the
// PA_OPT_DEBUG_CHECKS paragraph of include/pa.h.
cudaError_t launch_check_unique_slots(const int64_t* slot_mapping, int64_t num_tokens, int* err,
                                      cudaStream_t stream);
cudaError_t launch_check_pairs(const int64_t* pairs, int64_t num_pairs, bool same_pool, int* err,
                               cudaStream_t stream);
cudaError_t launch_check_decode_inputs(const int32_t* context_lens, const int32_t* block_tables, int num_seqs,
                                       int max_blocks, int block_size, int max_context_len, int64_t num_blocks,
                                       int* err, cudaStream_t stream);

// ---- decode (decode_*.cu) ----------------------------------------------------
// Partition size a pa_decode call runs with: partition_size itself when it is
// not 0, else the automatic choice for this batch on the current device;
// -1 if the device cannot be queried.  (pa_api.cu)
int decode_partition(int64_t num_seqs, int num_kv_heads, int max_context_len, int partition_size);

// Workspace bytes of a pa_decode call that runs with `partition`.  (pa_api.cu)
size_t decode_workspace_bytes(int num_seqs, int num_heads, int max_context_len, int partition, int head_dim);

// Everything one decode launch needs; passed by value as the kernel argument.
struct DecodeParams {
    void* out;
    int out_dtype;
    const void* query;
    const void* k_cache;
    const void* v_cache;
    const int32_t* block_tables;
    int max_blocks;            // block table row length
    const int32_t* context_lens;
    int num_seqs;
    int num_heads;
    int num_kv_heads;
    int64_t num_blocks;
    float scale_log2;          // scale * log2(e): scores are kept in base-2 units
    int partition_size;        // tokens per split-KV partition (multiple of the stage)
    int max_parts;             // partitions per sequence the workspace holds
    int ctx_cap;               // min(max_blocks * block_size, max_parts * partition_size)
    // workspace views
    int* next_item;            // dynamic work counter
    int* num_items;            // (sequence, partition) pairs x num_kv_heads
    int2* items;               // (sequence, partition) pairs
    int* num_multi;            // sequences with more than one partition
    int2* multi_seqs;          // [num_seqs] their (index, partition count)
    float* part_ml;            // [num_seqs * num_kv_heads * max_parts * G][2] (max, sum)
    float* part_o;             // [num_seqs * num_kv_heads * max_parts * G][head_dim]
    int* err;                  // device error word
    unsigned long long wait_limit_ns;
    int debug_flags;           // kDebugDropFirstFill: tests of the bounded waits
    // > 0: every sequence fits one partition and no planning kernel ran; item
    // i is (sequence i / num_kv_heads, partition 0), CTAs take items
    // blockIdx.x, blockIdx.x + gridDim.x, ...; the decode kernel checks the
    // context lengths itself.  0: the planning kernel wrote the work list.
    int direct_items;
};

// Test hook (environment variable PA_DEBUG_DROP_FIRST_FILL=1): every decode
// CTA leaves its first pipeline stage unfilled, so that its consumers' bounded
// wait runs out and the call reports PA_DEVERR_TIMEOUT.
constexpr int kDebugDropFirstFill = 1;

struct DecodeWorkspaceLayout {
    size_t next_item, num_items, num_multi, items, multi_seqs, part_ml, part_o, total;
};

DecodeWorkspaceLayout decode_workspace_layout(int num_seqs, int num_heads, int max_parts, int head_dim);

// Tokens per pipeline stage of the decode kernel for this head_dim/element
// size; partition sizes are multiples of it.
int decode_stage_tokens(int head_dim, int elem_bytes);

// Stage layout of the tensor-core decode kernel.  A (block, head) tile of
// head_dim 128 is two 128-byte column slabs per row.  With 8- and 16-token
// blocks a tile (2 or 4 KiB) is fetched as ONE box of a 3-D view
// [rows][2][64] -- rows interleaved in shared memory, 256 bytes apart --
// because each tensor copy has a cost of its own: 1 KiB boxes lose ~20% of
// the bandwidth, and one 4 KiB box per tile instead of two 2 KiB slab boxes
// is 0.5-2% faster.  With 32-token blocks (8 KiB tiles) each slab is its own
// box of the 2-D view [rows][d] (measured no faster interleaved) and the
// stage keeps the slabs apart.
constexpr bool interleaved_stage(int head_dim, int block_size) {
    return head_dim == 128 && (block_size == 8 || block_size == 16);
}

// Which decode consumer runs: the tensor-core one (16-bit pools, needs the
// two tensor maps) or the CUDA-core one (every dtype).
enum DecodeVariant { kDecodeMma = 0, kDecodeSimt = 1 };

// Launch the planning kernel and the decode kernel on `stream`.  tmap_k /
// tmap_v describe the K and V pools as 2-D tensors [rows = NB*Hkv*B][d] for
// the tensor-core variant (ignored by the CUDA-core one).
// Returns cudaErrorNotSupported when no kernel exists for the shape.
cudaError_t launch_decode(const DecodeParams& p, int dtype, int head_dim, int block_size, int group,
                          int grid_items_upper_bound, DecodeVariant variant, const CUtensorMap* tmap_k,
                          const CUtensorMap* tmap_v, cudaStream_t stream);

// ---- prefill over a cached prefix (prefill*.cu) -------------------------------
struct PrefillParams {
    void* out;
    int out_dtype;
    const int32_t* query_start;   // [num_seqs + 1] first query row of each sequence
    const int32_t* block_tables;
    int max_blocks;               // block table row length
    const int32_t* context_lens;  // cached tokens, the new ones included
    int num_seqs;
    int num_tokens;               // rows of the query / output arrays
    int max_query_len;            // upper bound of every sequence's new tokens
    int num_heads;
    int num_kv_heads;
    int group_shift;              // log2(num_heads / num_kv_heads)
    int block_size;
    int64_t num_blocks;
    int ctx_cap;                  // max_blocks * block_size
    int tile_tokens;              // new tokens per CTA: 128 >> group_shift
    int tiles_per_seq;            // ceil(max_query_len / tile_tokens)
    int tiles_adjacent;           // grid order: 1 = query tiles of a (sequence, KV head) adjacent
                                  // (pools larger than L2), 0 = level by level
    float scale_log2;             // scale * log2(e)
    int* err;
    unsigned long long wait_limit_ns;
};

// tmap_q: the query [num_tokens][num_heads][d] as a 3-D tensor, box
// {64, G, 128/G}; tmap_k / tmap_v: the pools as 2-D tensors [NB*Hkv*B][d],
// box {64, B}; all with the 128-byte swizzle.  dtype PA_F16 or PA_BF16.
cudaError_t launch_prefill(const PrefillParams& p, int dtype, int head_dim, const CUtensorMap* tmap_q,
                           const CUtensorMap* tmap_k, const CUtensorMap* tmap_v, cudaStream_t stream);

}  // namespace pa
