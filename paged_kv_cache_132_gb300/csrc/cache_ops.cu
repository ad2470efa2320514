// cache_ops.cu -- the two kernels that maintain the paged KV cache.
//
//  * reshape_and_cache: "fused reshape and block write" ("Efficient Memory
//    Management for Large Language Model Serving with PagedAttention Review",
//    §3-2).  Each new token's K and V rows go straight from the projection
//    layout [T][Hkv][d] into their slot of the block layout
//    [NB][Hkv][B][d] in one pass.  A row (token, K|V, head) of d elements is
//    C = d * e / 16 chunks of 16 bytes, handled by C consecutive lanes, so a
//    warp reads consecutive bytes of the source and writes whole rows of the
//    destination.  The row's indices and its slot are computed once per row
//    (32-bit arithmetic), and every thread keeps four rows' loads in flight
//    before it stores, which a bandwidth-bound copy of tens of MB needs.
//    Rows whose C is not a power of two up to 32 take a plain grid-stride
//    loop with one chunk per iteration.
//  * block copies: "fused block copy for copy-on-write" (same page, §3-2;
//    "PagedAttention 论文精读笔记", §6.1), and swapping between a GPU pool and
//    a page-locked host pool (same notes, §7.4) -- the GPU reads and writes
//    host memory directly through unified addressing, so one launch moves
//    every (pair, layer, K|V) block instead of one memcpy per block.  One CTA
//    per block, each thread keeping several 16-byte loads in flight.
#include "common.cuh"
#include "kernels.h"

namespace pa {
namespace {

constexpr int kWriteThreads = 256;
constexpr int kWriteRowsInFlight = 4;

// Rows r = (t * 2 + kv) * Hkv + h of T tokens, kv = 0 for K and 1 for V.
// Thread (row group, lane c) handles chunk c of rows r0, r0 + R, ..., with R
// the rows one pass of the CTA covers; 32-bit row indices (the host checks
// 2 * T * Hkv < 2^31).
__global__ void __launch_bounds__(kWriteThreads)
reshape_and_cache_rows_kernel(const uint4* __restrict__ key, const uint4* __restrict__ value,
                              uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                              const int64_t* __restrict__ slot_mapping, int num_rows, int num_kv_heads,
                              int block_size, int chunks_log2, int64_t num_slots, int* err) {
    pdl_launch_dependents();  // as in the general kernel below
    const int chunks = 1 << chunks_log2;
    const int c = threadIdx.x & (chunks - 1);
    const int rows_per_pass = kWriteThreads >> chunks_log2;
    const int first = blockIdx.x * rows_per_pass * kWriteRowsInFlight + (threadIdx.x >> chunks_log2);
    uint4 data[kWriteRowsInFlight];
    int64_t slot[kWriteRowsInFlight];
    int th[kWriteRowsInFlight];  // t * 2 + kv
    int head[kWriteRowsInFlight];
    // Loads of the source chunks and of the slots first, all independent...
#pragma unroll
    for (int u = 0; u < kWriteRowsInFlight; ++u) {
        const int r = first + u * rows_per_pass;
        slot[u] = -1;
        if (r < num_rows) {
            th[u] = (int)((unsigned)r / (unsigned)num_kv_heads);
            head[u] = r - th[u] * num_kv_heads;
            const int t = th[u] >> 1;
            const uint4* src = (th[u] & 1) ? value : key;
            data[u] = __ldcs(src + (((int64_t)t * num_kv_heads + head[u]) << chunks_log2) + c);
            slot[u] = __ldg(slot_mapping + t);
        }
    }
    // ...then the stores.
#pragma unroll
    for (int u = 0; u < kWriteRowsInFlight; ++u) {
        const int64_t sl = slot[u];
        if (sl < 0) continue;  // padding token (or no row): nothing to store
        if (sl >= num_slots) {
            if (c == 0 && head[u] == 0 && !(th[u] & 1)) set_error(err, PA_DEVERR_SLOT);
            continue;
        }
        int64_t block, offset;
        if (num_slots <= 0x7fffffffLL) {
            block = (int64_t)((unsigned)sl / (unsigned)block_size);
            offset = sl - block * block_size;
        } else {
            block = sl / block_size;
            offset = sl - block * block_size;
        }
        uint4* dst = (th[u] & 1) ? v_cache : k_cache;
        dst[((((block * num_kv_heads + head[u]) * block_size + offset)) << chunks_log2) + c] = data[u];
    }
}

__global__ void __launch_bounds__(kWriteThreads)
reshape_and_cache_kernel(const uint4* __restrict__ key, const uint4* __restrict__ value,
                         uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                         const int64_t* __restrict__ slot_mapping, int64_t num_tokens, int num_kv_heads,
                         int block_size, int chunks_per_row, int64_t num_slots, int* err) {
    // A kernel launched after this one as a programmatic dependent (the
    // decode planning kernel) may start now; it waits for this grid's
    // completion before anything it launches reads the pools.
    pdl_launch_dependents();
    // Thread index -> (token t, K|V, head h, 16-byte chunk c), chunk fastest.
    const int64_t total = num_tokens * 2 * num_kv_heads * chunks_per_row;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += stride) {
        const int c = (int)(idx % chunks_per_row);
        int64_t rest = idx / chunks_per_row;
        const int h = (int)(rest % num_kv_heads);
        rest /= num_kv_heads;
        const int is_value = (int)(rest & 1);
        const int64_t t = rest >> 1;
        const int64_t slot = __ldg(slot_mapping + t);
        if (slot < 0) continue;  // padding token: nothing to store
        if (slot >= num_slots) {
            if (h == 0 && c == 0 && !is_value) set_error(err, PA_DEVERR_SLOT);
            continue;
        }
        const int64_t block = slot / block_size;
        const int64_t offset = slot - block * block_size;
        const uint4* src = (is_value ? value : key) + ((t * num_kv_heads + h) * chunks_per_row + c);
        uint4* dst = (is_value ? v_cache : k_cache) +
                     (((block * num_kv_heads + h) * block_size + offset) * chunks_per_row + c);
        *dst = __ldg(src);
    }
}

// Source and destination pools of a block copy: the same pools for
// copy-on-write, a GPU pool and a page-locked host pool for swapping.
struct BlockPools {
    const uint4* src_k[kMaxCopyLayers];
    const uint4* src_v[kMaxCopyLayers];
    uint4* dst_k[kMaxCopyLayers];
    uint4* dst_v[kMaxCopyLayers];
};

constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 8;

__global__ void __launch_bounds__(kCopyThreads)
block_copy_kernel(const __grid_constant__ BlockPools pools, int num_layers, const int64_t* __restrict__ pairs,
                  int64_t src_num_blocks, int64_t dst_num_blocks, int64_t vecs_per_block, int* err) {
    // blockIdx.x -> (pair, layer, K|V), K|V fastest.
    const int64_t id = blockIdx.x;
    const int is_value = (int)(id & 1);
    const int layer = (int)((id >> 1) % num_layers);
    const int64_t pair = (id >> 1) / num_layers;
    const int64_t src = __ldg(pairs + 2 * pair);
    const int64_t dst = __ldg(pairs + 2 * pair + 1);
    if (src < 0 || src >= src_num_blocks || dst < 0 || dst >= dst_num_blocks) {
        if (threadIdx.x == 0 && layer == 0 && !is_value) set_error(err, PA_DEVERR_COPY_PAIR);
        return;
    }
    const uint4* from = (is_value ? pools.src_v[layer] : pools.src_k[layer]) + src * vecs_per_block;
    uint4* to = (is_value ? pools.dst_v[layer] : pools.dst_k[layer]) + dst * vecs_per_block;
    // Several 16-byte loads in flight per thread before the stores (the
    // source may be host memory, far away).
    for (int64_t i0 = threadIdx.x; i0 < vecs_per_block; i0 += (int64_t)kCopyThreads * kCopyUnroll) {
        uint4 buf[kCopyUnroll];
#pragma unroll
        for (int u = 0; u < kCopyUnroll; ++u) {
            const int64_t i = i0 + (int64_t)u * kCopyThreads;
            if (i < vecs_per_block) buf[u] = __ldcs(from + i);
        }
#pragma unroll
        for (int u = 0; u < kCopyUnroll; ++u) {
            const int64_t i = i0 + (int64_t)u * kCopyThreads;
            if (i < vecs_per_block) to[i] = buf[u];
        }
    }
}

cudaError_t launch_block_copy(const BlockPools& pools, int num_layers, const int64_t* pairs, int64_t num_pairs,
                              int64_t src_num_blocks, int64_t dst_num_blocks, const PoolShape& shape, int* err,
                              cudaStream_t stream) {
    if (num_pairs == 0) return cudaSuccess;
    const int64_t block_bytes =
        (int64_t)shape.num_kv_heads * shape.block_size * shape.head_dim * shape.elem_bytes;
    const int64_t ctas = num_pairs * num_layers * 2;
    if (ctas > 0x7fffffffLL) return cudaErrorInvalidValue;
    block_copy_kernel<<<(unsigned)ctas, kCopyThreads, 0, stream>>>(pools, num_layers, pairs, src_num_blocks,
                                                                    dst_num_blocks, block_bytes / 16, err);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_reshape_and_cache(const void* key, const void* value, void* k_cache, void* v_cache,
                                     const int64_t* slot_mapping, int64_t num_tokens,
                                     const PoolShape& shape, int* err, cudaStream_t stream) {
    if (num_tokens == 0) return cudaSuccess;
    const int chunks = shape.head_dim * shape.elem_bytes / 16;
    const int64_t rows = num_tokens * 2 * shape.num_kv_heads;
    const bool pow2 = (chunks & (chunks - 1)) == 0 && chunks <= 32;
    if (pow2 && rows < 0x7fffffffLL - kWriteThreads * kWriteRowsInFlight) {
        int log2c = 0;
        while ((1 << log2c) < chunks) ++log2c;
        const int64_t rows_per_cta = (int64_t)(kWriteThreads >> log2c) * kWriteRowsInFlight;
        const int64_t ctas = (rows + rows_per_cta - 1) / rows_per_cta;
        reshape_and_cache_rows_kernel<<<(unsigned)ctas, kWriteThreads, 0, stream>>>(
            static_cast<const uint4*>(key), static_cast<const uint4*>(value), static_cast<uint4*>(k_cache),
            static_cast<uint4*>(v_cache), slot_mapping, (int)rows, shape.num_kv_heads, shape.block_size, log2c,
            shape.num_blocks * shape.block_size, err);
        return cudaGetLastError();
    }
    const int64_t total = rows * chunks;
    int64_t blocks = (total + kWriteThreads - 1) / kWriteThreads;
    if (blocks > 65536) blocks = 65536;  // grid-stride beyond this
    reshape_and_cache_kernel<<<(unsigned)blocks, kWriteThreads, 0, stream>>>(
        static_cast<const uint4*>(key), static_cast<const uint4*>(value), static_cast<uint4*>(k_cache),
        static_cast<uint4*>(v_cache), slot_mapping, num_tokens, shape.num_kv_heads, shape.block_size, chunks,
        shape.num_blocks * shape.block_size, err);
    return cudaGetLastError();
}

cudaError_t launch_copy_blocks(void* const* k_caches, void* const* v_caches, int num_layers,
                               const int64_t* pairs, int64_t num_pairs, const PoolShape& shape,
                               int* err, cudaStream_t stream) {
    BlockPools pools{};
    for (int l = 0; l < num_layers; ++l) {
        pools.src_k[l] = pools.dst_k[l] = static_cast<uint4*>(k_caches[l]);
        pools.src_v[l] = pools.dst_v[l] = static_cast<uint4*>(v_caches[l]);
    }
    return launch_block_copy(pools, num_layers, pairs, num_pairs, shape.num_blocks, shape.num_blocks, shape, err,
                             stream);
}

cudaError_t launch_swap_blocks(void* const* src_k, void* const* src_v, int64_t src_num_blocks, void* const* dst_k,
                               void* const* dst_v, int64_t dst_num_blocks, int num_layers, const int64_t* pairs,
                               int64_t num_pairs, const PoolShape& shape, int* err, cudaStream_t stream) {
    BlockPools pools{};
    for (int l = 0; l < num_layers; ++l) {
        pools.src_k[l] = static_cast<const uint4*>(src_k[l]);
        pools.src_v[l] = static_cast<const uint4*>(src_v[l]);
        pools.dst_k[l] = static_cast<uint4*>(dst_k[l]);
        pools.dst_v[l] = static_cast<uint4*>(dst_v[l]);
    }
    return launch_block_copy(pools, num_layers, pairs, num_pairs, src_num_blocks, dst_num_blocks, shape, err,
                             stream);
}

}  // namespace pa
