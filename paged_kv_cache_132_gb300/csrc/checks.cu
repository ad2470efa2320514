// checks.cu -- pre-pass kernels of the checked mode (PA_OPT_DEBUG_CHECKS).
//
// The cache write and the block copies run their entries in parallel with no
// ordering between them, which is exact only under the preconditions the
// caller guarantees: distinct slots in one cache write, and for copy-on-write
// ("PagedAttention 论文精读笔记", §6.1) copies that are independent of each
// other -- distinct destinations, and no destination that another copy (or
// the same one) reads.  Decode reads contexts of at most the length the call
// was sized for, through block ids inside the pool.  In checked mode each
// call first runs one of these kernels, which compare the entries and set
// bits of the device error word; nothing traps, and each kernel reads only
// its n entries.
//
// The slot and pair checks compare every pair of entries (O(n^2) work, tiled
// through shared memory): cheap for decode-sized batches (hundreds of
// entries), a fraction of a millisecond for prefill-sized ones (tens of
// thousands), and meant for debugging only.
#include "common.cuh"
#include "kernels.h"

namespace pa {
namespace {

constexpr int kCheckThreads = 256;

// Entry i (one thread) against entries j > i: a repeated slot >= 0 sets
// PA_DEVERR_DUP_SLOT.
__global__ void __launch_bounds__(kCheckThreads)
check_unique_slots_kernel(const int64_t* __restrict__ slots, int64_t n, int* err) {
    __shared__ int64_t tile[kCheckThreads];
    const int64_t i = (int64_t)blockIdx.x * kCheckThreads + threadIdx.x;
    const int64_t mine = i < n ? slots[i] : -1;
    bool dup = false;
    for (int64_t base = (int64_t)blockIdx.x * kCheckThreads; base < n; base += kCheckThreads) {
        __syncthreads();
        if (base + threadIdx.x < n) tile[threadIdx.x] = slots[base + threadIdx.x];
        __syncthreads();
        const int count = (int)(n - base < kCheckThreads ? n - base : kCheckThreads);
        if (mine >= 0)
            for (int k = 0; k < count; ++k)
                if (base + k > i && tile[k] == mine) dup = true;
    }
    if (dup) set_error(err, PA_DEVERR_DUP_SLOT);
}

// Pair i (one thread) against every pair j: the same destination in two
// pairs, or -- when source and destination are the same pool -- a
// destination equal to any pair's source, its own included, sets
// PA_DEVERR_PAIR_CONFLICT.
__global__ void __launch_bounds__(kCheckThreads)
check_pairs_kernel(const int64_t* __restrict__ pairs, int64_t n, int same_pool, int* err) {
    __shared__ int64_t tile_src[kCheckThreads];
    __shared__ int64_t tile_dst[kCheckThreads];
    const int64_t i = (int64_t)blockIdx.x * kCheckThreads + threadIdx.x;
    const bool active = i < n;
    const int64_t dst = active ? pairs[2 * i + 1] : 0;
    bool conflict = false;
    for (int64_t base = 0; base < n; base += kCheckThreads) {
        __syncthreads();
        if (base + threadIdx.x < n) {
            tile_src[threadIdx.x] = pairs[2 * (base + threadIdx.x)];
            tile_dst[threadIdx.x] = pairs[2 * (base + threadIdx.x) + 1];
        }
        __syncthreads();
        const int count = (int)(n - base < kCheckThreads ? n - base : kCheckThreads);
        if (active)
            for (int k = 0; k < count; ++k) {
                if (base + k != i && tile_dst[k] == dst) conflict = true;
                if (same_pool && tile_src[k] == dst) conflict = true;
            }
    }
    if (conflict) set_error(err, PA_DEVERR_PAIR_CONFLICT);
}

// One warp per sequence: its length against the call's bound and the table's
// capacity (PA_DEVERR_CONTEXT_LEN), and every block id it reads against the
// pool (PA_DEVERR_BLOCK_ID).
__global__ void __launch_bounds__(kCheckThreads)
check_decode_inputs_kernel(const int32_t* __restrict__ context_lens, const int32_t* __restrict__ block_tables,
                           int num_seqs, int max_blocks, int block_size, int max_context_len, int64_t num_blocks,
                           int* err) {
    const int lane = threadIdx.x & 31;
    const int warps = gridDim.x * (kCheckThreads / 32);
    for (int s = blockIdx.x * (kCheckThreads / 32) + (threadIdx.x >> 5); s < num_seqs; s += warps) {
        const int ctx = context_lens[s];
        const int64_t cap = (int64_t)max_blocks * block_size;
        if (ctx < 0 || ctx > max_context_len || ctx > cap) {
            if (lane == 0) set_error(err, PA_DEVERR_CONTEXT_LEN);
        }
        int nblk = ctx <= 0 ? 0 : (ctx + block_size - 1) / block_size;
        if (nblk > max_blocks) nblk = max_blocks;
        bool bad = false;
        const int32_t* row = block_tables + (int64_t)s * max_blocks;
        for (int j = lane; j < nblk; j += 32) {
            const int32_t b = row[j];
            if (b < 0 || b >= num_blocks) bad = true;
        }
        if (__any_sync(0xffffffffu, bad) && lane == 0) set_error(err, PA_DEVERR_BLOCK_ID);
    }
}

}  // namespace

cudaError_t launch_check_unique_slots(const int64_t* slot_mapping, int64_t num_tokens, int* err,
                                      cudaStream_t stream) {
    if (num_tokens <= 0) return cudaSuccess;
    const int64_t ctas = (num_tokens + kCheckThreads - 1) / kCheckThreads;
    if (ctas > 0x7fffffffLL) return cudaErrorInvalidValue;
    check_unique_slots_kernel<<<(unsigned)ctas, kCheckThreads, 0, stream>>>(slot_mapping, num_tokens, err);
    return cudaGetLastError();
}

cudaError_t launch_check_pairs(const int64_t* pairs, int64_t num_pairs, bool same_pool, int* err,
                               cudaStream_t stream) {
    if (num_pairs <= 0) return cudaSuccess;
    const int64_t ctas = (num_pairs + kCheckThreads - 1) / kCheckThreads;
    if (ctas > 0x7fffffffLL) return cudaErrorInvalidValue;
    check_pairs_kernel<<<(unsigned)ctas, kCheckThreads, 0, stream>>>(pairs, num_pairs, same_pool ? 1 : 0, err);
    return cudaGetLastError();
}

cudaError_t launch_check_decode_inputs(const int32_t* context_lens, const int32_t* block_tables, int num_seqs,
                                       int max_blocks, int block_size, int max_context_len, int64_t num_blocks,
                                       int* err, cudaStream_t stream) {
    if (num_seqs <= 0) return cudaSuccess;
    int64_t ctas = ((int64_t)num_seqs + kCheckThreads / 32 - 1) / (kCheckThreads / 32);
    if (ctas > 4096) ctas = 4096;  // the kernel strides over the rest
    check_decode_inputs_kernel<<<(unsigned)ctas, kCheckThreads, 0, stream>>>(
        context_lens, block_tables, num_seqs, max_blocks, block_size, max_context_len, num_blocks, err);
    return cudaGetLastError();
}

}  // namespace pa
