// pa_noalloc.cu -- pa_decode_noalloc: decode attention for callers that may
// not allocate device memory.
//
// Some callers cannot call cudaMalloc or ask an allocator for a workspace:
// an engine that reserved all of its GPU memory at start-up and forbids any
// later allocation, code running where an allocation would synchronise the
// device or wait on a lock it must not take (a latency-critical serving loop,
// a callback from another runtime), or a plugin whose host framework owns all
// device memory.  This entry point takes the same inputs and outputs as
// pa_decode, but its workspace is a fixed array of device memory inside the
// library (PA_NOALLOC_SCRATCH_BYTES on every GPU where the library's code is
// loaded, held until the process exits).
//
// Its first call on a device looks up the array's device address (one
// cudaGetSymbolAddress with that device current) and caches it.  When CUDA
// loads modules lazily (the default since CUDA 12.2), that lookup is also
// what loads this file's module and commits the array's memory on the
// device, so a caller that reserves all remaining GPU memory makes the first
// call at start-up, before reserving, and before any stream capture; a call
// with num_seqs = 0 does only this set-up.  Every call shares the one array
// and the array keeps the last call's contents; pa_decode resets what it
// needs at the start of every call, so nothing has to be cleared by the
// caller.  Calls whose work overlaps on the GPU (other streams, other host
// threads) race on the array and must be serialised by the caller.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/pa.h"
#include "kernels.h"

namespace {

// The scratch array; in host code its name is only a handle for the runtime,
// never a device address.
__device__ __align__(256) unsigned char g_noalloc_scratch[PA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once
// per device), or nullptr if the lookup failed.
void* scratch_address() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_ptr[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) return nullptr;
        g_scratch_ptr[dev] = ptr;
    }
    return g_scratch_ptr[dev];
}

}  // namespace

extern "C" int pa_decode_noalloc(void* out, int32_t out_dtype, const void* query, const void* k_cache,
                                 const void* v_cache, const pa_cache_desc* cache, const int32_t* block_tables,
                                 int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t num_seqs,
                                 int32_t max_context_len, int32_t num_heads, int32_t num_kv_heads, float scale,
                                 int32_t partition_size, void* stream) {
    if (!cache) return PA_ERR_INVALID_ARG;
    // The first call on this device (any batch, num_seqs = 0 included) sets
    // up the array's address before anything else.
    void* scratch = scratch_address();
    if (!scratch) return PA_ERR_CUDA;
    if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || max_context_len < 0 || cache->head_dim <= 0 ||
        (partition_size != 0 && (partition_size < 0 || partition_size % 64 != 0)))
        return PA_ERR_INVALID_ARG;
    if (num_seqs > 0) {
        // Sized with the partition this call will run (the automatic choice
        // included), exactly as pa_decode checks its workspace.
        const int part = pa::decode_partition(num_seqs, num_kv_heads, max_context_len, partition_size);
        if (part <= 0) return PA_ERR_CUDA;
        const size_t need = pa::decode_workspace_bytes(num_seqs, num_heads, max_context_len, part, cache->head_dim);
        if (need > (size_t)PA_NOALLOC_SCRATCH_BYTES) return PA_ERR_WORKSPACE;  // batch too large for the array
    }
    return pa_decode(out, out_dtype, query, k_cache, v_cache, cache, block_tables, max_blocks_per_seq, context_lens,
                     num_seqs, max_context_len, num_heads, num_kv_heads, scale, partition_size, scratch,
                     (size_t)PA_NOALLOC_SCRATCH_BYTES, stream);
}
