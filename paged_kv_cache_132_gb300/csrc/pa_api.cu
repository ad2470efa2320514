// pa_api.cu -- the C ABI declared in include/pa.h: argument checks, the
// per-device error word, the library options, the partition choice, and the
// launches.
//
// Every argument error is caught here, before anything reaches the GPU; the
// kernels only report what depends on device data (ids, slots, lengths) or on
// time (a bounded wait that ran out), through the error word.
//
// Host cost per call is kept small because decode runs once per layer per
// step: per-device facts (error word address, SM count) are looked up once
// and then read with atomic loads, options are atomics initialised once from
// the environment, and the TMA descriptors of the pools are encoded once per
// (pool, shape) and cached per host thread.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <nvtx3/nvToolsExt.h>

#include <atomic>
#include <cmath>
#include <cstring>
#include <cstdint>
#include <cstdlib>
#include <mutex>

#include "../../include/pa.h"
#include "kernels.h"

namespace {

// One error word per device (a __device__ variable exists once per device
// that loads the library); read and cleared by pa_get_device_error.
__device__ int g_device_error;

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
std::atomic<int*> g_error_ptr[kMaxDevices];
std::atomic<int> g_sm_count[kMaxDevices];

int current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    return dev;
}

int* error_word(int dev) {
    int* p = g_error_ptr[dev].load(std::memory_order_acquire);
    if (p) return p;
    std::lock_guard<std::mutex> lock(g_mutex);
    p = g_error_ptr[dev].load(std::memory_order_relaxed);
    if (!p) {
        void* a = nullptr;
        if (cudaGetSymbolAddress(&a, g_device_error) != cudaSuccess) return nullptr;
        p = static_cast<int*>(a);
        g_error_ptr[dev].store(p, std::memory_order_release);
    }
    return p;
}

int l2_bytes(int dev) {
    static std::atomic<int> cached[kMaxDevices];
    int n = cached[dev].load(std::memory_order_acquire);
    if (n > 0) return n;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrL2CacheSize, dev) != cudaSuccess || n <= 0) return 0;
    cached[dev].store(n, std::memory_order_release);
    return n;
}

int sm_count(int dev) {
    int n = g_sm_count[dev].load(std::memory_order_acquire);
    if (n > 0) return n;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 0;
    g_sm_count[dev].store(n, std::memory_order_release);
    return n;
}

// ---- library options ---------------------------------------------------------
constexpr int kNumOptions = 3;
std::atomic<int> g_option[kNumOptions];
std::once_flag g_option_env_once;

bool env_is(const char* name, const char* value) {
    const char* v = std::getenv(name);
    return v && std::strcmp(v, value) == 0;
}

int option(int id) {
    std::call_once(g_option_env_once, [] {
        g_option[PA_OPT_DEBUG_CHECKS].store(env_is("PA_DEBUG_CHECKS", "1") ? 1 : 0);
        g_option[PA_OPT_DECODE_KERNEL].store(env_is("PA_DECODE_KERNEL", "simt") ? 1 : 0);
        g_option[PA_OPT_DROP_FIRST_FILL].store(env_is("PA_DEBUG_DROP_FIRST_FILL", "1") ? 1 : 0);
    });
    return g_option[id].load(std::memory_order_relaxed);
}

// An NVTX range around each entry point (free when no tool is attached).
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
};

// Wall-time limit of every wait inside a kernel (environment variable
// PA_WAIT_TIMEOUT_MS, default 2000 ms).
unsigned long long wait_limit_ns() {
    static const unsigned long long limit = [] {
        const char* s = std::getenv("PA_WAIT_TIMEOUT_MS");
        long long ms = s ? std::atoll(s) : 2000;
        if (ms <= 0) ms = 2000;
        return (unsigned long long)ms * 1000000ull;
    }();
    return limit;
}

int elem_bytes(int dtype) {
    switch (dtype) {
        case PA_F32: return 4;
        case PA_F16:
        case PA_BF16: return 2;
        default: return 0;
    }
}

bool aligned(const void* p, uintptr_t a) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_cache(const pa_cache_desc* c, pa::PoolShape* shape) {
    if (!c) return PA_ERR_INVALID_ARG;
    const int eb = elem_bytes(c->dtype);
    if (c->num_blocks <= 0 || c->num_kv_heads <= 0 || c->block_size <= 0 || c->head_dim <= 0 || eb == 0)
        return PA_ERR_INVALID_ARG;
    if (((int64_t)c->head_dim * eb) % 16 != 0) return PA_ERR_INVALID_ARG;
    shape->num_blocks = c->num_blocks;
    shape->num_kv_heads = c->num_kv_heads;
    shape->block_size = c->block_size;
    shape->head_dim = c->head_dim;
    shape->elem_bytes = eb;
    return PA_OK;
}

int max_parts_for(int max_context_len, int partition) {
    const int parts = (max_context_len + partition - 1) / partition;
    return parts < 1 ? 1 : parts;
}

bool partition_ok(int32_t partition_size) { return partition_size == 0 || (partition_size > 0 && partition_size % 64 == 0); }

// cuTensorMapEncodeTiled, fetched through the runtime so that the library
// does not link against the driver library directly.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }();
    return fn;
}

// The pool [NB][Hkv][B][d] as a 2-D tensor of NB*Hkv*B rows of d 16-bit
// elements; a box is 64 elements (128 bytes, the swizzle span) x B rows.
// With interleave (the decode kernel, head_dim 128 and 8- or 16-token blocks) the
// view is 3-D instead, one box per (block, head) tile.
bool encode_pool_map(CUtensorMap* map, const void* base, int dtype, const pa::PoolShape& shape,
                     bool interleave = true) {
    const int64_t rows = shape.num_blocks * shape.num_kv_heads * shape.block_size;
    if (rows <= 0 || rows >= (1LL << 31) || shape.head_dim % 64 != 0) return false;
    PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (!encode) return false;
    const CUtensorMapDataType type =
        dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    std::memset(map, 0, sizeof(*map));
    CUresult r;
    if (interleave && pa::interleaved_stage(shape.head_dim, shape.block_size)) {
        // [rows][2 slabs][64]: one box = one whole (block, head) tile.
        const cuuint64_t dims[3] = {64, 2, (cuuint64_t)rows};
        const cuuint64_t strides[2] = {128, 256};
        const cuuint32_t box[3] = {64, 2, (cuuint32_t)shape.block_size};
        const cuuint32_t elem_strides[3] = {1, 1, 1};
        r = encode(map, type, 3, const_cast<void*>(base), dims, strides, box, elem_strides,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {
        // [rows][d]: one box = one 64-element column slab of a tile.
        const cuuint64_t dims[2] = {(cuuint64_t)shape.head_dim, (cuuint64_t)rows};
        const cuuint64_t strides[1] = {(cuuint64_t)shape.head_dim * 2};
        const cuuint32_t box[2] = {64, (cuuint32_t)shape.block_size};
        const cuuint32_t elem_strides[2] = {1, 1};
        r = encode(map, type, 2, const_cast<void*>(base), dims, strides, box, elem_strides,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    return r == CUDA_SUCCESS;
}

// The query [num_tokens][num_heads][d] as a 3-D tensor {d, heads, tokens};
// a box is 64 elements x the G heads of one KV head x 128/G tokens, i.e. the
// 128 rows (token, grouped head) of one prefill tile, 128 bytes each.
bool encode_query_map(CUtensorMap* map, const void* base, int dtype, int num_tokens, int num_heads, int head_dim,
                      int group) {
    PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (!encode || head_dim % 64 != 0) return false;
    const CUtensorMapDataType type =
        dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    std::memset(map, 0, sizeof(*map));
    const cuuint64_t dims[3] = {(cuuint64_t)head_dim, (cuuint64_t)num_heads, (cuuint64_t)num_tokens};
    const cuuint64_t strides[2] = {(cuuint64_t)head_dim * 2, (cuuint64_t)num_heads * head_dim * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)group, (cuuint32_t)(128 / group)};
    const cuuint32_t elem_strides[3] = {1, 1, 1};
    return encode(map, type, 3, const_cast<void*>(base), dims, strides, box, elem_strides,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Cache of encoded tensor maps, per host thread (no lock).  An encoding is a
// pure function of its key (base address, shape, dtype, view), so a cached
// map is valid for as long as the key matches, whatever the caller did with
// the memory in between.  Kernel parameters are copied at launch, so the
// returned pointer is only used before the next lookup on this thread.
struct MapKey {
    int kind;  // 0: pool, 2-D view; 1: pool, decode's view; 2: query
    int dtype;
    const void* base;
    int64_t a, b, c, d;
    bool operator==(const MapKey& o) const {
        return kind == o.kind && dtype == o.dtype && base == o.base && a == o.a && b == o.b && c == o.c && d == o.d;
    }
};
struct MapSlot {
    CUtensorMap map;  // 64-byte aligned type
    MapKey key;
    bool valid;
};
constexpr int kMapSlots = 16;
thread_local MapSlot t_maps[kMapSlots];
thread_local unsigned t_map_next = 0;

const CUtensorMap* find_map(const MapKey& key) {
    for (int i = 0; i < kMapSlots; ++i)
        if (t_maps[i].valid && t_maps[i].key == key) return &t_maps[i].map;
    return nullptr;
}

MapSlot& next_map_slot() {
    MapSlot& slot = t_maps[t_map_next % kMapSlots];
    ++t_map_next;
    slot.valid = false;
    return slot;
}

const CUtensorMap* pool_map(const void* base, int dtype, const pa::PoolShape& shape, bool interleave) {
    const MapKey key{interleave ? 1 : 0, dtype, base, shape.num_blocks, shape.num_kv_heads, shape.block_size,
                     shape.head_dim};
    if (const CUtensorMap* m = find_map(key)) return m;
    MapSlot& slot = next_map_slot();
    if (!encode_pool_map(&slot.map, base, dtype, shape, interleave)) return nullptr;
    slot.key = key;
    slot.valid = true;
    return &slot.map;
}

const CUtensorMap* query_map(const void* base, int dtype, int num_tokens, int num_heads, int head_dim, int group) {
    const MapKey key{2, dtype, base, num_tokens, num_heads, head_dim, group};
    if (const CUtensorMap* m = find_map(key)) return m;
    MapSlot& slot = next_map_slot();
    if (!encode_query_map(&slot.map, base, dtype, num_tokens, num_heads, head_dim, group)) return nullptr;
    slot.key = key;
    slot.valid = true;
    return &slot.map;
}

int status_of(cudaError_t e) {
    if (e == cudaSuccess) return PA_OK;
    if (e == cudaErrorNotSupported) return PA_ERR_UNSUPPORTED;
    return PA_ERR_CUDA;
}

constexpr int kAutoPartitionSmall = 256;
constexpr int kAutoPartition = 512;

}  // namespace

namespace pa {

int decode_partition(int64_t num_seqs, int num_kv_heads, int max_context_len, int partition_size) {
    if (partition_size != 0) return partition_size;
    const int dev = current_device();
    const int sms = dev < 0 ? 0 : sm_count(dev);
    if (sms <= 0) return -1;
    // Enough independent (sequence, KV head, partition) items to keep every
    // SM busy through the tail; shorter partitions when the batch is small.
    const int64_t units = num_seqs * num_kv_heads;
    return units * max_parts_for(max_context_len, kAutoPartition) < 4LL * sms ? kAutoPartitionSmall
                                                                             : kAutoPartition;
}

size_t decode_workspace_bytes(int num_seqs, int num_heads, int max_context_len, int partition, int head_dim) {
    return decode_workspace_layout(num_seqs, num_heads, max_parts_for(max_context_len, partition), head_dim).total;
}

}  // namespace pa

extern "C" {

int pa_abi_version(void) { return PA_ABI_VERSION; }

int pa_set_option(int opt, int value) {
    if (opt < 0 || opt >= kNumOptions || (value != 0 && value != 1)) return PA_ERR_INVALID_ARG;
    option(opt);  // the environment's value first, so that it never overrides this one
    return g_option[opt].exchange(value);
}

int pa_get_option(int opt) {
    if (opt < 0 || opt >= kNumOptions) return PA_ERR_INVALID_ARG;
    return option(opt);
}

const char* pa_status_string(int status) {
    switch (status) {
        case PA_OK: return "PA_OK";
        case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG";
        case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
        case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE";
        case PA_ERR_CUDA: return "PA_ERR_CUDA";
        case PA_ERR_DEVICE_FAULT: return "PA_ERR_DEVICE_FAULT";
        case PA_ERR_DEVICE_TIMEOUT: return "PA_ERR_DEVICE_TIMEOUT";
        default: return "PA_ERR_UNKNOWN";
    }
}

int pa_reshape_and_cache(const void* key, const void* value, void* k_cache, void* v_cache,
                         const int64_t* slot_mapping, int64_t num_tokens, const pa_cache_desc* cache,
                         void* stream) {
    NvtxRange range("pa_reshape_and_cache");
    pa::PoolShape shape;
    int rc = check_cache(cache, &shape);
    if (rc != PA_OK) return rc;
    if (num_tokens < 0) return PA_ERR_INVALID_ARG;
    if (num_tokens == 0) return PA_OK;
    if (!aligned(key, 16) || !aligned(value, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(slot_mapping, 8))
        return PA_ERR_INVALID_ARG;
    const int dev = current_device();
    if (dev < 0) return PA_ERR_CUDA;
    int* err = error_word(dev);
    if (!err) return PA_ERR_CUDA;
    if (option(PA_OPT_DEBUG_CHECKS)) {
        rc = status_of(pa::launch_check_unique_slots(slot_mapping, num_tokens, err, static_cast<cudaStream_t>(stream)));
        if (rc != PA_OK) return rc;
    }
    return status_of(pa::launch_reshape_and_cache(key, value, k_cache, v_cache, slot_mapping, num_tokens, shape,
                                                  err, static_cast<cudaStream_t>(stream)));
}

size_t pa_decode_workspace_size(int32_t num_seqs, int32_t num_heads, int32_t max_context_len,
                                int32_t partition_size, int32_t head_dim) {
    if (num_seqs < 0 || num_heads <= 0 || max_context_len < 0 || head_dim <= 0 || !partition_ok(partition_size))
        return 0;
    const int part = partition_size ? partition_size : kAutoPartitionSmall;
    return pa::decode_workspace_layout(num_seqs, num_heads, max_parts_for(max_context_len, part), head_dim).total;
}

int pa_decode(void* out, int32_t out_dtype, const void* query, const void* k_cache, const void* v_cache,
              const pa_cache_desc* cache, const int32_t* block_tables, int32_t max_blocks_per_seq,
              const int32_t* context_lens, int32_t num_seqs, int32_t max_context_len, int32_t num_heads,
              int32_t num_kv_heads, float scale, int32_t partition_size, void* workspace,
              size_t workspace_bytes, void* stream) {
    NvtxRange range("pa_decode");
    pa::PoolShape shape;
    int rc = check_cache(cache, &shape);
    if (rc != PA_OK) return rc;
    if (elem_bytes(out_dtype) == 0) return PA_ERR_INVALID_ARG;
    if (num_seqs < 0 || num_heads <= 0 || num_kv_heads != cache->num_kv_heads || num_heads % num_kv_heads != 0 ||
        max_blocks_per_seq <= 0 || max_context_len < 0 || !std::isfinite(scale) || !partition_ok(partition_size))
        return PA_ERR_INVALID_ARG;
    if (num_seqs == 0) return PA_OK;
    if (!aligned(out, 16) || !aligned(query, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(block_tables, 4) || !aligned(context_lens, 4))
        return PA_ERR_INVALID_ARG;
    const int group = num_heads / num_kv_heads;
    if (!(group == 1 || group == 2 || group == 4 || group == 8)) return PA_ERR_UNSUPPORTED;
    if (!(shape.head_dim == 64 || shape.head_dim == 128)) return PA_ERR_UNSUPPORTED;
    if (!(shape.block_size == 8 || shape.block_size == 16 || shape.block_size == 32)) return PA_ERR_UNSUPPORTED;

    const int dev = current_device();
    if (dev < 0) return PA_ERR_CUDA;
    int* err = error_word(dev);
    if (!err) return PA_ERR_CUDA;

    const int part = pa::decode_partition(num_seqs, num_kv_heads, max_context_len, partition_size);
    if (part <= 0) return PA_ERR_CUDA;
    const int max_parts = max_parts_for(max_context_len, part);
    const pa::DecodeWorkspaceLayout lay = pa::decode_workspace_layout(num_seqs, num_heads, max_parts, shape.head_dim);
    if (!aligned(workspace, 256) || workspace_bytes < lay.total) return PA_ERR_WORKSPACE;
    const int64_t items_ub = (int64_t)num_seqs * max_parts * num_kv_heads;
    if (items_ub > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;

    char* ws = static_cast<char*>(workspace);
    pa::DecodeParams p{};
    p.out = out;
    p.out_dtype = out_dtype;
    p.query = query;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.block_tables = block_tables;
    p.max_blocks = max_blocks_per_seq;
    p.context_lens = context_lens;
    p.num_seqs = num_seqs;
    p.num_heads = num_heads;
    p.num_kv_heads = num_kv_heads;
    p.num_blocks = shape.num_blocks;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.partition_size = part;
    p.max_parts = max_parts;
    const int64_t table_cap = (int64_t)max_blocks_per_seq * shape.block_size;
    const int64_t part_cap = (int64_t)max_parts * part;
    const int64_t cap = table_cap < part_cap ? table_cap : part_cap;
    p.ctx_cap = (int)(cap < 0x7fffffffLL ? cap : 0x7fffffffLL);
    p.next_item = reinterpret_cast<int*>(ws + lay.next_item);
    p.num_items = reinterpret_cast<int*>(ws + lay.num_items);
    p.items = reinterpret_cast<int2*>(ws + lay.items);
    p.num_multi = reinterpret_cast<int*>(ws + lay.num_multi);
    p.multi_seqs = reinterpret_cast<int2*>(ws + lay.multi_seqs);
    p.part_ml = reinterpret_cast<float*>(ws + lay.part_ml);
    p.part_o = reinterpret_cast<float*>(ws + lay.part_o);
    p.err = err;
    p.wait_limit_ns = wait_limit_ns();
    p.debug_flags = option(PA_OPT_DROP_FIRST_FILL) ? pa::kDebugDropFirstFill : 0;
    // Every context fits one partition: no planning kernel, items are implicit.
    p.direct_items = max_parts == 1 ? (int)items_ub : 0;

    if (option(PA_OPT_DEBUG_CHECKS)) {
        rc = status_of(pa::launch_check_decode_inputs(context_lens, block_tables, num_seqs, max_blocks_per_seq,
                                                      shape.block_size, max_context_len, shape.num_blocks, err,
                                                      static_cast<cudaStream_t>(stream)));
        if (rc != PA_OK) return rc;
    }

    pa::DecodeVariant variant = option(PA_OPT_DECODE_KERNEL) ? pa::kDecodeSimt : pa::kDecodeMma;
    const CUtensorMap* tmap_k = nullptr;
    const CUtensorMap* tmap_v = nullptr;
    CUtensorMap k_map, v_map;  // copies: a second lookup may reuse the first one's cache slot
    if (cache->dtype != PA_F32 && variant == pa::kDecodeMma) {
        tmap_k = pool_map(k_cache, cache->dtype, shape, true);
        if (tmap_k) {
            k_map = *tmap_k;
            tmap_v = pool_map(v_cache, cache->dtype, shape, true);
        }
        if (tmap_v) v_map = *tmap_v;
    }
    if (!tmap_k || !tmap_v) variant = pa::kDecodeSimt;
    return status_of(pa::launch_decode(p, cache->dtype, shape.head_dim, shape.block_size, group, (int)items_ub,
                                       variant, &k_map, &v_map, static_cast<cudaStream_t>(stream)));
}

int pa_prefill(void* out, int32_t out_dtype, const void* query, const int32_t* query_start_loc,
               int32_t num_query_tokens, int32_t max_query_len, const void* k_cache, const void* v_cache,
               const pa_cache_desc* cache, const int32_t* block_tables, int32_t max_blocks_per_seq,
               const int32_t* context_lens, int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads, float scale,
               void* stream) {
    NvtxRange range("pa_prefill");
    pa::PoolShape shape;
    int rc = check_cache(cache, &shape);
    if (rc != PA_OK) return rc;
    if (elem_bytes(out_dtype) == 0) return PA_ERR_INVALID_ARG;
    if (num_seqs < 0 || num_query_tokens < 0 || max_query_len < 0 || num_heads <= 0 ||
        num_kv_heads != cache->num_kv_heads || num_heads % num_kv_heads != 0 || max_blocks_per_seq <= 0 ||
        !std::isfinite(scale) || !(scale > 0.f))
        return PA_ERR_INVALID_ARG;
    if (num_seqs == 0 || num_query_tokens == 0 || max_query_len == 0) return PA_OK;
    if (!aligned(out, 16) || !aligned(query, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(block_tables, 4) || !aligned(context_lens, 4) || !aligned(query_start_loc, 4))
        return PA_ERR_INVALID_ARG;
    const int group = num_heads / num_kv_heads;
    if (!(group == 1 || group == 2 || group == 4 || group == 8)) return PA_ERR_UNSUPPORTED;
    if (cache->dtype == PA_F32) return PA_ERR_UNSUPPORTED;
    if (!(shape.head_dim == 64 || shape.head_dim == 128)) return PA_ERR_UNSUPPORTED;
    if (!(shape.block_size == 8 || shape.block_size == 16 || shape.block_size == 32)) return PA_ERR_UNSUPPORTED;

    const int dev = current_device();
    if (dev < 0) return PA_ERR_CUDA;
    int* err = error_word(dev);
    if (!err) return PA_ERR_CUDA;

    pa::PrefillParams p{};
    p.out = out;
    p.out_dtype = out_dtype;
    p.query_start = query_start_loc;
    p.block_tables = block_tables;
    p.max_blocks = max_blocks_per_seq;
    p.context_lens = context_lens;
    p.num_seqs = num_seqs;
    p.num_tokens = num_query_tokens;
    p.max_query_len = max_query_len;
    p.num_heads = num_heads;
    p.num_kv_heads = num_kv_heads;
    p.group_shift = group == 1 ? 0 : group == 2 ? 1 : group == 4 ? 2 : 3;
    p.block_size = shape.block_size;
    p.num_blocks = shape.num_blocks;
    const int64_t cap = (int64_t)max_blocks_per_seq * shape.block_size;
    p.ctx_cap = (int)(cap < 0x7fffffffLL ? cap : 0x7fffffffLL);
    p.tile_tokens = 128 / group;
    p.tiles_per_seq = (max_query_len + p.tile_tokens - 1) / p.tile_tokens;
    // Pools (K and V) larger than L2: keep each (sequence, KV head)'s query
    // tiles together so that its keys and values are read from HBM once.
    const double pool_bytes = 2.0 * (double)shape.num_blocks * shape.num_kv_heads * shape.block_size *
                              shape.head_dim * shape.elem_bytes;
    p.tiles_adjacent = pool_bytes > (double)l2_bytes(dev) ? 1 : 0;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.err = err;
    p.wait_limit_ns = wait_limit_ns();

    CUtensorMap tmap_q, tmap_k, tmap_v;  // copies: later lookups may reuse a cache slot
    const CUtensorMap* m = query_map(query, cache->dtype, num_query_tokens, num_heads, shape.head_dim, group);
    if (!m) return PA_ERR_UNSUPPORTED;
    tmap_q = *m;
    if (!(m = pool_map(k_cache, cache->dtype, shape, false))) return PA_ERR_UNSUPPORTED;
    tmap_k = *m;
    if (!(m = pool_map(v_cache, cache->dtype, shape, false))) return PA_ERR_UNSUPPORTED;
    tmap_v = *m;
    return status_of(pa::launch_prefill(p, cache->dtype, shape.head_dim, &tmap_q, &tmap_k, &tmap_v,
                                        static_cast<cudaStream_t>(stream)));
}

int pa_copy_blocks(void* const* k_caches, void* const* v_caches, int32_t num_layers, const int64_t* src_dst_pairs,
                   int64_t num_pairs, const pa_cache_desc* cache, void* stream) {
    NvtxRange range("pa_copy_blocks");
    pa::PoolShape shape;
    int rc = check_cache(cache, &shape);
    if (rc != PA_OK) return rc;
    if (num_layers < 1 || num_layers > pa::kMaxCopyLayers || num_pairs < 0 || !k_caches || !v_caches)
        return PA_ERR_INVALID_ARG;
    if (num_pairs == 0) return PA_OK;
    if (!aligned(src_dst_pairs, 8)) return PA_ERR_INVALID_ARG;
    for (int l = 0; l < num_layers; ++l)
        if (!aligned(k_caches[l], 16) || !aligned(v_caches[l], 16)) return PA_ERR_INVALID_ARG;
    const int dev = current_device();
    if (dev < 0) return PA_ERR_CUDA;
    int* err = error_word(dev);
    if (!err) return PA_ERR_CUDA;
    if (option(PA_OPT_DEBUG_CHECKS)) {
        rc = status_of(pa::launch_check_pairs(src_dst_pairs, num_pairs, true, err, static_cast<cudaStream_t>(stream)));
        if (rc != PA_OK) return rc;
    }
    return status_of(pa::launch_copy_blocks(k_caches, v_caches, num_layers, src_dst_pairs, num_pairs, shape, err,
                                            static_cast<cudaStream_t>(stream)));
}

namespace {
// Pool memory the GPU can address: device memory, page-locked host memory
// or managed memory -- not pageable host memory.
bool gpu_addressable(const void* p) {
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();  // a failed query leaves no error behind for later calls
        return false;
    }
    return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeHost || a.type == cudaMemoryTypeManaged;
}
}  // namespace

int pa_swap_blocks(void* const* src_k, void* const* src_v, int64_t src_num_blocks, void* const* dst_k,
                   void* const* dst_v, int64_t dst_num_blocks, int32_t num_layers, const int64_t* src_dst_pairs,
                   int64_t num_pairs, const pa_cache_desc* cache, void* stream) {
    NvtxRange range("pa_swap_blocks");
    pa::PoolShape shape;
    int rc = check_cache(cache, &shape);
    if (rc != PA_OK) return rc;
    if (num_layers < 1 || num_layers > pa::kMaxCopyLayers || num_pairs < 0 || src_num_blocks <= 0 ||
        dst_num_blocks <= 0 || !src_k || !src_v || !dst_k || !dst_v)
        return PA_ERR_INVALID_ARG;
    if (num_pairs == 0) return PA_OK;
    if (!aligned(src_dst_pairs, 8)) return PA_ERR_INVALID_ARG;
    for (int l = 0; l < num_layers; ++l)
        if (!aligned(src_k[l], 16) || !aligned(src_v[l], 16) || !aligned(dst_k[l], 16) || !aligned(dst_v[l], 16))
            return PA_ERR_INVALID_ARG;
    const int dev = current_device();
    if (dev < 0) return PA_ERR_CUDA;
    if (!gpu_addressable(src_dst_pairs)) return PA_ERR_INVALID_ARG;
    for (int l = 0; l < num_layers; ++l)
        if (!gpu_addressable(src_k[l]) || !gpu_addressable(src_v[l]) || !gpu_addressable(dst_k[l]) ||
            !gpu_addressable(dst_v[l]))
            return PA_ERR_INVALID_ARG;
    int* err = error_word(dev);
    if (!err) return PA_ERR_CUDA;
    if (option(PA_OPT_DEBUG_CHECKS)) {
        bool same_pool = true;
        for (int l = 0; l < num_layers; ++l)
            if (src_k[l] != dst_k[l] || src_v[l] != dst_v[l]) same_pool = false;
        rc = status_of(pa::launch_check_pairs(src_dst_pairs, num_pairs, same_pool, err,
                                              static_cast<cudaStream_t>(stream)));
        if (rc != PA_OK) return rc;
    }
    return status_of(pa::launch_swap_blocks(src_k, src_v, src_num_blocks, dst_k, dst_v, dst_num_blocks, num_layers,
                                            src_dst_pairs, num_pairs, shape, err, static_cast<cudaStream_t>(stream)));
}

int pa_get_device_error(void* stream, int32_t* code) {
    NvtxRange range("pa_get_device_error");
    if (!code) return PA_ERR_INVALID_ARG;
    *code = 0;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return PA_ERR_CUDA;
    int word = 0;
    if (cudaMemcpyFromSymbol(&word, g_device_error, sizeof(int)) != cudaSuccess) return PA_ERR_CUDA;
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int)) != cudaSuccess) return PA_ERR_CUDA;
    *code = word;
    if (word == 0) return PA_OK;
    return (word & PA_DEVERR_TIMEOUT) ? PA_ERR_DEVICE_TIMEOUT : PA_ERR_DEVICE_FAULT;
}

}  // extern "C"
