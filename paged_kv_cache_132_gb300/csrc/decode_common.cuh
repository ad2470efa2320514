// decode_common.cuh -- the parts of the decode kernels that do not depend on
// how the scores are computed: the work-item producer warp with its
// shared-memory stage ring, and the end-of-item merge.
//
// What the kernels compute: "PagedAttention 论文精读笔记", §2.1 (attention
// equation) in the block-wise order of §4.2: a sequence's keys and values are
// read one physical block at a time, located through the block table (§5.2),
// and the per-block results are combined exactly ("PagedAttention paper
// review", "How does this work?") by the running-max / running-sum softmax.
// A context longer than the partition size is split into partitions that
// different CTAs compute; each stores its (max, sum, normalised output) and
// the reduce kernel (decode.cu) merges them.  Scores are kept in base-2 units
// (scale * log2 e is folded in).
//
// CTA structure (persistent, one or two CTAs per SM):
//   producer warp: takes (sequence, partition, KV head) items from a device
//     counter, reads the block table, and copies each (block, head) K and V
//     tile -- one contiguous [B][d] slab of the pool -- into a 3-stage
//     shared-memory ring guarded by mbarriers.  The copy engine does the
//     gathering ("warp-level block read" with coalesced access in
//     "Efficient Memory Management ... Review", §3-2).
//   consumer warps: each takes a quarter of a stage's tokens and keeps its own
//     running max / sum / output for the G query heads of the KV head (GQA
//     grouping on the CTA).  At an item's end they leave their state in a
//     shared-memory slot and go on with the next item.
//   merge warp: merges the consumer warps' states of a finished item and
//     stores the output, or the partition's partial for the reduce kernel.
// Every wait is bounded by a wall-time limit; a wait that runs out sets
// PA_DEVERR_TIMEOUT, and the CTA drains its copies and returns.
#pragma once

#include <cuda.h>

#include "common.cuh"
#include "kernels.h"

namespace pa {

constexpr int kDecodeConsumerWarps = 4;
constexpr int kDecodeStages = 3;
constexpr unsigned kFullMask = 0xffffffffu;

// Tokens per pipeline stage: K+V of a stage within 32 KiB, at most 64 tokens.
__host__ __device__ constexpr int stage_tokens_for_row(int row_bytes) {
    return (32768 / (2 * row_bytes)) < 64 ? (32768 / (2 * row_bytes)) : 64;
}

struct StageMeta {
    int item;    // -1: no more work
    int seq;
    int kv_head;
    int part;
    int nparts;
    int t0;      // first token of this stage
    int te;      // end of the item's tokens (exclusive)
    int first;   // first stage of the item
    int last;    // last stage of the item
};

// Compile-time shape of one decode kernel instance.
template <typename T, int D, int BS, int G>
struct DecodeShape {
    static constexpr int E = sizeof(T);
    static constexpr int NCW = kDecodeConsumerWarps;
    static constexpr int NSTAGE = kDecodeStages;
    static constexpr int PRODUCER_WARP = NCW;         // fills the stage ring
    static constexpr int MERGE_WARP = NCW + 1;        // merges and stores finished items
    static constexpr int THREADS = (NCW + 2) * 32;
    static constexpr int ROW = D * E;                 // bytes of one token's row
    static constexpr int STAGE_TOK = stage_tokens_for_row(ROW);
    static_assert(STAGE_TOK % BS == 0, "a stage holds whole blocks");
    static constexpr int BPS = STAGE_TOK / BS;        // blocks per stage
    static_assert(BPS <= 31, "one producer lane per block; lane 31 copies q");
    static constexpr int TPW = STAGE_TOK / NCW;       // tokens per consumer warp per stage
    static constexpr int TILE = BS * ROW;             // bytes of one (block, head) slab
    static constexpr int KV_STAGE_BYTES = STAGE_TOK * ROW;
    static constexpr int QBYTES = G * D * E;
    static_assert(QBYTES % 16 == 0, "the q tile is one bulk copy");
    static constexpr bool INTERLEAVED = interleaved_stage(D, BS);
    static_assert(D % 128 == 0 || D == 64, "the merge warp stores 4 consecutive dims per lane");

    struct Smem {
        alignas(1024) uint8_t kv[NSTAGE][2][KV_STAGE_BYTES];
        alignas(16) uint8_t q[NSTAGE][QBYTES];
        alignas(16) float mo[NCW][G][D];   // per-warp output accumulators of the finished item
        float mm[NCW][G];      // per-warp running max (base-2 units)
        float ml[NCW][G];      // per-warp running sum
        StageMeta meta[NSTAGE];
        StageMeta merge_meta;  // the finished item handed to the merge warp
        uint64_t full[NSTAGE];
        uint64_t empty[NSTAGE];
        uint64_t merge_full;   // consumers -> merge warp: the slot holds an item
        uint64_t merge_free;   // merge warp -> consumers: the slot may be reused
        int abort_flag;
    };
    // 1 KiB of slack to align the dynamic shared memory base to 1024 bytes.
    static constexpr int SMEM_BYTES = sizeof(Smem) + 1024;
};

template <class Smem>
__device__ inline Smem& decode_smem(uint8_t* raw) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(raw);
    return *reinterpret_cast<Smem*>((a + 1023) & ~uintptr_t(1023));
}

template <class Smem>
__device__ inline void decode_smem_init(Smem& sm, int stages, int consumer_warps) {
    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], consumer_warps);
        }
        mbar_init(&sm.merge_full, consumer_warps);
        mbar_init(&sm.merge_free, 1);
        sm.abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    // The planning kernel before this one writes the work list; wait for it
    // (the set-up above overlapped with it).
    pdl_wait_prerequisites();
}

// L2 policy for data read exactly once (the KV tiles): evict first, so that
// the stream does not push out what is read again (partials, tables).
__device__ inline uint64_t l2_evict_first_policy() {
    uint64_t policy;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
    return policy;
}

// 2-D tiled TMA load of one box into shared memory, completed on `bar`, with
// an L2 cache policy.
__device__ inline void tma_load_2d(void* smem_dst, const CUtensorMap* map, int x, int y, uint64_t* bar,
                                   uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;"
        ::"r"(smem_addr(smem_dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar)),
        "l"(policy)
        : "memory");
}

// 3-D variant: box {64 elements, 2 slabs, BS rows} of the view [rows][2][64].
__device__ inline void tma_load_3d(void* smem_dst, const CUtensorMap* map, int x, int z, int y, uint64_t* bar,
                                   uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;"
        ::"r"(smem_addr(smem_dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(z), "r"(y),
        "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// Shared-memory address of 16-byte chunk c of stage row r, as the tensor
// copies (128-byte swizzle: chunk k of a 128-byte line L sits at k ^ (L % 8))
// laid the stage out.
//   slab layout:        line (c/8, r) at (c/8)*STAGE_TOK*128 + r*128, L = r
//   interleaved layout: line (r, c/8) at r*256 + (c/8)*128,            L = 2r + c/8
template <class Shape>
__device__ inline uint32_t stage_chunk_addr(uint32_t base, int r, int c) {
    const int slab = c >> 3, k = c & 7;
    if constexpr (Shape::INTERLEAVED) {
        const int line = 2 * r + slab;
        return base + (uint32_t)(line * 128 + ((k ^ (line & 7)) << 4));
    } else {
        return base + (uint32_t)(slab * Shape::STAGE_TOK * 128 + r * 128 + ((k ^ (r & 7)) << 4));
    }
}

__device__ inline void store_out4(void* out, int dtype, int64_t index, float4 v) {
    if (dtype == PA_F32) {
        *reinterpret_cast<float4*>(static_cast<float*>(out) + index) = v;
    } else if (dtype == PA_F16) {
        __half2 a = __floats2half2_rn(v.x, v.y), b = __floats2half2_rn(v.z, v.w);
        uint2 w;
        memcpy(&w.x, &a, 4);
        memcpy(&w.y, &b, 4);
        *reinterpret_cast<uint2*>(static_cast<__half*>(out) + index) = w;
    } else {
        __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
        uint2 w;
        memcpy(&w.x, &a, 4);
        memcpy(&w.y, &b, 4);
        *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(out) + index) = w;
    }
}

// ---------------------------------------------------------------------------
// producer warp
//   TENSOR = false: one linear bulk copy per (block, head) tile; the stage
//                   holds rows in token order, ROW bytes apart.
//   TENSOR = true : tensor copies with 128-byte swizzle.  Slab layout: one
//                   2-D box of 64 elements x BS rows per 128-byte column slab;
//                   the stage holds slab s of row r at s*STAGE_TOK*128 +
//                   r*128, with 16-byte chunk c stored at chunk c ^ (r % 8).
//                   Interleaved layout (Shape::INTERLEAVED): one 3-D box per
//                   whole (block, head) tile; row r's two slabs at r*256 and
//                   r*256 + 128, chunk c of line L = 2r + s at c ^ (L % 8).
// ---------------------------------------------------------------------------
template <class Shape, int BS, int G, bool TENSOR>
__device__ void decode_producer(const DecodeParams& p, typename Shape::Smem& sm, int lane, const CUtensorMap* tk,
                                const CUtensorMap* tv) {
    constexpr int D = Shape::ROW / Shape::E;
    const bool direct = p.direct_items > 0;
    const int num_items = direct ? p.direct_items : *p.num_items;
    const int part_size = p.partition_size;
    const char* kbase = static_cast<const char*>(p.k_cache);
    const char* vbase = static_cast<const char*>(p.v_cache);
    const char* qbase = static_cast<const char*>(p.query);

    int st = 0;
    uint32_t ph = 0;
    uint32_t filled = 0;        // bit j: stage j was filled at least once
    uint32_t fill_parity = 0;   // bit j: parity of stage j's last fill
    bool drop_next_fill = (p.debug_flags & kDebugDropFirstFill) != 0;
    bool aborted = false;
    const uint64_t stream_policy = l2_evict_first_policy();

    // Item metadata travels one item ahead: while item k streams, the id of
    // item k+1, its (sequence, partition) pair and its context length are
    // already being fetched, so a new item starts without dependent loads.
    auto item_pair = [&](int it) {
        if (it >= num_items) return make_int2(0, 0);
        return direct ? make_int2(it / p.num_kv_heads, 0) : p.items[it / p.num_kv_heads];
    };
    // Work items: from the device counter, or (direct) a fixed stride.
    auto take_item = [&](int previous) {
        int it = 0;
        if (direct)
            it = previous < 0 ? (int)blockIdx.x : previous + (int)gridDim.x;
        else if (lane == 0)
            it = atomicAdd(p.next_item, 1);
        return it;
    };
    int item = __shfl_sync(kFullMask, take_item(-1), 0);
    int2 sp = item_pair(item);
    int ctx_raw = item < num_items ? __ldg(p.context_lens + sp.x) : 0;
    while (item < num_items) {
        int next = take_item(item);
        const int h = item - (item / p.num_kv_heads) * p.num_kv_heads;
        const int s = sp.x, part = sp.y;
        if (direct && lane == 0 && h == 0 && (ctx_raw < 0 || ctx_raw > p.ctx_cap))
            set_error(p.err, PA_DEVERR_CONTEXT_LEN);
        const int ctx = ctx_raw < 0 ? 0 : (ctx_raw > p.ctx_cap ? p.ctx_cap : ctx_raw);
        const int nparts = ctx == 0 ? 1 : (ctx + part_size - 1) / part_size;
        const int tb = part * part_size;
        const int te = min(tb + part_size, ctx);
        const int ntok = te > tb ? te - tb : 0;
        const int nst = ntok == 0 ? 1 : (ntok + Shape::STAGE_TOK - 1) / Shape::STAGE_TOK;
        const int32_t* trow = p.block_tables + (int64_t)s * p.max_blocks;
        int2 sp_next = make_int2(0, 0);
        int ctx_next = 0;

        for (int c = 0; c < nst; ++c) {
            const int t0 = tb + c * Shape::STAGE_TOK;
            const int t1 = min(t0 + Shape::STAGE_TOK, te);
            const int nblk = t1 > t0 ? (t1 - t0 + BS - 1) / BS : 0;
            int phys = -1;
            bool ok = false;
            if (lane < nblk) {
                phys = __ldg(trow + t0 / BS + lane);
                ok = phys >= 0 && (int64_t)phys < p.num_blocks;
                if (!ok) set_error(p.err, PA_DEVERR_BLOCK_ID);
            }
            const unsigned okmask = __ballot_sync(kFullMask, ok);
            const uint32_t bytes = (uint32_t)__popc(okmask) * 2u * Shape::TILE + (c == 0 ? Shape::QBYTES : 0u);
            bool free_ok = true;
            if (lane == 0) free_ok = mbar_wait_bounded(&sm.empty[st], ph ^ 1u, p.wait_limit_ns);
            free_ok = __shfl_sync(kFullMask, free_ok, 0);
            if (!free_ok) {
                aborted = true;
                break;
            }
            // Test hook: leave this stage unfilled (no copies, no arrival);
            // the rest of the loop body runs as usual.  Uniform across lanes.
            const bool drop = drop_next_fill;
            drop_next_fill = false;
            if (!drop) {
                if (lane == 0) {
                    StageMeta m;
                    m.item = item;
                    m.seq = s;
                    m.kv_head = h;
                    m.part = part;
                    m.nparts = nparts;
                    m.t0 = t0;
                    m.te = te;
                    m.first = c == 0;
                    m.last = c == nst - 1;
                    sm.meta[st] = m;
                    mbar_arrive_expect_tx(&sm.full[st], bytes);
                }
                __syncwarp();
                if (ok) {
                    if constexpr (TENSOR && Shape::INTERLEAVED) {
                        const int y = (int)(((int64_t)phys * p.num_kv_heads + h) * BS);
                        tma_load_3d(sm.kv[st][0] + lane * Shape::TILE, tk, 0, 0, y, &sm.full[st], stream_policy);
                        tma_load_3d(sm.kv[st][1] + lane * Shape::TILE, tv, 0, 0, y, &sm.full[st], stream_policy);
                    } else if constexpr (TENSOR) {
                        const int y = (int)(((int64_t)phys * p.num_kv_heads + h) * BS);
#pragma unroll
                        for (int slab = 0; slab < D / 64; ++slab) {
                            const int off = slab * Shape::STAGE_TOK * 128 + lane * BS * 128;
                            tma_load_2d(sm.kv[st][0] + off, tk, slab * 64, y, &sm.full[st], stream_policy);
                            tma_load_2d(sm.kv[st][1] + off, tv, slab * 64, y, &sm.full[st], stream_policy);
                        }
                    } else {
                        const int64_t tile = ((int64_t)phys * p.num_kv_heads + h) * Shape::TILE;
                        bulk_copy_g2s(sm.kv[st][0] + lane * Shape::TILE, kbase + tile, Shape::TILE, &sm.full[st]);
                        bulk_copy_g2s(sm.kv[st][1] + lane * Shape::TILE, vbase + tile, Shape::TILE, &sm.full[st]);
                    }
                }
                if (c == 0 && lane == 31) {
                    const int64_t qoff = ((int64_t)s * p.num_heads + (int64_t)h * G) * D * Shape::E;
                    bulk_copy_g2s(sm.q[st], qbase + qoff, Shape::QBYTES, &sm.full[st]);
                }
                filled |= 1u << st;
                fill_parity = (fill_parity & ~(1u << st)) | (ph << st);
            }
            if (++st == Shape::NSTAGE) {
                st = 0;
                ph ^= 1u;
            }
            if (c == 0) {
                // Start fetching the next item's metadata.
                next = __shfl_sync(kFullMask, next, 0);
                sp_next = item_pair(next);
                ctx_next = next < num_items ? __ldg(p.context_lens + sp_next.x) : 0;
            }
        }
        if (aborted) break;
        item = next;
        sp = sp_next;
        ctx_raw = ctx_next;
    }

    if (!aborted) {
        // End-of-work marker: a fill with no bytes.
        bool free_ok = true;
        if (lane == 0) free_ok = mbar_wait_bounded(&sm.empty[st], ph ^ 1u, p.wait_limit_ns);
        free_ok = __shfl_sync(kFullMask, free_ok, 0);
        if (free_ok) {
            if (lane == 0) {
                sm.meta[st].item = -1;
                mbar_arrive(&sm.full[st]);
            }
            filled |= 1u << st;
            fill_parity = (fill_parity & ~(1u << st)) | (ph << st);
        } else {
            aborted = true;
        }
    }
    if (aborted && lane == 0) {
        set_error(p.err, PA_DEVERR_TIMEOUT);
        atomicExch(&sm.abort_flag, 1);
    }
    // This CTA takes no more work: the reduce kernel may start launching.
    pdl_launch_dependents();
    // Drain: every copy this warp issued must land before the CTA exits --
    // wait for the last fill of every stage (bounded).
    if (lane == 0) {
        for (int j = 0; j < Shape::NSTAGE; ++j) {
            if (!(filled & (1u << j))) continue;
            if (!mbar_wait_bounded(&sm.full[j], (fill_parity >> j) & 1u, p.wait_limit_ns))
                set_error(p.err, PA_DEVERR_TIMEOUT);
        }
    }
    __syncwarp();
}

// ---------------------------------------------------------------------------
// end of an item
//   consumers: wait until the merge slot is free, store their per-warp
//     (max, sum, output) in it, and go on with the next item;
//   merge warp: merges the consumer warps' states and stores the output (one
//     partition) or the partition's partial (max, sum, normalised output) for
//     the reduce kernel.
// ---------------------------------------------------------------------------
template <class Smem>
__device__ inline bool acquire_merge_slot(Smem& sm, uint32_t fph, unsigned long long limit) {
    const bool ok = mbar_wait_bounded(&sm.merge_free, fph ^ 1u, limit);
    return __all_sync(kFullMask, ok);
}

// Called by every consumer warp after it wrote its part of the slot.
template <class Smem>
__device__ inline void release_to_merger(Smem& sm, const StageMeta& mt, int warp, int lane) {
    if (warp == 0 && lane == 0) sm.merge_meta = mt;
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.merge_full);
}

template <class Shape, int D, int G>
__device__ void merge_worker(const DecodeParams& p, typename Shape::Smem& sm, int lane) {
    constexpr int NCW = Shape::NCW;
    const float NEG_INF = __int_as_float(0xff800000);
    uint32_t mph = 0;
    while (true) {
        const bool ok = mbar_wait_bounded(&sm.merge_full, mph, p.wait_limit_ns);
        if (!__all_sync(kFullMask, ok)) {
            if (lane == 0) {
                set_error(p.err, PA_DEVERR_TIMEOUT);
                atomicExch(&sm.abort_flag, 1);
            }
            return;
        }
        mph ^= 1u;
        const StageMeta mt = sm.merge_meta;
        if (mt.item < 0) return;
        const int s = mt.seq, h = mt.kv_head;
        const int64_t unit = (int64_t)s * p.num_kv_heads + h;
        for (int i = lane; i < G * D / 4; i += 32) {
            const int g = (4 * i) / D, dd = 4 * i - g * D;
            float M = NEG_INF;
#pragma unroll
            for (int w = 0; w < NCW; ++w) M = fmaxf(M, sm.mm[w][g]);
            float L = 0.f;
            float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int w = 0; w < NCW; ++w) {
                const float mw = sm.mm[w][g];
                const float f = mw == NEG_INF ? 0.f : exp2_approx(mw - M);
                const float4 v = *reinterpret_cast<const float4*>(&sm.mo[w][g][dd]);
                L = fmaf(f, sm.ml[w][g], L);
                O.x = fmaf(f, v.x, O.x);
                O.y = fmaf(f, v.y, O.y);
                O.z = fmaf(f, v.z, O.z);
                O.w = fmaf(f, v.w, O.w);
            }
            const float inv = L > 0.f ? 1.f / L : 0.f;
            const float4 o = make_float4(O.x * inv, O.y * inv, O.z * inv, O.w * inv);
            if (mt.nparts == 1) {
                store_out4(p.out, p.out_dtype, ((int64_t)s * p.num_heads + (int64_t)h * G + g) * D + dd, o);
            } else {
                const int64_t pi = (unit * p.max_parts + mt.part) * G + g;
                *reinterpret_cast<float4*>(p.part_o + pi * D + dd) = o;
                if (dd == 0) *reinterpret_cast<float2*>(p.part_ml + 2 * pi) = make_float2(M, L);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.merge_free);
    }
}

__device__ inline void consumer_abort(const DecodeParams& p, int* abort_flag, int lane) {
    if (lane == 0) {
        set_error(p.err, PA_DEVERR_TIMEOUT);
        atomicExch(abort_flag, 1);
    }
}

// Occupancy-sized persistent launch of `kernel`.  The shared-memory opt-in
// and the resident-CTA count are set up once per (kernel, device) and cached.
template <class Shape, typename Kernel, typename... Args>
cudaError_t launch_persistent(Kernel kernel, int items_upper_bound, cudaStream_t stream, Args... args) {
    constexpr int smem = Shape::SMEM_BYTES;
    constexpr int kMaxDevices = 64;
    static int resident[kMaxDevices];  // SMs x CTAs per SM; 0 = not set up yet
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    int slots = __atomic_load_n(&resident[dev], __ATOMIC_ACQUIRE);
    if (slots == 0) {
        int sms = 0, occ = 0;
        if ((e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess)
            return e;
        if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
        if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, Shape::THREADS, smem)) != cudaSuccess)
            return e;
        if (occ < 1) return cudaErrorInvalidConfiguration;
        slots = sms * occ;
        __atomic_store_n(&resident[dev], slots, __ATOMIC_RELEASE);
    }
    int grid = slots;
    if (items_upper_bound < grid) grid = items_upper_bound > 0 ? items_upper_bound : 1;
    // Launched as a programmatic dependent of the planning kernel.
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(Shape::THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace pa
