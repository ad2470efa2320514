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
// different CTAs compute; the CTA that finishes the last partition of a
// (sequence, KV head) merges them with
//     M = max_p m_p,  L = sum_p l_p 2^(m_p - M),  o = sum_p (l_p 2^(m_p - M) / L) o_p
// (scores are kept in base-2 units: scale * log2 e is folded in).
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
//     grouping on the CTA).  At an item's end they merge through shared memory.
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
    static constexpr int THREADS = (NCW + 1) * 32;
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

    struct Smem {
        alignas(1024) uint8_t kv[NSTAGE][2][KV_STAGE_BYTES];
        alignas(16) uint8_t q[NSTAGE][QBYTES];
        float mo[NCW][G][D];   // per-warp output accumulators at the item's end
        float mm[NCW][G];      // per-warp running max (base-2 units)
        float ml[NCW][G];      // per-warp running sum
        float fin_m[G];        // merged max / sum over partitions
        float fin_l[G];
        StageMeta meta[NSTAGE];
        uint64_t full[NSTAGE];
        uint64_t empty[NSTAGE];
        uint64_t group_bar;    // consumer-warp barrier
        int abort_flag;
        int is_last;
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
        mbar_init(&sm.group_bar, consumer_warps * 32);
        sm.abort_flag = 0;
        sm.is_last = 0;
        fence_mbar_init();
    }
    __syncthreads();
}

// 2-D tiled TMA load of one box into shared memory, completed on `bar`.
__device__ inline void tma_load_2d(void* smem_dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(smem_addr(smem_dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}

// Consumer-group barrier on an mbarrier (count = consumer threads) with a
// bounded wait, so that a CTA whose wait ran out cannot hang its siblings.
template <class Smem>
__device__ inline bool group_sync(Smem& sm, uint32_t& phase, unsigned long long limit) {
    mbar_arrive(&sm.group_bar);
    const bool ok = mbar_wait_bounded(&sm.group_bar, phase, limit);
    phase ^= 1u;
    return __all_sync(kFullMask, ok);
}

__device__ inline void store_out(void* out, int dtype, int64_t index, float v) {
    if (dtype == PA_F32)
        static_cast<float*>(out)[index] = v;
    else if (dtype == PA_F16)
        static_cast<__half*>(out)[index] = __float2half_rn(v);
    else
        static_cast<__nv_bfloat16*>(out)[index] = __float2bfloat16_rn(v);
}

// ---------------------------------------------------------------------------
// producer warp
//   TENSOR = false: one linear bulk copy per (block, head) tile; the stage
//                   holds rows in token order, ROW bytes apart.
//   TENSOR = true : 2-D tensor copies with 128-byte swizzle, one box of
//                   64 elements x BS rows per 128-byte column slab; the stage
//                   holds slab s of row r at s*STAGE_TOK*128 + r*128, with
//                   16-byte chunk c stored at chunk c ^ (r % 8).
// ---------------------------------------------------------------------------
template <class Shape, int BS, int G, bool TENSOR>
__device__ void decode_producer(const DecodeParams& p, typename Shape::Smem& sm, int lane, const CUtensorMap* tk,
                                const CUtensorMap* tv) {
    constexpr int D = Shape::ROW / Shape::E;
    const int num_items = *p.num_items;
    const int part_size = p.partition_size;
    const char* kbase = static_cast<const char*>(p.k_cache);
    const char* vbase = static_cast<const char*>(p.v_cache);
    const char* qbase = static_cast<const char*>(p.query);

    int st = 0;
    uint32_t ph = 0;
    unsigned total_fills = 0;
    bool aborted = false;

    int item = 0;
    if (lane == 0) item = atomicAdd(p.next_item, 1);
    item = __shfl_sync(kFullMask, item, 0);
    while (item < num_items) {
        int next = 0;
        if (lane == 0) next = atomicAdd(p.next_item, 1);  // its latency overlaps this item
        const int pair = item / p.num_kv_heads;
        const int h = item - pair * p.num_kv_heads;
        const int2 sp = p.items[pair];
        const int s = sp.x, part = sp.y;
        int ctx = __ldg(p.context_lens + s);
        ctx = ctx < 0 ? 0 : (ctx > p.ctx_cap ? p.ctx_cap : ctx);
        const int nparts = ctx == 0 ? 1 : (ctx + part_size - 1) / part_size;
        const int tb = part * part_size;
        const int te = min(tb + part_size, ctx);
        const int ntok = te > tb ? te - tb : 0;
        const int nst = ntok == 0 ? 1 : (ntok + Shape::STAGE_TOK - 1) / Shape::STAGE_TOK;
        const int32_t* trow = p.block_tables + (int64_t)s * p.max_blocks;

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
                if constexpr (TENSOR) {
                    const int y = (int)(((int64_t)phys * p.num_kv_heads + h) * BS);
#pragma unroll
                    for (int slab = 0; slab < D / 64; ++slab) {
                        const int off = slab * Shape::STAGE_TOK * 128 + lane * BS * 128;
                        tma_load_2d(sm.kv[st][0] + off, tk, slab * 64, y, &sm.full[st]);
                        tma_load_2d(sm.kv[st][1] + off, tv, slab * 64, y, &sm.full[st]);
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
            ++total_fills;
            if (++st == Shape::NSTAGE) {
                st = 0;
                ph ^= 1u;
            }
        }
        if (aborted) break;
        item = __shfl_sync(kFullMask, next, 0);
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
            ++total_fills;
        } else {
            aborted = true;
        }
    }
    if (aborted && lane == 0) {
        set_error(p.err, PA_DEVERR_TIMEOUT);
        atomicExch(&sm.abort_flag, 1);
    }
    // Drain: every copy this warp issued must land before the CTA exits.
    if (lane == 0) {
        for (int j = 0; j < Shape::NSTAGE; ++j) {
            const unsigned fills =
                total_fills > (unsigned)j ? (total_fills - j + Shape::NSTAGE - 1) / Shape::NSTAGE : 0u;
            if (fills == 0) continue;
            if (!mbar_wait_bounded(&sm.full[j], (fills - 1u) & 1u, p.wait_limit_ns))
                set_error(p.err, PA_DEVERR_TIMEOUT);
        }
    }
    __syncwarp();
}

// ---------------------------------------------------------------------------
// end of an item: merge the consumer warps' (max, sum, output) held in
// sm.mm / sm.ml / sm.mo, then write the output (one partition) or a partial
// and, in the CTA that completes a (sequence, KV head), merge all partials.
// Called by all consumer threads; returns false if a bounded wait ran out.
// ---------------------------------------------------------------------------
template <class Shape, int D, int G>
__device__ bool finish_item(const DecodeParams& p, typename Shape::Smem& sm, const StageMeta& mt, int warp, int lane,
                            uint32_t& gph) {
    constexpr int NCW = Shape::NCW;
    const float NEG_INF = __int_as_float(0xff800000);
    const int ct = warp * 32 + lane;
    bool gok = group_sync(sm, gph, p.wait_limit_ns);
    const int s = mt.seq, h = mt.kv_head;
    const int64_t unit = (int64_t)s * p.num_kv_heads + h;
    if (gok) {
        for (int i = ct; i < G * D; i += NCW * 32) {
            const int g = i / D, dd = i - (i / D) * D;
            float M = NEG_INF;
#pragma unroll
            for (int w = 0; w < NCW; ++w) M = fmaxf(M, sm.mm[w][g]);
            float L = 0.f, O = 0.f;
#pragma unroll
            for (int w = 0; w < NCW; ++w) {
                const float mw = sm.mm[w][g];
                const float f = mw == NEG_INF ? 0.f : exp2_approx(mw - M);
                L = fmaf(f, sm.ml[w][g], L);
                O = fmaf(f, sm.mo[w][g][dd], O);
            }
            const float o = L > 0.f ? O / L : 0.f;
            if (mt.nparts == 1) {
                store_out(p.out, p.out_dtype, ((int64_t)s * p.num_heads + (int64_t)h * G + g) * D + dd, o);
            } else {
                const int64_t pi = (unit * p.max_parts + mt.part) * G + g;
                p.part_o[pi * D + dd] = o;
                if (dd == 0) {
                    p.part_ml[2 * pi] = M;
                    p.part_ml[2 * pi + 1] = L;
                }
            }
        }
    }
    if (gok && mt.nparts > 1) {
        __threadfence();
        gok = group_sync(sm, gph, p.wait_limit_ns);
        if (gok && ct == 0) {
            const int done = atomicAdd(p.counters + unit, 1);
            sm.is_last = done == mt.nparts - 1;
        }
        if (gok) gok = group_sync(sm, gph, p.wait_limit_ns);
        if (gok && sm.is_last) {
            __threadfence();
            // Per-head max and sum over the partitions, one warp per head.
            for (int g = warp; g < G; g += NCW) {
                const int64_t base = unit * p.max_parts * G + g;
                float M = NEG_INF;
                for (int q = lane; q < mt.nparts; q += 32)
                    M = fmaxf(M, __ldcg(p.part_ml + 2 * (base + (int64_t)q * G)));
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(kFullMask, M, off));
                float L = 0.f;
                for (int q = lane; q < mt.nparts; q += 32) {
                    const int64_t pi = base + (int64_t)q * G;
                    L += __ldcg(p.part_ml + 2 * pi + 1) * exp2_approx(__ldcg(p.part_ml + 2 * pi) - M);
                }
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1) L += __shfl_xor_sync(kFullMask, L, off);
                if (lane == 0) {
                    sm.fin_m[g] = M;
                    sm.fin_l[g] = L;
                }
            }
            gok = group_sync(sm, gph, p.wait_limit_ns);
            if (gok) {
                for (int i = ct; i < G * D; i += NCW * 32) {
                    const int g = i / D, dd = i - (i / D) * D;
                    const int64_t base = unit * p.max_parts * G + g;
                    const float M = sm.fin_m[g];
                    const float invL = 1.f / sm.fin_l[g];
                    float O = 0.f;
#pragma unroll 4
                    for (int q = 0; q < mt.nparts; ++q) {
                        const int64_t pi = base + (int64_t)q * G;
                        const float wgt = __ldcg(p.part_ml + 2 * pi + 1) * exp2_approx(__ldcg(p.part_ml + 2 * pi) - M);
                        O = fmaf(wgt, __ldcg(p.part_o + pi * D + dd), O);
                    }
                    store_out(p.out, p.out_dtype, ((int64_t)s * p.num_heads + (int64_t)h * G + g) * D + dd, O * invL);
                }
                if (ct == 0) p.counters[unit] = 0;
            }
        }
    }
    // The merge buffers are free again only when every warp is done reading.
    if (gok) gok = group_sync(sm, gph, p.wait_limit_ns);
    return gok;
}

__device__ inline void consumer_abort(const DecodeParams& p, int* abort_flag, int lane) {
    if (lane == 0) {
        set_error(p.err, PA_DEVERR_TIMEOUT);
        atomicExch(abort_flag, 1);
    }
}

// Occupancy-sized persistent launch of `kernel`.
template <class Shape, typename Kernel, typename... Args>
cudaError_t launch_persistent(Kernel kernel, int items_upper_bound, cudaStream_t stream, Args... args) {
    constexpr int smem = Shape::SMEM_BYTES;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0, occ = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, Shape::THREADS, smem)) != cudaSuccess)
        return e;
    if (occ < 1) return cudaErrorInvalidConfiguration;
    int grid = sms * occ;
    if (items_upper_bound < grid) grid = items_upper_bound > 0 ? items_upper_bound : 1;
    kernel<<<grid, Shape::THREADS, smem, stream>>>(args...);
    return cudaGetLastError();
}

}  // namespace pa
