// decode_simt.cuh -- paged decode attention, CUDA-core variant (all dtypes).
//
// What it computes: "PagedAttention 论文精读笔记", §2.1 (attention equation)
// in the block-wise order of §4.2: the keys and values of a sequence are read
// one physical block at a time, located through the block table (§5.2), and
// the per-block results are combined exactly ("PagedAttention paper review",
// "How does this work?").  The combination is the running-max / running-sum
// (online) softmax; a context longer than the partition size is split into
// partitions computed by different CTAs and merged by
//     M = max_p m_p,  L = sum_p l_p 2^(m_p - M),  o = sum_p (l_p 2^(m_p - M) / L) o_p
// (scores are kept in base-2 units: q is pre-scaled by scale * log2 e).
//
// CTA structure (persistent, one or two CTAs per SM):
//   warp 4 (producer): takes (sequence, partition, KV head) work items from a
//     device counter, reads the block table, and issues one bulk copy
//     (cp.async.bulk) per K tile and per V tile -- a tile is one (block, head)
//     slab [B][d], contiguous in the pool -- into a 3-stage shared-memory ring
//     guarded by mbarriers ("warp-level block read" with coalesced access,
//     "Efficient Memory Management ... Review", §3-2; here the copy engine
//     does the gathering).
//   warps 0-3 (consumers): each takes a quarter of the stage's tokens; lanes
//     own 16-byte chunks of a row, compute q.k for the G query heads that share
//     the KV head (GQA grouping on the CTA), reduce across the row with
//     shuffles, update the running max/sum with a lazy rescale, and accumulate
//     p.v.  At the item's end the four warps merge through shared memory and
//     write the output (one partition) or a partial (several partitions); the
//     CTA that finishes the last partition of a (sequence, KV head) merges the
//     partials (variable length without padding, Review §3-2).
// Every wait is bounded (global timer); a wait that runs out sets
// PA_DEVERR_TIMEOUT and the CTA drains its copies and returns.
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace pa {

constexpr int kDecodeConsumerWarps = 4;
constexpr int kDecodeStages = 3;

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

template <typename T, int D, int BS, int G>
struct SimtDecode {
    static constexpr int E = sizeof(T);
    static constexpr int NCW = kDecodeConsumerWarps;
    static constexpr int NSTAGE = kDecodeStages;
    static constexpr int THREADS = (NCW + 1) * 32;
    static constexpr int ROW = D * E;                 // bytes of one token's row
    static constexpr int STAGE_TOK = stage_tokens_for_row(ROW);
    static_assert(STAGE_TOK % BS == 0, "stage must hold whole blocks");
    static constexpr int BPS = STAGE_TOK / BS;        // blocks per stage
    static_assert(BPS <= 31, "one producer lane per block, lane 31 copies q");
    static constexpr int TPW = STAGE_TOK / NCW;       // tokens per consumer warp per stage
    static constexpr int VEC = 16 / E;                // elements per 16-byte chunk
    static constexpr int CPR = D / VEC;               // chunks per row
    static_assert(CPR <= 32 && 32 % CPR == 0, "a row must map onto a power-of-two lane group");
    static constexpr int TPI = 32 / CPR;              // rows per warp-wide load
    static_assert(TPW % TPI == 0, "warp's rows must be whole loads");
    static constexpr int RPL = TPW / TPI;             // rows per lane per stage
    static constexpr int RSUB = RPL < 4 ? RPL : 4;    // rows per softmax update
    static_assert(RPL % RSUB == 0, "rows per lane must split evenly");
    static constexpr int TILE = BS * ROW;             // bytes of one (block, head) slab
    static constexpr int KV_STAGE_BYTES = STAGE_TOK * ROW;
    static constexpr int QBYTES = G * D * E;
    static_assert(QBYTES % 16 == 0, "q tile must be a bulk-copy multiple");

    struct Smem {
        alignas(128) uint8_t kv[NSTAGE][2][KV_STAGE_BYTES];
        alignas(16) uint8_t q[NSTAGE][QBYTES];
        float mo[NCW][G][D];   // per-warp accumulators at the item's end
        float mm[NCW][G];      // per-warp running max (base-2 units)
        float ml[NCW][G];      // per-warp running sum
        float fin_m[G];        // merged max / sum of all partitions
        float fin_l[G];
        StageMeta meta[NSTAGE];
        uint64_t full[NSTAGE];
        uint64_t empty[NSTAGE];
        uint64_t group_bar;    // consumer-warp barrier
        int abort_flag;
        int is_last;
    };
    static constexpr int SMEM_BYTES = sizeof(Smem);
};

namespace simt_detail {

constexpr unsigned kFull = 0xffffffffu;

// Consumer-group barrier on an mbarrier (count = consumer threads) with a
// bounded wait, so that a CTA whose wait ran out cannot hang its siblings.
template <class S>
__device__ inline bool group_sync(S& sm, uint32_t& phase, unsigned long long limit) {
    mbar_arrive(&sm.group_bar);
    const bool ok = mbar_wait_bounded(&sm.group_bar, phase, limit);
    phase ^= 1u;
    return __all_sync(kFull, ok);
}

template <typename T>
__device__ inline void store_out(void* out, int dtype, int64_t index, float v) {
    if (dtype == PA_F32)
        static_cast<float*>(out)[index] = v;
    else if (dtype == PA_F16)
        static_cast<__half*>(out)[index] = __float2half_rn(v);
    else
        static_cast<__nv_bfloat16*>(out)[index] = __float2bfloat16_rn(v);
}

}  // namespace simt_detail

// ---------------------------------------------------------------------------
// producer warp
// ---------------------------------------------------------------------------
template <typename T, int D, int BS, int G>
__device__ void simt_producer(const DecodeParams& p, typename SimtDecode<T, D, BS, G>::Smem& sm, int lane) {
    using K = SimtDecode<T, D, BS, G>;
    using namespace simt_detail;
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
    item = __shfl_sync(kFull, item, 0);
    while (item < num_items) {
        int next = 0;
        if (lane == 0) next = atomicAdd(p.next_item, 1);  // latency overlaps this item
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
        const int nst = ntok == 0 ? 1 : (ntok + K::STAGE_TOK - 1) / K::STAGE_TOK;
        const int32_t* trow = p.block_tables + (int64_t)s * p.max_blocks;

        for (int c = 0; c < nst; ++c) {
            const int t0 = tb + c * K::STAGE_TOK;
            const int t1 = min(t0 + K::STAGE_TOK, te);
            const int nblk = t1 > t0 ? (t1 - t0 + BS - 1) / BS : 0;
            int phys = -1;
            bool ok = false;
            if (lane < nblk) {
                phys = __ldg(trow + t0 / BS + lane);
                ok = phys >= 0 && (int64_t)phys < p.num_blocks;
                if (!ok) set_error(p.err, PA_DEVERR_BLOCK_ID);
            }
            const unsigned okmask = __ballot_sync(kFull, ok);
            const uint32_t bytes = (uint32_t)__popc(okmask) * 2u * K::TILE + (c == 0 ? K::QBYTES : 0u);
            bool free_ok = true;
            if (lane == 0) free_ok = mbar_wait_bounded(&sm.empty[st], ph ^ 1u, p.wait_limit_ns);
            free_ok = __shfl_sync(kFull, free_ok, 0);
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
                const int64_t tile = ((int64_t)phys * p.num_kv_heads + h) * K::TILE;
                bulk_copy_g2s(sm.kv[st][0] + lane * K::TILE, kbase + tile, K::TILE, &sm.full[st]);
                bulk_copy_g2s(sm.kv[st][1] + lane * K::TILE, vbase + tile, K::TILE, &sm.full[st]);
            }
            if (c == 0 && lane == 31) {
                const int64_t qoff = ((int64_t)s * p.num_heads + (int64_t)h * G) * D * K::E;
                bulk_copy_g2s(sm.q[st], qbase + qoff, K::QBYTES, &sm.full[st]);
            }
            ++total_fills;
            if (++st == K::NSTAGE) {
                st = 0;
                ph ^= 1u;
            }
        }
        if (aborted) break;
        item = __shfl_sync(kFull, next, 0);
    }

    if (!aborted) {
        // End-of-work marker: a fill with no bytes.
        bool free_ok = true;
        if (lane == 0) free_ok = mbar_wait_bounded(&sm.empty[st], ph ^ 1u, p.wait_limit_ns);
        free_ok = __shfl_sync(kFull, free_ok, 0);
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
    if (aborted) {
        if (lane == 0) {
            set_error(p.err, PA_DEVERR_TIMEOUT);
            atomicExch(&sm.abort_flag, 1);
        }
    }
    // Drain: every bulk copy this warp issued must land before the CTA exits.
    if (lane == 0) {
        for (int j = 0; j < K::NSTAGE; ++j) {
            const unsigned fills = total_fills > (unsigned)j ? (total_fills - j + K::NSTAGE - 1) / K::NSTAGE : 0u;
            if (fills == 0) continue;
            if (!mbar_wait_bounded(&sm.full[j], (fills - 1u) & 1u, p.wait_limit_ns))
                set_error(p.err, PA_DEVERR_TIMEOUT);
        }
    }
    __syncwarp();
}

// ---------------------------------------------------------------------------
// consumer warps
// ---------------------------------------------------------------------------
template <typename T, int D, int BS, int G>
__device__ void simt_consumer(const DecodeParams& p, typename SimtDecode<T, D, BS, G>::Smem& sm, int warp,
                              int lane) {
    using K = SimtDecode<T, D, BS, G>;
    using namespace simt_detail;
    constexpr int VEC = K::VEC, CPR = K::CPR, TPI = K::TPI;
    const int tg = lane / CPR;  // row group within a warp-wide load
    const int c = lane % CPR;   // 16-byte chunk of the row this lane owns
    const int ct = warp * 32 + lane;
    const float NEG_INF = __int_as_float(0xff800000);

    float qf[G][VEC];
    float m[G], l[G], acc[G][VEC];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        m[g] = NEG_INF;
        l[g] = 0.f;
#pragma unroll
        for (int e = 0; e < VEC; ++e) acc[g][e] = 0.f, qf[g][e] = 0.f;
    }

    int st = 0;
    uint32_t ph = 0, gph = 0;
    while (true) {
        bool ok = mbar_wait_bounded(&sm.full[st], ph, p.wait_limit_ns);
        if (!__all_sync(kFull, ok)) {
            if (lane == 0) {
                set_error(p.err, PA_DEVERR_TIMEOUT);
                atomicExch(&sm.abort_flag, 1);
            }
            break;
        }
        const StageMeta mt = sm.meta[st];
        if (mt.item < 0) break;

        if (mt.first) {
            const T* qs = reinterpret_cast<const T*>(sm.q[st]);
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const uint4 w = *reinterpret_cast<const uint4*>(qs + g * D + c * VEC);
                float f[VEC];
                unpack16(w, f, T());
#pragma unroll
                for (int e = 0; e < VEC; ++e) qf[g][e] = f[e] * p.scale_log2;
                m[g] = NEG_INF;
                l[g] = 0.f;
#pragma unroll
                for (int e = 0; e < VEC; ++e) acc[g][e] = 0.f;
            }
        }

        const int row0 = warp * K::TPW;
        if (mt.t0 + row0 < mt.te) {
            const uint8_t* ks = sm.kv[st][0] + row0 * K::ROW + c * 16;
            const uint8_t* vs = sm.kv[st][1] + row0 * K::ROW + c * 16;
#pragma unroll
            for (int sub = 0; sub < K::RPL; sub += K::RSUB) {
                float sc[K::RSUB][G];
                bool valid[K::RSUB];
#pragma unroll
                for (int u = 0; u < K::RSUB; ++u) {
                    const int r = (sub + u) * TPI + tg;
                    valid[u] = mt.t0 + row0 + r < mt.te;
                    const uint4 w = *reinterpret_cast<const uint4*>(ks + r * K::ROW);
                    float kf[VEC];
                    unpack16(w, kf, T());
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        float a = 0.f;
#pragma unroll
                        for (int e = 0; e < VEC; ++e) a = fmaf(qf[g][e], kf[e], a);
                        sc[u][g] = a;
                    }
                }
                // Sum the partial dot products over the CPR lanes of each row.
#pragma unroll
                for (int u = 0; u < K::RSUB; ++u)
#pragma unroll
                    for (int g = 0; g < G; ++g)
#pragma unroll
                        for (int off = CPR / 2; off >= 1; off >>= 1)
                            sc[u][g] += __shfl_xor_sync(kFull, sc[u][g], off);
                // Row maximum over the warp's valid rows, then a lazy rescale.
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    float mx = NEG_INF;
#pragma unroll
                    for (int u = 0; u < K::RSUB; ++u) mx = valid[u] ? fmaxf(mx, sc[u][g]) : mx;
#pragma unroll
                    for (int off = CPR; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, off));
                    if (mx > m[g]) {  // warp-uniform
                        const float alpha = exp2_approx(m[g] - mx);
                        l[g] *= alpha;
#pragma unroll
                        for (int e = 0; e < VEC; ++e) acc[g][e] *= alpha;
                        m[g] = mx;
                    }
                }
                // p = 2^(s - m) and the weighted sum of the value rows.
#pragma unroll
                for (int u = 0; u < K::RSUB; ++u) {
                    const int r = (sub + u) * TPI + tg;
                    const uint4 w = *reinterpret_cast<const uint4*>(vs + r * K::ROW);
                    float vf[VEC];
                    unpack16(w, vf, T());
#pragma unroll
                    for (int e = 0; e < VEC; ++e) vf[e] = valid[u] ? vf[e] : 0.f;
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        const float pr = valid[u] ? exp2_approx(sc[u][g] - m[g]) : 0.f;
                        l[g] += pr;
#pragma unroll
                        for (int e = 0; e < VEC; ++e) acc[g][e] = fmaf(pr, vf[e], acc[g][e]);
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty[st]);

        if (mt.last) {
            // ---- finish the item: merge the four warps --------------------
            float lw[G], aw[G][VEC];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                lw[g] = l[g];
#pragma unroll
                for (int off = CPR; off < 32; off <<= 1) lw[g] += __shfl_xor_sync(kFull, lw[g], off);
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    aw[g][e] = acc[g][e];
#pragma unroll
                    for (int off = CPR; off < 32; off <<= 1) aw[g][e] += __shfl_xor_sync(kFull, aw[g][e], off);
                }
            }
            if (tg == 0) {
#pragma unroll
                for (int g = 0; g < G; ++g)
#pragma unroll
                    for (int e = 0; e < VEC; ++e) sm.mo[warp][g][c * VEC + e] = aw[g][e];
            }
            if (lane == 0) {
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    sm.mm[warp][g] = m[g];
                    sm.ml[warp][g] = lw[g];
                }
            }
            bool gok = group_sync(sm, gph, p.wait_limit_ns);
            const int s = mt.seq, h = mt.kv_head;
            const int64_t unit = (int64_t)s * p.num_kv_heads + h;
            if (gok) {
                for (int i = ct; i < G * D; i += K::NCW * 32) {
                    const int g = i / D, dd = i - (i / D) * D;
                    float M = NEG_INF;
#pragma unroll
                    for (int w = 0; w < K::NCW; ++w) M = fmaxf(M, sm.mm[w][g]);
                    float L = 0.f, O = 0.f;
#pragma unroll
                    for (int w = 0; w < K::NCW; ++w) {
                        const float mw = sm.mm[w][g];
                        const float f = mw == NEG_INF ? 0.f : exp2_approx(mw - M);
                        L = fmaf(f, sm.ml[w][g], L);
                        O = fmaf(f, sm.mo[w][g][dd], O);
                    }
                    const float o = L > 0.f ? O / L : 0.f;
                    if (mt.nparts == 1) {
                        const int64_t oi = ((int64_t)s * p.num_heads + (int64_t)h * G + g) * D + dd;
                        store_out<T>(p.out, p.out_dtype, oi, o);
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
                    // Merge all partitions of (s, h): per-head max and sum first.
                    for (int g = warp; g < G; g += K::NCW) {
                        const int64_t base = unit * p.max_parts * G + g;
                        float M = NEG_INF;
                        for (int q = lane; q < mt.nparts; q += 32) M = fmaxf(M, __ldcg(p.part_ml + 2 * (base + (int64_t)q * G)));
#pragma unroll
                        for (int off = 16; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, off));
                        float L = 0.f;
                        for (int q = lane; q < mt.nparts; q += 32) {
                            const int64_t pi = base + (int64_t)q * G;
                            L += __ldcg(p.part_ml + 2 * pi + 1) * exp2_approx(__ldcg(p.part_ml + 2 * pi) - M);
                        }
#pragma unroll
                        for (int off = 16; off >= 1; off >>= 1) L += __shfl_xor_sync(kFull, L, off);
                        if (lane == 0) {
                            sm.fin_m[g] = M;
                            sm.fin_l[g] = L;
                        }
                    }
                    gok = group_sync(sm, gph, p.wait_limit_ns);
                    if (gok) {
                        for (int i = ct; i < G * D; i += K::NCW * 32) {
                            const int g = i / D, dd = i - (i / D) * D;
                            const int64_t base = unit * p.max_parts * G + g;
                            const float M = sm.fin_m[g];
                            const float invL = 1.f / sm.fin_l[g];
                            float O = 0.f;
#pragma unroll 4
                            for (int q = 0; q < mt.nparts; ++q) {
                                const int64_t pi = base + (int64_t)q * G;
                                const float w = __ldcg(p.part_ml + 2 * pi + 1) * exp2_approx(__ldcg(p.part_ml + 2 * pi) - M);
                                O = fmaf(w, __ldcg(p.part_o + pi * D + dd), O);
                            }
                            const int64_t oi = ((int64_t)s * p.num_heads + (int64_t)h * G + g) * D + dd;
                            store_out<T>(p.out, p.out_dtype, oi, O * invL);
                        }
                        if (ct == 0) p.counters[unit] = 0;
                    }
                }
            }
            // The merge buffers are free again only when every warp is done.
            if (gok) gok = group_sync(sm, gph, p.wait_limit_ns);
            if (!gok) {
                if (lane == 0) {
                    set_error(p.err, PA_DEVERR_TIMEOUT);
                    atomicExch(&sm.abort_flag, 1);
                }
                break;
            }
        }
        if (++st == K::NSTAGE) {
            st = 0;
            ph ^= 1u;
        }
        if (*reinterpret_cast<volatile int*>(&sm.abort_flag)) break;
    }
}

template <typename T, int D, int BS, int G>
__global__ void __launch_bounds__(SimtDecode<T, D, BS, G>::THREADS)
decode_simt_kernel(const __grid_constant__ DecodeParams p) {
    using K = SimtDecode<T, D, BS, G>;
    extern __shared__ __align__(128) uint8_t smem_raw[];
    auto& sm = *reinterpret_cast<typename K::Smem*>(smem_raw);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        for (int s = 0; s < K::NSTAGE; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], K::NCW);
        }
        mbar_init(&sm.group_bar, K::NCW * 32);
        sm.abort_flag = 0;
        sm.is_last = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (warp == K::NCW)
        simt_producer<T, D, BS, G>(p, sm, lane);
    else
        simt_consumer<T, D, BS, G>(p, sm, warp, lane);
}

template <typename T, int D, int BS, int G>
cudaError_t run_decode_simt(const DecodeParams& p, int items_upper_bound, cudaStream_t stream) {
    using K = SimtDecode<T, D, BS, G>;
    auto kernel = decode_simt_kernel<T, D, BS, G>;
    constexpr int smem = K::SMEM_BYTES;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0, occ = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, K::THREADS, smem)) != cudaSuccess) return e;
    if (occ < 1) return cudaErrorInvalidConfiguration;
    int grid = sms * occ;
    if (items_upper_bound < grid) grid = items_upper_bound > 0 ? items_upper_bound : 1;
    kernel<<<grid, K::THREADS, smem, stream>>>(p);
    return cudaGetLastError();
}

// Dispatch on (head_dim, block_size, group) for one element type.
template <typename T>
cudaError_t dispatch_decode_simt(const DecodeParams& p, int head_dim, int block_size, int group, int ub,
                                 cudaStream_t stream) {
#define PA_DECODE_CASE(DD, BB, GG)                                           \
    if (head_dim == DD && block_size == BB && group == GG)                 \
        return run_decode_simt<T, DD, BB, GG>(p, ub, stream);
#define PA_DECODE_GROUPS(DD, BB) \
    PA_DECODE_CASE(DD, BB, 1) PA_DECODE_CASE(DD, BB, 2) PA_DECODE_CASE(DD, BB, 4) PA_DECODE_CASE(DD, BB, 8)
    PA_DECODE_GROUPS(64, 8)
    PA_DECODE_GROUPS(64, 16)
    PA_DECODE_GROUPS(64, 32)
    PA_DECODE_GROUPS(128, 8)
    PA_DECODE_GROUPS(128, 16)
    PA_DECODE_GROUPS(128, 32)
#undef PA_DECODE_GROUPS
#undef PA_DECODE_CASE
    return cudaErrorNotSupported;
}

}  // namespace pa
