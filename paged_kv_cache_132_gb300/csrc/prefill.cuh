// prefill.cuh -- prompt-phase attention over a cached prefix, on the
// Blackwell tensor cores (tcgen05.mma, accumulators in tensor memory).
//
// What it computes: "PagedAttention 论文精读笔记", §6.3 -- with a shared
// prefix already cached in physical blocks, the prompt phase computes only
// the request's own tokens -- with the attention equation of §2.1 evaluated
// through the block table (§5.2, §5.3).  Sequence s has n new tokens, the
// last n of its ctx cached tokens (their K/V were written by
// pa_reshape_and_cache); new token i sits at position ctx - n + i and
// attends to positions 0..ctx-n+i.
//
// One CTA computes a tile of 128 query rows of one (sequence, KV head): the
// rows are (token, grouped query head) pairs, 128/G tokens x G heads, so the
// G query heads that share a KV head share every K/V tile (GQA).  The keys
// and values are streamed in tiles of 128 positions.  Per tile j:
//   S_j = Q K_j^T          tcgen05.mma, M=128 N=128 K=d, into TMEM (2 buffers)
//   P_j = 2^(S_j*c - m)    softmax warps, one thread per row, P to shared
//                          memory as 16-bit K-major rows
//   O  += P_j V_j          tcgen05.mma, M=128 N=d K=128, O in TMEM
// with the running max m kept in base-2 units (c = scale * log2 e) and O
// rescaled only when a row's max grows by more than 8 (a factor of 256).
//
// Warp roles (192 threads, one CTA per SM):
//   warps 0-3 softmax: thread r owns row r = TMEM lane r; mask, exponentials,
//             row sums, P, the rare rescale of O, and at the end O / sum;
//   warp 4    producer: Q once (3-D tensor copy: 128/G tokens x G heads x
//             64-element slabs), then K and V tiles through the block table,
//             one 2-D tensor copy per (block, 64-element slab), into a
//             2-stage ring;
//   warp 5    MMA issuer (one thread) and owner of the TMEM allocation.
// The MMA thread issues S_{j+1} before P_j.V_j, so the tensor cores compute
// the next scores while the softmax warps work on the current ones.
// Every wait is bounded; a wait that runs out sets PA_DEVERR_TIMEOUT, the
// CTA stops issuing work, waits for what it issued and releases TMEM.
#pragma once

#include <cuda.h>

#include <type_traits>

#include "common.cuh"
#include "decode_common.cuh"  // kFullMask, store_out4
#include "kernels.h"
#include "tcgen05.cuh"

namespace pa {

template <int D>
struct PrefillShape {
    static constexpr int BM = 128;          // query rows per CTA
    static constexpr int BN = 128;          // key/value positions per tile
    static constexpr int SLABS = D / 64;    // 64-element (128-byte) column slabs of a row
    static constexpr int SLAB = 128 * 128;  // bytes of one slab of 128 rows
    static constexpr int NSTAGE = 3;
    static constexpr int SOFTMAX_WARPS = 4;
    static constexpr int PRODUCER_WARP = 4;
    static constexpr int MMA_WARP = 5;
    static constexpr int THREADS = 6 * 32;
    static constexpr uint32_t TMEM_COLS = 512;
    // TMEM columns: S buffer b at b*BN; its P (16-bit, two per column) is
    // written over it: P (or P_hi) in the first BN/2 columns, P_lo in the
    // next BN/2.  The output accumulator O after the two buffers.
    static constexpr uint32_t O_COL = 2 * BN;
    static_assert(D == 64 || D == 128, "head_dim 64 or 128");
    static_assert(O_COL + D <= TMEM_COLS, "TMEM columns");

    struct Smem {
        alignas(1024) uint8_t q[SLABS][SLAB];
        alignas(1024) uint8_t k[NSTAGE][SLABS][SLAB];
        alignas(1024) uint8_t v[NSTAGE][SLABS][SLAB];
        uint64_t q_full;
        uint64_t k_full[NSTAGE];
        uint64_t v_full[NSTAGE];
        uint64_t kv_empty[NSTAGE];
        uint64_t s_full[2];    // S_j in buffer j % 2 (MMA commit)
        uint64_t p_full[2];    // P_j written over it (softmax warps)
        uint64_t pv_done[2];   // P_j V_j complete: buffer j % 2 and O free again
        uint64_t mma_done;
        uint32_t tmem_base;
        int abort_flag;
    };
    // At least 120 KiB, so that no two CTAs share an SM: the 512-column TMEM
    // allocation then never has to wait for another CTA.
    static constexpr int SMEM_BYTES =
        (int)sizeof(Smem) + 1024 > 120 * 1024 ? (int)sizeof(Smem) + 1024 : 120 * 1024;
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory of one CTA");
};

// Tensor copies without an L2 hint: a K/V tile is read again by the other
// query tiles of its sequence and, for a shared prefix, by other sequences.
__device__ inline void tma_load_2d_plain(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}

__device__ inline void tma_load_3d_plain(void* dst, const CUtensorMap* map, int x, int y, int z, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, "
        "%4}], [%5];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar))
        : "memory");
}

template <class Smem>
__device__ inline void prefill_abort(const PrefillParams& p, Smem& sm) {
    set_error(p.err, PA_DEVERR_TIMEOUT);
    atomicExch(&sm.abort_flag, 1);
}

// What one CTA works on.
struct PrefillTile {
    int seq, kv_head;
    int n;       // new tokens of the sequence
    int ctx;     // its context length (cached prefix + new tokens)
    int q0;      // first new token of the tile
    int qrow0;   // its row in the query / output arrays
    int kv_end;  // positions [0, kv_end) are read by the tile
    int nt;      // key/value tiles
};

// ---------------------------------------------------------------------------
// producer warp
// ---------------------------------------------------------------------------
template <class Shape>
__device__ void prefill_producer(const PrefillParams& p, typename Shape::Smem& sm, int lane, const PrefillTile& w,
                                 const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv) {
    const int BS = p.block_size;
    const uint32_t box_bytes = (uint32_t)BS * 128u;
    const int32_t* trow = p.block_tables + (int64_t)w.seq * p.max_blocks;
    if (lane == 0) {
        mbar_arrive_expect_tx(&sm.q_full, Shape::SLABS * Shape::SLAB);
#pragma unroll
        for (int slab = 0; slab < Shape::SLABS; ++slab)
            tma_load_3d_plain(sm.q[slab], tq, slab * 64, w.kv_head << p.group_shift, w.qrow0, &sm.q_full);
    }
    uint32_t filled = 0, parity = 0;  // per stage: filled at least once / parity of its last fill
    bool ok_run = true;
    for (int j = 0; j < w.nt; ++j) {
        const int st = j % Shape::NSTAGE;
        const uint32_t ph = (uint32_t)(j / Shape::NSTAGE) & 1u;
        bool free_ok = true;
        if (lane == 0) free_ok = mbar_wait_bounded(&sm.kv_empty[st], ph ^ 1u, p.wait_limit_ns);
        free_ok = __shfl_sync(kFullMask, free_ok, 0);
        if (!free_ok) {
            ok_run = false;
            break;
        }
        if (*reinterpret_cast<volatile int*>(&sm.abort_flag)) break;
        const int kv0 = j * Shape::BN;
        const int ntok = min(Shape::BN, w.kv_end - kv0);
        const int nblk = (ntok + BS - 1) / BS;  // <= 16: block_size >= 8
        int phys = -1;
        bool ok = false;
        if (lane < nblk) {
            phys = __ldg(trow + kv0 / BS + lane);
            ok = phys >= 0 && (int64_t)phys < p.num_blocks;
            if (!ok) set_error(p.err, PA_DEVERR_BLOCK_ID);
        }
        const uint32_t bytes = (uint32_t)__popc(__ballot_sync(kFullMask, ok)) * Shape::SLABS * box_bytes;
        if (lane == 0) {
            mbar_arrive_expect_tx(&sm.k_full[st], bytes);
            mbar_arrive_expect_tx(&sm.v_full[st], bytes);
        }
        __syncwarp();
        if (ok) {
            const int y = (int)(((int64_t)phys * p.num_kv_heads + w.kv_head) * BS);
#pragma unroll
            for (int slab = 0; slab < Shape::SLABS; ++slab)
                tma_load_2d_plain(sm.k[st][slab] + lane * box_bytes, tk, slab * 64, y, &sm.k_full[st]);
#pragma unroll
            for (int slab = 0; slab < Shape::SLABS; ++slab)
                tma_load_2d_plain(sm.v[st][slab] + lane * box_bytes, tv, slab * 64, y, &sm.v_full[st]);
        }
        filled |= 1u << st;
        parity = (parity & ~(1u << st)) | (ph << st);
    }
    if (!ok_run && lane == 0) prefill_abort(p, sm);
    pdl_launch_dependents();
    // Every copy this warp issued lands before the CTA exits (bounded).
    if (lane == 0) {
        bool drained = mbar_wait_bounded(&sm.q_full, 0, p.wait_limit_ns);
        for (int st = 0; st < Shape::NSTAGE; ++st) {
            if (!(filled & (1u << st))) continue;
            const uint32_t ph = (parity >> st) & 1u;
            drained = mbar_wait_bounded(&sm.k_full[st], ph, p.wait_limit_ns) && drained;
            drained = mbar_wait_bounded(&sm.v_full[st], ph, p.wait_limit_ns) && drained;
        }
        if (!drained) set_error(p.err, PA_DEVERR_TIMEOUT);
    }
    __syncwarp();
}

// ---------------------------------------------------------------------------
// MMA issuer (one thread)
// ---------------------------------------------------------------------------
template <class Shape, uint32_t IDESC_S, uint32_t IDESC_O, bool SPLIT_P>
__device__ void prefill_mma(const PrefillParams& p, typename Shape::Smem& sm, uint32_t tmem, int nt) {
    constexpr int KS_S = Shape::SLABS * 4;  // 16-element steps over head_dim
    constexpr int KS_O = Shape::BN / 16;    // 16-position steps over the tile
    const uint64_t lim = p.wait_limit_ns;
    const uint32_t q_base = smem_addr(sm.q[0]);

    // O += P_jj V_jj: A = P from TMEM (8 columns per 16 positions), B = V
    // MN-major (head_dim along N, slabs Shape::SLAB bytes apart).  With
    // SPLIT_P the 16-bit P is P_hi + P_lo and both halves are multiplied.
    auto issue_pv = [&](int jj) -> bool {
        const int b = jj & 1, st = jj % Shape::NSTAGE;
        if (!mbar_wait_bounded(&sm.p_full[b], (uint32_t)(jj >> 1) & 1u, lim)) return false;
        if (!mbar_wait_bounded(&sm.v_full[st], (uint32_t)(jj / Shape::NSTAGE) & 1u, lim)) return false;
        tc_fence_after_sync();
        const uint32_t v_base = smem_addr(sm.v[st][0]);
        const uint32_t p_tmem = tmem + b * Shape::BN;
#pragma unroll
        for (int ks = 0; ks < KS_O; ++ks)
            mma_f16_ts(tmem + Shape::O_COL, p_tmem + ks * 8,
                       smem_desc_sw128(v_base + ks * 16 * 128, Shape::SLAB, 1024), IDESC_O,
                       (jj > 0 || ks > 0) ? 1u : 0u);
        if constexpr (SPLIT_P) {
#pragma unroll
            for (int ks = 0; ks < KS_O; ++ks)
                mma_f16_ts(tmem + Shape::O_COL, p_tmem + Shape::BN / 2 + ks * 8,
                           smem_desc_sw128(v_base + ks * 16 * 128, Shape::SLAB, 1024), IDESC_O, 1u);
        }
        mma_commit(&sm.pv_done[b]);
        mma_commit(&sm.kv_empty[st]);
        return true;
    };

    bool ok = mbar_wait_bounded(&sm.q_full, 0, lim);
    for (int j = 0; ok && j < nt; ++j) {
        const int b = j & 1, st = j % Shape::NSTAGE;
        // K_j landed, and buffer b is free (P_{j-2} V_{j-2} complete).
        ok = mbar_wait_bounded(&sm.k_full[st], (uint32_t)(j / Shape::NSTAGE) & 1u, lim) &&
             mbar_wait_bounded(&sm.pv_done[b], ((uint32_t)(j >> 1) & 1u) ^ 1u, lim);
        if (!ok) break;
        tc_fence_after_sync();
        const uint32_t k_base = smem_addr(sm.k[st][0]);
#pragma unroll
        for (int ks = 0; ks < KS_S; ++ks) {
            const uint32_t off = (ks >> 2) * Shape::SLAB + (ks & 3) * 32;
            mma_f16_ss(tmem + b * Shape::BN, smem_desc_sw128(q_base + off, 16, 1024),
                       smem_desc_sw128(k_base + off, 16, 1024), IDESC_S, ks > 0 ? 1u : 0u);
        }
        mma_commit(&sm.s_full[b]);
        if (j >= 1) ok = issue_pv(j - 1);
    }
    if (ok) ok = issue_pv(nt - 1);
    if (!ok) prefill_abort(p, sm);
    // Nothing this thread issued may still be running when TMEM is released.
    mma_commit(&sm.mma_done);
    if (!mbar_wait_bounded(&sm.mma_done, 0, lim)) set_error(p.err, PA_DEVERR_TIMEOUT);
}

// ---------------------------------------------------------------------------
// softmax warps (thread r = row r = TMEM lane r)
// ---------------------------------------------------------------------------
// Two 16-bit values in one 32-bit word, the first in the low half.
__device__ inline uint32_t pack_hi_halves(float a, float b) {
    // the high 16 bits of each binary32: bfloat16 truncation
    return __byte_perm(__float_as_uint(a), __float_as_uint(b), 0x7632);
}

template <typename T>
__device__ inline uint32_t pack_rn(float a, float b) {
    uint32_t w;
    if constexpr (std::is_same<T, __nv_bfloat16>::value) {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        memcpy(&w, &h, 4);
    } else {
        __half2 h = __floats2half2_rn(a, b);
        memcpy(&w, &h, 4);
    }
    return w;
}

template <typename T, class Shape>
__device__ void prefill_softmax(const PrefillParams& p, typename Shape::Smem& sm, uint32_t tmem, int warp,
                                int lane, const PrefillTile& w) {
    constexpr int BN = Shape::BN;
    constexpr int D = Shape::SLABS * 64;
    constexpr bool SPLIT_P = std::is_same<T, __nv_bfloat16>::value;
    const float NEG_INF = __int_as_float(0xff800000);
    const uint64_t lim = p.wait_limit_ns;
    const int r = warp * 32 + lane;
    const int t = r >> p.group_shift;
    const int g = r & ((1 << p.group_shift) - 1);
    const int i = w.q0 + t;
    const bool valid = i < w.n;
    // Last position this row attends: its own (causal within the chunk).
    // Rows past the chunk's end compute something finite and are not stored.
    const int last = valid ? w.ctx - w.n + i : w.kv_end - 1;
    const uint32_t row_addr = tmem + ((uint32_t)(warp * 32) << 16);
    const float c = p.scale_log2;
    float m = NEG_INF, l = 0.f;
    bool ok = true;

    for (int j = 0; j < w.nt; ++j) {
        const int b = j & 1;
        ok = __all_sync(kFullMask, mbar_wait_bounded(&sm.s_full[b], (uint32_t)(j >> 1) & 1u, lim));
        if (!ok) break;
        tc_fence_after_sync();
        float x[BN];
#pragma unroll
        for (int h = 0; h < BN / 64; ++h) {
            uint32_t u[64];
            tmem_ld_x64(row_addr + b * BN + h * 64, u);
#pragma unroll
            for (int k = 0; k < 64; ++k) x[h * 64 + k] = __uint_as_float(u[k]);
        }

        // Scores in base-2 units; positions after `last` get -inf.  Eight
        // independent partial maxima / sums keep the dependency chains short.
        const int kv0 = j * BN;
        float pm[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) pm[q] = NEG_INF;
        if (kv0 + BN - 1 <= last) {
#pragma unroll
            for (int k = 0; k < BN; ++k) {
                x[k] *= c;
                pm[k & 7] = fmaxf(pm[k & 7], x[k]);
            }
        } else {
#pragma unroll
            for (int k = 0; k < BN; ++k) {
                x[k] = kv0 + k <= last ? x[k] * c : NEG_INF;
                pm[k & 7] = fmaxf(pm[k & 7], x[k]);
            }
        }
        const float mx = fmaxf(fmaxf(fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3])),
                               fmaxf(fmaxf(pm[4], pm[5]), fmaxf(pm[6], pm[7])));
        const float m_new = fmaxf(m, mx);
        const bool grow = m_new > m + 8.f;  // always on the first tile (m = -inf)
        float alpha = 1.f;
        if (grow) {
            alpha = exp2_approx(m - m_new);
            m = m_new;
            l *= alpha;
        }
        float ps[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) ps[q] = 0.f;
#pragma unroll
        for (int k = 0; k < BN; ++k) {
            x[k] = exp2_approx(x[k] - m);
            ps[k & 7] += x[k];
        }
        l += ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));

        // P over S in TMEM.  bf16: P = P_hi + P_lo, both truncated to 16
        // bits (relative error below 2^-14); f16: P rounded once (2^-11).
        {
            uint32_t u[64];
            if constexpr (SPLIT_P) {
#pragma unroll
                for (int k = 0; k < 64; ++k) u[k] = pack_hi_halves(x[2 * k], x[2 * k + 1]);
                tmem_st_x64(row_addr + b * BN, u);
#pragma unroll
                for (int k = 0; k < 64; ++k) {
                    const float a = x[2 * k] - __uint_as_float(__float_as_uint(x[2 * k]) & 0xffff0000u);
                    const float e = x[2 * k + 1] - __uint_as_float(__float_as_uint(x[2 * k + 1]) & 0xffff0000u);
                    u[k] = pack_hi_halves(a, e);
                }
                tmem_st_x64(row_addr + b * BN + BN / 2, u);
            } else {
#pragma unroll
                for (int k = 0; k < 64; ++k) u[k] = pack_rn<T>(x[2 * k], x[2 * k + 1]);
                tmem_st_x64(row_addr + b * BN, u);
            }
        }

        // Value rows past kv_end (slots after the context, blocks not loaded)
        // may hold anything, NaN included; their weight is 0 but 0 * NaN is
        // NaN, so the last tile's rows there are zeroed.
        if (j == w.nt - 1 && w.kv_end - kv0 < BN) {
            const int st = j % Shape::NSTAGE;
            ok = __all_sync(kFullMask,
                            mbar_wait_bounded(&sm.v_full[st], (uint32_t)(j / Shape::NSTAGE) & 1u, lim));
            if (!ok) break;
            if (r >= w.kv_end - kv0) {
#pragma unroll
                for (int slab = 0; slab < Shape::SLABS; ++slab) {
                    uint4* row = reinterpret_cast<uint4*>(sm.v[st][slab] + r * 128);
#pragma unroll
                    for (int k = 0; k < 8; ++k) row[k] = make_uint4(0u, 0u, 0u, 0u);
                }
            }
            fence_proxy_async_smem();
        }
        // A grown max rescales O, once P_{j-1} V_{j-1} has completed.
        if (j >= 1 && __any_sync(kFullMask, grow)) {
            const int pb = (j - 1) & 1;
            ok = __all_sync(kFullMask, mbar_wait_bounded(&sm.pv_done[pb], (uint32_t)((j - 1) >> 1) & 1u, lim));
            if (!ok) break;
            tc_fence_after_sync();
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t u[32];
                tmem_ld_x32(row_addr + Shape::O_COL + c0, u);
#pragma unroll
                for (int k = 0; k < 32; ++k) u[k] = __float_as_uint(__uint_as_float(u[k]) * alpha);
                tmem_st_x32(row_addr + Shape::O_COL + c0, u);
            }
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.p_full[b]);
    }
    const int lb = (w.nt - 1) & 1;
    if (ok) ok = __all_sync(kFullMask, mbar_wait_bounded(&sm.pv_done[lb], (uint32_t)((w.nt - 1) >> 1) & 1u, lim));
    if (!ok) {
        if (lane == 0) prefill_abort(p, sm);
        return;
    }
    tc_fence_after_sync();
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const int64_t orow = ((int64_t)(w.qrow0 + t) * p.num_heads + ((int64_t)w.kv_head << p.group_shift) + g) * D;
#pragma unroll 1
    for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t u[32];
        tmem_ld_x32(row_addr + Shape::O_COL + c0, u);
        if (valid) {
#pragma unroll
            for (int k = 0; k < 32; k += 4)
                store_out4(p.out, p.out_dtype, orow + c0 + k,
                           make_float4(__uint_as_float(u[k]) * inv, __uint_as_float(u[k + 1]) * inv,
                                       __uint_as_float(u[k + 2]) * inv, __uint_as_float(u[k + 3]) * inv));
        }
    }
}

// ---------------------------------------------------------------------------
// the kernel: one CTA per (query tile, sequence, KV head)
// ---------------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(PrefillShape<D>::THREADS, 1)
    prefill_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap tmap_q,
                   const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v) {
    using Shape = PrefillShape<D>;
    using Smem = typename Shape::Smem;
    constexpr bool BF16 = std::is_same<T, __nv_bfloat16>::value;
    constexpr uint32_t IDESC_S = mma_idesc_f16(BF16, false, Shape::BM, Shape::BN);
    constexpr uint32_t IDESC_O = mma_idesc_f16(BF16, true, Shape::BM, D);
    extern __shared__ uint8_t prefill_smem_raw[];

    // Block index -> (query tile, sequence, KV head); the last query tiles of
    // every sequence (the longest key ranges) come first.
    PrefillTile w;
    int u = blockIdx.x;
    w.kv_head = u % p.num_kv_heads;
    u /= p.num_kv_heads;
    w.seq = u % p.num_seqs;
    const int qt = p.tiles_per_seq - 1 - u / p.num_seqs;

    // The cache write before this kernel may still be finishing.
    pdl_wait_prerequisites();
    const int qs0 = __ldg(p.query_start + w.seq), qs1 = __ldg(p.query_start + w.seq + 1);
    w.ctx = __ldg(p.context_lens + w.seq);
    w.n = qs1 - qs0;
    if (qs0 < 0 || w.n < 0 || qs1 > p.num_tokens || w.n > p.max_query_len || w.ctx < w.n || w.ctx > p.ctx_cap) {
        if (threadIdx.x == 0 && w.kv_head == 0 && qt == 0) set_error(p.err, PA_DEVERR_CONTEXT_LEN);
        return;
    }
    w.q0 = qt * p.tile_tokens;
    if (w.q0 >= w.n) return;  // the whole CTA leaves, before any set-up
    w.qrow0 = qs0 + w.q0;
    w.kv_end = w.ctx - w.n + w.q0 + min(p.tile_tokens, w.n - w.q0);
    w.nt = (w.kv_end + Shape::BN - 1) / Shape::BN;

    const uintptr_t a = reinterpret_cast<uintptr_t>(prefill_smem_raw);
    Smem& sm = *reinterpret_cast<Smem*>((a + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        mbar_init(&sm.q_full, 1);
        for (int st = 0; st < Shape::NSTAGE; ++st) {
            mbar_init(&sm.k_full[st], 1);
            mbar_init(&sm.v_full[st], 1);
            mbar_init(&sm.kv_empty[st], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sm.s_full[b], 1);
            mbar_init(&sm.p_full[b], Shape::SOFTMAX_WARPS);
            mbar_init(&sm.pv_done[b], 1);
        }
        mbar_init(&sm.mma_done, 1);
        sm.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == Shape::MMA_WARP) tmem_alloc(&sm.tmem_base, Shape::TMEM_COLS);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = sm.tmem_base;

    if (warp == Shape::PRODUCER_WARP) {
        prefill_producer<Shape>(p, sm, lane, w, &tmap_q, &tmap_k, &tmap_v);
    } else if (warp == Shape::MMA_WARP) {
        if (lane == 0) prefill_mma<Shape, IDESC_S, IDESC_O, BF16>(p, sm, tmem, w.nt);
        __syncwarp();
    } else {
        prefill_softmax<T, Shape>(p, sm, tmem, warp, lane, w);
    }

    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (warp == Shape::MMA_WARP) tmem_dealloc(tmem, Shape::TMEM_COLS);
}

}  // namespace pa
