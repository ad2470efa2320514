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
// and values are streamed in tiles of 64 positions.  Per tile j:
//   S_j = Q K_j^T          tcgen05.mma, M=128 N=64 K=d, into TMEM (2 buffers)
//   P_j = 2^(S_j*c - m)    softmax warps, one thread per row; P is written
//                          over S_j in TMEM as 16-bit values
//   O  += P_j V_j          tcgen05.mma with A = P read from TMEM,
//                          M=128 N=d K=64, O in TMEM
// with the running max m kept in base-2 units (c = scale * log2 e) and O
// rescaled only when a row's max grows by more than 8 (a factor of 256).
// For bf16 pools P = P_hi + P_lo (two bf16 halves, two P.V products), which
// keeps the output error near 2^-14 relative instead of the 2^-9 of one
// bf16 rounding; f16 keeps one rounding (2^-11).
//
// Two CTAs share an SM (each ~97 KiB of shared memory and 256 TMEM columns):
// while one waits on its chain S_j -> softmax_j -> P_j V_j, the other's
// MMAs keep the tensor cores busy, and one CTA's set-up and epilogue overlap
// the other's work.
//
// Warp roles (224 threads):
//   warps 0-3 softmax: thread r owns row r = TMEM lane r: mask,
//             exponentials, row sums, P, the rare rescale of O, and at the
//             end O / sum;
//   warp 4    producer of Q (once; 3-D tensor copy: 128/G tokens x G heads
//             x 64-element slabs) and of the K tiles, through the block
//             table, one 2-D tensor copy per (block, 64-element slab), into
//             a ring of slots released as soon as S_j has completed;
//   warp 5    producer of the V tiles, likewise (slots released when
//             P_j V_j has completed); it also zeroes the rows of the last V
//             tile past kv_end (slots after the context may hold NaN);
//   warp 6    MMA issuer (one thread) and owner of the TMEM allocation.
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
    static constexpr int BM = 128;                 // query rows per CTA
    static constexpr int BN = 64;                  // key/value positions per tile
    static constexpr int SLABS = D / 64;           // 64-element (128-byte) column slabs of a row
    static constexpr int Q_SLAB = BM * 128;        // bytes of one Q slab
    static constexpr int KV_SLAB = BN * 128;       // bytes of one K or V slab
    static constexpr int NSTAGE = D == 128 ? 2 : 4;
    static constexpr int SOFTMAX_WARPS = 4;
    static constexpr int K_WARP = 4;    // Q and the K tiles
    static constexpr int V_WARP = 5;    // the V tiles
    static constexpr int MMA_WARP = 6;
    static constexpr int THREADS = 7 * 32;
    static constexpr int CTAS_PER_SM = 2;
    static constexpr uint32_t TMEM_COLS = 256;     // half of an SM's: two CTAs
    // TMEM columns: S buffer b at b*BN; its P (16-bit, two per column) is
    // written over it: P (or P_hi) in the first BN/2 columns, P_lo in the
    // next BN/2.  The output accumulator O after the two buffers.
    static constexpr uint32_t O_COL = 2 * BN;
    static_assert(D == 64 || D == 128, "head_dim 64 or 128");
    static_assert(O_COL + D <= TMEM_COLS, "TMEM columns");

    struct Smem {
        alignas(1024) uint8_t q[SLABS][Q_SLAB];
        alignas(1024) uint8_t k[NSTAGE][SLABS][KV_SLAB];
        alignas(1024) uint8_t v[NSTAGE][SLABS][KV_SLAB];
        uint64_t q_full;
        uint64_t k_full[NSTAGE];
        uint64_t v_full[NSTAGE];
        uint64_t k_empty[NSTAGE];  // S_j complete: K slot free (MMA commit)
        uint64_t v_empty[NSTAGE];  // P_j V_j complete: V slot free (MMA commit)
        uint64_t s_full[2];    // S_j in buffer j % 2 (MMA commit)
        uint64_t p_full[2];    // P_j written over it (softmax warps)
        uint64_t pv_done[2];   // P_j V_j complete: buffer j % 2 free again
        uint64_t v_tail;       // last V tile landed, its rows past kv_end zeroed (V producer)
        uint64_t mma_done;
        uint32_t tmem_base;
        int abort_flag;
    };
    static constexpr int SMEM_BYTES = (int)sizeof(Smem) + 1024;
    // Two CTAs per SM, and never three: the two 256-column TMEM allocations
    // then never wait for one another.
    static_assert(SMEM_BYTES <= 113 * 1024 && 3 * (SMEM_BYTES + 1024) > 228 * 1024, "two CTAs per SM");
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

// Non-blocking test of an mbarrier phase (the MMA issuer polls two
// conditions and must not sleep on either).
__device__ inline bool mbar_test(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
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
// One producer warp streams either the K tiles (and Q first) or the V tiles
// of the CTA's positions into its ring; slot st of tile j is refilled once
// the MMA that read tile j - NSTAGE from it has completed (empty[st]).
template <class Shape, bool IS_K>
__device__ void prefill_producer(const PrefillParams& p, typename Shape::Smem& sm, int lane, const PrefillTile& w,
                                 const CUtensorMap* tq, const CUtensorMap* tkv) {
    const int BS = p.block_size;
    const uint32_t box_bytes = (uint32_t)BS * 128u;
    const int32_t* trow = p.block_tables + (int64_t)w.seq * p.max_blocks;
    const uint64_t lim = p.wait_limit_ns;
    uint64_t* full = IS_K ? sm.k_full : sm.v_full;
    uint64_t* empty = IS_K ? sm.k_empty : sm.v_empty;
    if (IS_K && lane == 0) {
        mbar_arrive_expect_tx(&sm.q_full, Shape::SLABS * Shape::Q_SLAB);
#pragma unroll
        for (int slab = 0; slab < Shape::SLABS; ++slab)
            tma_load_3d_plain(sm.q[slab], tq, slab * 64, w.kv_head << p.group_shift, w.qrow0, &sm.q_full);
    }
    // Blocks of tile jj: lane l < (blocks of the tile) holds its l-th
    // physical block, other lanes -2.  Each entry is loaded two tiles before
    // its use (the loop body runs twice per iteration so that no copy of a
    // register still in flight is needed).
    auto blocks_of = [&](int jj) -> int {
        if (jj >= w.nt) return -2;
        const int kv0 = jj * Shape::BN;
        const int nblk = (min(Shape::BN, w.kv_end - kv0) + BS - 1) / BS;  // <= 8: block_size >= 8
        return lane < nblk ? __ldg(trow + kv0 / BS + lane) : -2;
    };
    uint32_t fill = 0, par = 0;  // per slot: filled / parity of its last fill
    bool ok_run = true;
    int ea = blocks_of(0), eb = blocks_of(1);
    for (int j = 0; j < w.nt; j += 2) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int jj = j + h;
            if (jj >= w.nt) break;
            const int phys = h == 0 ? ea : eb;
            const int st = jj % Shape::NSTAGE;
            const uint32_t ph = (uint32_t)(jj / Shape::NSTAGE) & 1u;
            const bool needed = phys != -2;
            const bool ok = needed && phys >= 0 && (int64_t)phys < p.num_blocks;
            if (IS_K && needed && !ok) set_error(p.err, PA_DEVERR_BLOCK_ID);
            const uint32_t bytes = (uint32_t)__popc(__ballot_sync(kFullMask, ok)) * Shape::SLABS * box_bytes;
            bool free_ok = true;
            if (lane == 0) free_ok = mbar_wait_bounded(&empty[st], ph ^ 1u, lim);
            if (!__shfl_sync(kFullMask, free_ok, 0)) {
                ok_run = false;
                break;
            }
            if (lane == 0) mbar_arrive_expect_tx(&full[st], bytes);
            __syncwarp();
            if (ok) {
                const int y = (int)(((int64_t)phys * p.num_kv_heads + w.kv_head) * BS);
                uint8_t* dst = IS_K ? sm.k[st][0] : sm.v[st][0];
#pragma unroll
                for (int slab = 0; slab < Shape::SLABS; ++slab)
                    tma_load_2d_plain(dst + slab * Shape::KV_SLAB + lane * box_bytes, tkv, slab * 64, y, &full[st]);
            }
            fill |= 1u << st;
            par = (par & ~(1u << st)) | (ph << st);
            if (h == 0) ea = blocks_of(jj + 2);
            else eb = blocks_of(jj + 2);
        }
        if (!ok_run || *reinterpret_cast<volatile int*>(&sm.abort_flag)) break;
    }
    if (!IS_K && ok_run) {
        // The last V tile: rows past kv_end (slots after the context, blocks
        // not loaded) may hold anything, NaN included; their weight is 0 but
        // 0 * NaN is NaN, so they are zeroed before the last P.V reads the
        // tile.  Done here rather than by the softmax warps, so that the
        // tile's load latency does not delay the last P.
        const int jl = w.nt - 1, st = jl % Shape::NSTAGE;
        const int vrow0 = w.kv_end - jl * Shape::BN;
        // Every lane observes the tile's arrival before writing into it.
        const bool landed = mbar_wait_bounded(&full[st], (uint32_t)(jl / Shape::NSTAGE) & 1u, lim);
        if (__all_sync(kFullMask, landed)) {
            for (int idx = lane; idx < (Shape::BN - vrow0) * Shape::SLABS * 8; idx += 32) {
                const int row = vrow0 + idx / (Shape::SLABS * 8);
                const int rest = idx % (Shape::SLABS * 8);
                reinterpret_cast<uint4*>(sm.v[st][rest >> 3] + row * 128)[rest & 7] = make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.v_tail);
        } else {
            ok_run = false;
        }
    }
    if (!ok_run && lane == 0) prefill_abort(p, sm);
    if (IS_K) pdl_launch_dependents();
    // Every copy this warp issued lands before the CTA exits (bounded).
    if (lane == 0) {
        bool drained = IS_K ? mbar_wait_bounded(&sm.q_full, 0, lim) : true;
        for (int st = 0; st < Shape::NSTAGE; ++st)
            if (fill & (1u << st)) drained = mbar_wait_bounded(&full[st], (par >> st) & 1u, lim) && drained;
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
    // Every operand sits at a fixed shared-memory address: descriptor bases
    // are computed once and each MMA adds a compile-time offset (the start
    // address field is the low 14 bits, address / 16, below 2^14).
    constexpr uint64_t STAGE16 = sizeof(sm.k[0]) >> 4;  // descriptor step between stages
    const uint64_t dq = smem_desc_sw128(smem_addr(sm.q[0]), 16, 1024);
    const uint64_t dk0 = smem_desc_sw128(smem_addr(sm.k[0][0]), 16, 1024);
    const uint64_t dv0 = smem_desc_sw128(smem_addr(sm.v[0][0]), Shape::KV_SLAB, 1024);

    // S_js = Q K_js^T into buffer js % 2; the K slot is released when it completes.
    auto issue_s = [&](int js) {
        const int b = js & 1, st = js % Shape::NSTAGE;
        const uint64_t dk = dk0 + (uint64_t)st * STAGE16;
#pragma unroll
        for (int ks = 0; ks < KS_S; ++ks)
            mma_f16_ss(tmem + b * Shape::BN, dq + (uint64_t)((ks >> 2) * (Shape::Q_SLAB >> 4) + (ks & 3) * 2),
                       dk + (uint64_t)((ks >> 2) * (Shape::KV_SLAB >> 4) + (ks & 3) * 2), IDESC_S,
                       ks > 0 ? 1u : 0u);
        mma_commit(&sm.s_full[b]);
        mma_commit(&sm.k_empty[st]);
    };
    // O += P_jp V_jp: A = P from TMEM (8 columns per 16 positions), B = V
    // MN-major (head_dim along N, slabs Shape::KV_SLAB bytes apart; rows
    // 16 ks .. 16 ks + 15 start 2048 bytes apart).  With SPLIT_P the 16-bit
    // P is P_hi + P_lo and both halves are multiplied.
    auto issue_pv = [&](int jp) {
        const int b = jp & 1, st = jp % Shape::NSTAGE;
        const uint64_t dv = dv0 + (uint64_t)st * STAGE16;
        const uint32_t p_tmem = tmem + b * Shape::BN;
        const uint32_t acc0 = jp > 0 ? 1u : 0u;
#pragma unroll
        for (int ks = 0; ks < KS_O; ++ks)
            mma_f16_ts(tmem + Shape::O_COL, p_tmem + ks * 8, dv + (uint64_t)ks * 128, IDESC_O, ks > 0 ? 1u : acc0);
        if constexpr (SPLIT_P) {
#pragma unroll
            for (int ks = 0; ks < KS_O; ++ks)
                mma_f16_ts(tmem + Shape::O_COL, p_tmem + Shape::BN / 2 + ks * 8, dv + (uint64_t)ks * 128, IDESC_O,
                           1u);
        }
        mma_commit(&sm.pv_done[b]);
        mma_commit(&sm.v_empty[st]);
    };

    // Issue, in order within each kind, whichever is ready first: S_js (its
    // K landed and buffer js % 2 is free: P_{js-2} V_{js-2} complete) or
    // P_jp V_jp (P written, V landed).  At most two S ahead of the P.V.
    bool ok = mbar_wait_bounded(&sm.q_full, 0, lim);
    int js = 0, jp = 0;
    uint64_t idle_since = 0;
    while (ok && jp < nt) {
        bool did = false;
        if (js < nt && js < jp + 2 &&
            mbar_test(&sm.k_full[js % Shape::NSTAGE], (uint32_t)(js / Shape::NSTAGE) & 1u) &&
            mbar_test(&sm.pv_done[js & 1], ((uint32_t)(js >> 1) & 1u) ^ 1u)) {
            tc_fence_after_sync();
            issue_s(js++);
            did = true;
        }
        if (jp < js && mbar_test(&sm.p_full[jp & 1], (uint32_t)(jp >> 1) & 1u) &&
            (jp == nt - 1 ? mbar_test(&sm.v_tail, 0u)
                          : mbar_test(&sm.v_full[jp % Shape::NSTAGE], (uint32_t)(jp / Shape::NSTAGE) & 1u))) {
            tc_fence_after_sync();
            issue_pv(jp++);
            did = true;
        }
        if (did) {
            idle_since = 0;
        } else {
            const uint64_t now = global_timer_ns();
            if (idle_since == 0) idle_since = now;
            else if (now - idle_since > lim) ok = false;
        }
    }
    if (!ok) prefill_abort(p, sm);
    // Nothing this thread issued may still be running when TMEM is released.
    mma_commit(&sm.mma_done);
    if (!mbar_wait_bounded(&sm.mma_done, 0, lim)) set_error(p.err, PA_DEVERR_TIMEOUT);
}

// ---------------------------------------------------------------------------
// softmax warps (thread r = row r = TMEM lane r)
// ---------------------------------------------------------------------------
// Packed pairs of binary32 (Blackwell f32x2 arithmetic): each half is
// rounded to nearest like the scalar instruction, two results per issue.
// (x0, x1) = (x0 * a0 + b0, x1 * a1 + b1)
__device__ __forceinline__ void fma2_rn(float& x0, float& x1, float a0, float a1, float b0, float b1) {
    asm("{\n\t.reg .b64 x, a, b;\n\t"
        "mov.b64 x, {%0, %1};\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
        "fma.rn.f32x2 x, x, a, b;\n\tmov.b64 {%0, %1}, x;\n\t}"
        : "+f"(x0), "+f"(x1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
// (x0, x1) += (y0, y1)
__device__ __forceinline__ void add2_rn(float& x0, float& x1, float y0, float y1) {
    asm("{\n\t.reg .b64 x, y;\n\t"
        "mov.b64 x, {%0, %1};\n\tmov.b64 y, {%2, %3};\n\t"
        "add.rn.f32x2 x, x, y;\n\tmov.b64 {%0, %1}, x;\n\t}"
        : "+f"(x0), "+f"(x1)
        : "f"(y0), "f"(y1));
}
// (x0, x1) -= (y0, y1)
__device__ __forceinline__ void sub2_rn(float& x0, float& x1, float y0, float y1) {
    asm("{\n\t.reg .b64 x, y;\n\t"
        "mov.b64 x, {%0, %1};\n\tmov.b64 y, {%2, %3};\n\t"
        "sub.rn.f32x2 x, x, y;\n\tmov.b64 {%0, %1}, x;\n\t}"
        : "+f"(x0), "+f"(x1)
        : "f"(y0), "f"(y1));
}

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
    const float c = p.scale_log2;  // > 0
    float m = NEG_INF, l = 0.f;
    bool ok = true;

    for (int j = 0; j < w.nt; ++j) {
        const int b = j & 1;
        ok = __all_sync(kFullMask, mbar_wait_bounded(&sm.s_full[b], (uint32_t)(j >> 1) & 1u, lim));
        if (!ok) break;
        tc_fence_after_sync();
        float x[BN];
        {
            uint32_t u[BN];
            tmem_ld_x64(row_addr + b * BN, u);
#pragma unroll
            for (int k = 0; k < BN; ++k) x[k] = __uint_as_float(u[k]);
        }

        // Raw-score maximum (positions after `last` are -inf), with eight
        // independent partial maxima.
        const int kv0 = j * BN;
        if (kv0 + BN - 1 > last) {
#pragma unroll
            for (int k = 0; k < BN; ++k) x[k] = kv0 + k <= last ? x[k] : NEG_INF;
        }
        float pm[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) pm[q] = x[q];
#pragma unroll
        for (int k = 8; k < BN; ++k) pm[k & 7] = fmaxf(pm[k & 7], x[k]);
        const float mx =
            fmaxf(fmaxf(fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3])), fmaxf(fmaxf(pm[4], pm[5]), fmaxf(pm[6], pm[7])));
        // Reference max in base-2 units.
        const float m_new = fmaxf(m, mx * c);
        const bool grow = m_new > m + 8.f;  // always on the first tile (m = -inf)
        float alpha = 1.f;
        if (grow) {
            alpha = exp2_approx(m - m_new);
            m = m_new;
            l *= alpha;
        }
        // Exponent arguments and row sum two positions per instruction
        // (packed f32x2 FMA / add, each half rounded as its scalar form).
        const float nm = -m;
#pragma unroll
        for (int k = 0; k < BN; k += 2) fma2_rn(x[k], x[k + 1], c, c, nm, nm);
#pragma unroll
        for (int k = 0; k < BN; ++k) x[k] = exp2_approx(x[k]);
        float ps[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) ps[q] = x[q];
#pragma unroll
        for (int k = 8; k < BN; k += 2) add2_rn(ps[k & 7], ps[(k & 7) + 1], x[k], x[k + 1]);
        l += ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));

        // P over S in TMEM.  bf16: P = P_hi + P_lo, both truncated to 16 bits
        // (relative error below 2^-14); f16: P rounded once (2^-11).  The
        // stores complete before P's arrival is signalled (one wait below).
        {
            uint32_t u[BN / 2];
            if constexpr (SPLIT_P) {
#pragma unroll
                for (int k = 0; k < BN / 2; ++k) u[k] = pack_hi_halves(x[2 * k], x[2 * k + 1]);
                tmem_st_x32_async(row_addr + b * BN, u);
#pragma unroll
                for (int k = 0; k < BN / 2; ++k) {
                    // P_lo = P - P_hi, exact: P_hi is P with its low 16 bits cleared
                    float a = x[2 * k], e = x[2 * k + 1];
                    sub2_rn(a, e, __uint_as_float(__float_as_uint(a) & 0xffff0000u),
                            __uint_as_float(__float_as_uint(e) & 0xffff0000u));
                    u[k] = pack_hi_halves(a, e);
                }
                tmem_st_x32_async(row_addr + b * BN + BN / 2, u);
            } else {
#pragma unroll
                for (int k = 0; k < BN / 2; ++k) u[k] = pack_rn<T>(x[2 * k], x[2 * k + 1]);
                tmem_st_x32_async(row_addr + b * BN, u);
            }
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
        tmem_wait_st();
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
            if (p.out_dtype == PA_F32) {
#pragma unroll
                for (int k = 0; k < 32; k += 4)
                    store_out4(p.out, p.out_dtype, orow + c0 + k,
                               make_float4(__uint_as_float(u[k]) * inv, __uint_as_float(u[k + 1]) * inv,
                                           __uint_as_float(u[k + 2]) * inv, __uint_as_float(u[k + 3]) * inv));
            } else {
                // 16-bit output: eight values per 16-byte store
#pragma unroll
                for (int k = 0; k < 32; k += 8) {
                    uint4 q;
                    uint32_t* qw = reinterpret_cast<uint32_t*>(&q);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float a = __uint_as_float(u[k + 2 * e]) * inv, b = __uint_as_float(u[k + 2 * e + 1]) * inv;
                        qw[e] = p.out_dtype == PA_F16 ? pack_rn<__half>(a, b) : pack_rn<__nv_bfloat16>(a, b);
                    }
                    *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + orow + c0 + k) = q;
                }
            }
        }
    }
}

// ---------------------------------------------------------------------------
// the kernel: one CTA per (query tile, sequence, KV head)
// ---------------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(PrefillShape<D>::THREADS, PrefillShape<D>::CTAS_PER_SM)
    prefill_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap tmap_q,
                   const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v) {
    using Shape = PrefillShape<D>;
    using Smem = typename Shape::Smem;
    constexpr bool BF16 = std::is_same<T, __nv_bfloat16>::value;
    constexpr uint32_t IDESC_S = mma_idesc_f16(BF16, false, Shape::BM, Shape::BN);
    constexpr uint32_t IDESC_O = mma_idesc_f16(BF16, true, Shape::BM, D);
    extern __shared__ uint8_t prefill_smem_raw[];

    // Block index -> (query tile, sequence, KV head).  Level order (the
    // default): the last query tiles of every sequence (the longest key
    // ranges) first, then the next level, and so on.  When the pools exceed
    // L2 every level would read them from HBM again, so then the query tiles
    // of one (sequence, KV head) are adjacent instead (last tile first) and
    // its keys and values stay in L2 while they are read.
    PrefillTile w;
    int u = blockIdx.x;
    int qt;
    if (p.tiles_adjacent) {
        qt = p.tiles_per_seq - 1 - u % p.tiles_per_seq;
        u /= p.tiles_per_seq;
        w.kv_head = u % p.num_kv_heads;
        w.seq = u / p.num_kv_heads;
    } else {
        w.kv_head = u % p.num_kv_heads;
        u /= p.num_kv_heads;
        w.seq = u % p.num_seqs;
        qt = p.tiles_per_seq - 1 - u / p.num_seqs;
    }

    // Fetch the tensor-copy descriptors while the lengths load.
    if (threadIdx.x == 0) {
        prefetch_tensormap(&tmap_q);
        prefetch_tensormap(&tmap_k);
        prefetch_tensormap(&tmap_v);
    }
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
            mbar_init(&sm.k_empty[st], 1);
            mbar_init(&sm.v_empty[st], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sm.s_full[b], 1);
            mbar_init(&sm.p_full[b], Shape::SOFTMAX_WARPS);
            mbar_init(&sm.pv_done[b], 1);
        }
        mbar_init(&sm.v_tail, 1);
        mbar_init(&sm.mma_done, 1);
        sm.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == Shape::MMA_WARP) tmem_alloc(&sm.tmem_base, Shape::TMEM_COLS);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = sm.tmem_base;

    if (warp == Shape::K_WARP) {
        prefill_producer<Shape, true>(p, sm, lane, w, &tmap_q, &tmap_k);
    } else if (warp == Shape::V_WARP) {
        prefill_producer<Shape, false>(p, sm, lane, w, &tmap_q, &tmap_v);
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
