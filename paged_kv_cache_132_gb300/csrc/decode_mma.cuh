// decode_mma.cuh -- decode consumer on the tensor cores (binary16 / bfloat16).
//
// For one KV head the G query heads form a [G x d] tile, and a block of 16
// tokens gives the contractions S = Q K^T ([G x d] x [d x 16]) and
// O += P V ([G x 16] x [16 x d]).  Each is a sequence of m16n8k16 MMAs with
// the G heads on the M dimension (rows G..15 are zero), fp32 accumulation.
//
//  * Q K^T: the A fragments of q are loaded once per item; the B fragments of
//    K come from the stage with ldmatrix.  The stage is filled by tensor
//    copies with 128-byte swizzle (a line's 16-byte chunk k sits at k ^ (line
//    % 8)), so the eight rows an ldmatrix reads fall in eight different bank
//    groups (four with the interleaved layout of 8- and 16-token blocks).
//  * The accumulator of S has exactly the register layout of the A operand of
//    P V (row g = lane/4, tokens 2j, 2j+1 and 8+2j, 8+2j+1 for j = lane%4),
//    so the softmax runs in registers and P feeds the next MMA directly.
//  * P in [0, 1] is split into hi + lo halves of the input precision (hi =
//    round(P), lo = round(P - hi)) and both are multiplied by V: the product
//    then carries ~16 significant bits of P instead of 8 (bfloat16), which
//    keeps the result within the fp32-accumulation error of the exact sum.
//  * V's B fragments come from ldmatrix.trans of the same swizzled stage.
//    Value rows past the context end (stale slots, possibly NaN) are zeroed in
//    registers before the MMA: a zero weight times NaN would be NaN.
#pragma once

#include "decode_common.cuh"

namespace pa {

template <typename T> struct MmaOps;

template <> struct MmaOps<__nv_bfloat16> {
    __device__ static inline void mma(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                      uint32_t b0, uint32_t b1) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
    // (lo element in the low half, hi element in the high half)
    __device__ static inline uint32_t pack(float lo, float hi) {
        __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    }
    __device__ static inline float round_trip(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }
};

template <> struct MmaOps<__half> {
    __device__ static inline void mma(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                      uint32_t b0, uint32_t b1) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
    __device__ static inline uint32_t pack(float lo, float hi) {
        __half2 v = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    }
    __device__ static inline float round_trip(float x) { return __half2float(__float2half_rn(x)); }
};

__device__ inline void ldmatrix_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3, uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ inline void ldmatrix_x4_trans(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3, uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

template <typename T, int D, int BS, int G>
__device__ void mma_consumer(const DecodeParams& p, typename DecodeShape<T, D, BS, G>::Smem& sm, int warp,
                             int lane) {
    using S = DecodeShape<T, D, BS, G>;
    using Ops = MmaOps<T>;
    static_assert(S::E == 2, "tensor-core path takes 16-bit pools");
    static_assert(S::TPW == 16, "each consumer warp takes 16 tokens (one k16 step) per stage");
    static_assert(G <= 8, "the G query heads occupy rows 0..7 of the MMA");
    constexpr int KSTEPS = D / 16;   // k16 steps of Q K^T
    constexpr int NT = D / 8;        // n8 dim tiles of P V
    const float NEG_INF = __int_as_float(0xff800000);
    const int g = lane >> 2;         // accumulator row = query head within the group
    const int j = lane & 3;

    uint32_t qa[KSTEPS][2];  // A fragments of q: (row g, k 2j..2j+1) and (row g, k 8+2j..8+2j+1)
    float o[NT][4];          // P V accumulators; [0..1] = row g, dims 8n+2j, 8n+2j+1
    float m = NEG_INF, l = 0.f;
#pragma unroll
    for (int n = 0; n < NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
#pragma unroll
    for (int k = 0; k < KSTEPS; ++k) qa[k][0] = qa[k][1] = 0u;

    int st = 0;
    uint32_t ph = 0, fph = 0;
    while (true) {
        const bool ok = mbar_wait_bounded(&sm.full[st], ph, p.wait_limit_ns);
        if (!__all_sync(kFullMask, ok)) {
            consumer_abort(p, &sm.abort_flag, lane);
            break;
        }
        const StageMeta mt = sm.meta[st];
        if (mt.item < 0) {
            // No more work: tell the merge warp to stop.
            if (acquire_merge_slot(sm, fph, p.wait_limit_ns)) {
                StageMeta end = mt;
                release_to_merger(sm, end, warp, lane);
            }
            break;
        }

        if (mt.first) {
            const T* qs = reinterpret_cast<const T*>(sm.q[st]);
#pragma unroll
            for (int k = 0; k < KSTEPS; ++k) {
                qa[k][0] = g < G ? *reinterpret_cast<const uint32_t*>(qs + g * D + 16 * k + 2 * j) : 0u;
                qa[k][1] = g < G ? *reinterpret_cast<const uint32_t*>(qs + g * D + 16 * k + 8 + 2 * j) : 0u;
            }
            m = NEG_INF;
            l = 0.f;
#pragma unroll
            for (int n = 0; n < NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
        }

        const int row0 = warp * 16;
        const int tok0 = mt.t0 + row0;  // absolute index of the warp's first token
        if (tok0 < mt.te) {
            const uint32_t kst = smem_addr(sm.kv[st][0]);
            const uint32_t vst = smem_addr(sm.kv[st][1]);
            // ---- S = Q K^T over two n8 tiles (tokens row0..+7, row0+8..+15);
            // even and odd k steps go to separate accumulators (shorter
            // dependency chains), summed afterwards.
            float sacc[2][4], sodd[2][4];
#pragma unroll
            for (int t = 0; t < 2; ++t)
#pragma unroll
                for (int e = 0; e < 4; ++e) sacc[t][e] = sodd[t][e] = 0.f;
#pragma unroll
            for (int kp = 0; kp < KSTEPS / 2; ++kp) {
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    uint32_t b0, b1, b2, b3;
                    ldmatrix_x4(b0, b1, b2, b3,
                                stage_chunk_addr<S>(kst, row0 + t * 8 + (lane & 7), kp * 4 + (lane >> 3)));
                    Ops::mma(sacc[t], qa[2 * kp][0], 0u, qa[2 * kp][1], 0u, b0, b1);
                    Ops::mma(sodd[t], qa[2 * kp + 1][0], 0u, qa[2 * kp + 1][1], 0u, b2, b3);
                }
            }
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                sacc[t][0] += sodd[t][0];
                sacc[t][1] += sodd[t][1];
            }
            // ---- online softmax on row g (tokens 2j, 2j+1, 8+2j, 8+2j+1)
            float sv[4];
            bool valid[4];
#pragma unroll
            for (int t = 0; t < 2; ++t)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    valid[2 * t + e] = tok0 + 8 * t + 2 * j + e < mt.te;
                    sv[2 * t + e] = valid[2 * t + e] ? sacc[t][e] * p.scale_log2 : NEG_INF;
                }
            float mx = fmaxf(fmaxf(sv[0], sv[1]), fmaxf(sv[2], sv[3]));
            mx = fmaxf(mx, __shfl_xor_sync(kFullMask, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(kFullMask, mx, 2));
            if (__any_sync(kFullMask, mx > m)) {
                const float alpha = mx > m ? exp2_approx(m - mx) : 1.f;
                m = fmaxf(m, mx);
                l *= alpha;
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    o[n][0] *= alpha;
                    o[n][1] *= alpha;
                }
            }
            float pr[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                pr[i] = valid[i] ? exp2_approx(sv[i] - m) : 0.f;
                l += pr[i];
            }
            float hi[4], lo[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                hi[i] = Ops::round_trip(pr[i]);
                lo[i] = pr[i] - hi[i];
            }
            const uint32_t ah0 = Ops::pack(hi[0], hi[1]), ah2 = Ops::pack(hi[2], hi[3]);
            const uint32_t al0 = Ops::pack(lo[0], lo[1]), al2 = Ops::pack(lo[2], lo[3]);
            // ---- O += P V over the NT dim tiles, two per ldmatrix.x4.trans
            const bool partial = tok0 + 16 > mt.te;  // warp-uniform
            const uint32_t mask_lo = (valid[0] ? 0x0000ffffu : 0u) | (valid[1] ? 0xffff0000u : 0u);
            const uint32_t mask_hi = (valid[2] ? 0x0000ffffu : 0u) | (valid[3] ? 0xffff0000u : 0u);
#pragma unroll
            for (int dp = 0; dp < NT / 2; ++dp) {
                uint32_t v0, v1, v2, v3;
                ldmatrix_x4_trans(v0, v1, v2, v3,
                                  stage_chunk_addr<S>(vst, row0 + (lane & 7) + ((lane >> 3) & 1) * 8,
                                                      2 * dp + (lane >> 4)));
                if (partial) {
                    v0 &= mask_lo;
                    v2 &= mask_lo;
                    v1 &= mask_hi;
                    v3 &= mask_hi;
                }
                Ops::mma(o[2 * dp], ah0, 0u, ah2, 0u, v0, v1);
                Ops::mma(o[2 * dp], al0, 0u, al2, 0u, v0, v1);
                Ops::mma(o[2 * dp + 1], ah0, 0u, ah2, 0u, v2, v3);
                Ops::mma(o[2 * dp + 1], al0, 0u, al2, 0u, v2, v3);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty[st]);

        if (mt.last) {
            // Hand the item's state to the merge warp and move on.
            float lw = l;
            lw += __shfl_xor_sync(kFullMask, lw, 1);
            lw += __shfl_xor_sync(kFullMask, lw, 2);
            if (!acquire_merge_slot(sm, fph, p.wait_limit_ns)) {
                consumer_abort(p, &sm.abort_flag, lane);
                break;
            }
            if (g < G) {
#pragma unroll
                for (int n = 0; n < NT; ++n)
                    *reinterpret_cast<float2*>(&sm.mo[warp][g][8 * n + 2 * j]) = make_float2(o[n][0], o[n][1]);
                if (j == 0) {
                    sm.mm[warp][g] = m;
                    sm.ml[warp][g] = lw;
                }
            }
            release_to_merger(sm, mt, warp, lane);
            fph ^= 1u;
        }
        if (++st == S::NSTAGE) {
            st = 0;
            ph ^= 1u;
        }
        // Another warp's wait ran out: stop too (decided for the whole warp).
        if (__any_sync(kFullMask, *reinterpret_cast<volatile int*>(&sm.abort_flag) != 0)) break;
    }
}

template <typename T, int D, int BS, int G>
__global__ void __launch_bounds__(DecodeShape<T, D, BS, G>::THREADS, 2)
decode_mma_kernel(const __grid_constant__ DecodeParams p, const __grid_constant__ CUtensorMap tmap_k,
                  const __grid_constant__ CUtensorMap tmap_v) {
    using S = DecodeShape<T, D, BS, G>;
    extern __shared__ uint8_t smem_raw[];
    auto& sm = decode_smem<typename S::Smem>(smem_raw);
    decode_smem_init(sm, S::NSTAGE, S::NCW);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (warp < S::NCW)
        mma_consumer<T, D, BS, G>(p, sm, warp, lane);
    else if (warp == S::PRODUCER_WARP)
        decode_producer<S, BS, G, true>(p, sm, lane, &tmap_k, &tmap_v);
    else
        merge_worker<S, D, G>(p, sm, lane);
}

}  // namespace pa
