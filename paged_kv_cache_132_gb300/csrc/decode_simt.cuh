// decode_simt.cuh -- decode consumer on the CUDA cores (every element type).
//
// Lanes own 16-byte chunks of a token's row: a warp-wide 16-byte load covers
// TPI = 32 / CPR rows.  Each lane forms partial q.k dot products for the G
// query heads over its chunk, the CPR lanes of a row sum them with shuffles,
// and the running max / sum and the p.v accumulators follow.  Linear bulk
// copies fill the stage: rows are contiguous, so a warp-wide load touches
// consecutive bytes and has no bank conflicts.
#pragma once

#include "decode_common.cuh"

namespace pa {

template <typename T, int D, int BS, int G>
struct SimtShape : DecodeShape<T, D, BS, G> {
    using Base = DecodeShape<T, D, BS, G>;
    static constexpr int VEC = 16 / Base::E;          // elements per 16-byte chunk
    static constexpr int CPR = D / VEC;               // chunks per row
    static_assert(CPR <= 32 && 32 % CPR == 0, "a row maps onto a power-of-two lane group");
    static constexpr int TPI = 32 / CPR;              // rows per warp-wide load
    static_assert(Base::TPW % TPI == 0, "a warp's rows are whole loads");
    static constexpr int RPL = Base::TPW / TPI;       // rows per lane per stage
    static constexpr int RSUB = RPL < 4 ? RPL : 4;    // rows per softmax update
    static_assert(RPL % RSUB == 0, "rows per lane split evenly");
};

template <typename T, int D, int BS, int G>
__device__ void simt_consumer(const DecodeParams& p, typename DecodeShape<T, D, BS, G>::Smem& sm, int warp,
                              int lane) {
    using K = SimtShape<T, D, BS, G>;
    using Base = DecodeShape<T, D, BS, G>;
    constexpr int VEC = K::VEC, CPR = K::CPR, TPI = K::TPI;
    const int tg = lane / CPR;  // row group within a warp-wide load
    const int c = lane % CPR;   // 16-byte chunk of the row this lane owns
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

        const int row0 = warp * Base::TPW;
        if (mt.t0 + row0 < mt.te) {
            const uint8_t* ks = sm.kv[st][0] + row0 * Base::ROW + c * 16;
            const uint8_t* vs = sm.kv[st][1] + row0 * Base::ROW + c * 16;
#pragma unroll
            for (int sub = 0; sub < K::RPL; sub += K::RSUB) {
                float sc[K::RSUB][G];
                bool valid[K::RSUB];
#pragma unroll
                for (int u = 0; u < K::RSUB; ++u) {
                    const int r = (sub + u) * TPI + tg;
                    valid[u] = mt.t0 + row0 + r < mt.te;
                    const uint4 w = *reinterpret_cast<const uint4*>(ks + r * Base::ROW);
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
                            sc[u][g] += __shfl_xor_sync(kFullMask, sc[u][g], off);
                // Row maximum over the warp's valid rows, then a lazy rescale.
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    float mx = NEG_INF;
#pragma unroll
                    for (int u = 0; u < K::RSUB; ++u) mx = valid[u] ? fmaxf(mx, sc[u][g]) : mx;
#pragma unroll
                    for (int off = CPR; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(kFullMask, mx, off));
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
                    const uint4 w = *reinterpret_cast<const uint4*>(vs + r * Base::ROW);
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
            // Sum over the warp's row groups, then hand the item's state to
            // the merge warp and move on.
            if (!acquire_merge_slot(sm, fph, p.wait_limit_ns)) {
                consumer_abort(p, &sm.abort_flag, lane);
                break;
            }
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float lw = l[g];
#pragma unroll
                for (int off = CPR; off < 32; off <<= 1) lw += __shfl_xor_sync(kFullMask, lw, off);
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    float a = acc[g][e];
#pragma unroll
                    for (int off = CPR; off < 32; off <<= 1) a += __shfl_xor_sync(kFullMask, a, off);
                    if (tg == 0) sm.mo[warp][g][c * VEC + e] = a;
                }
                if (lane == 0) {
                    sm.mm[warp][g] = m[g];
                    sm.ml[warp][g] = lw;
                }
            }
            release_to_merger(sm, mt, warp, lane);
            fph ^= 1u;
        }
        if (++st == Base::NSTAGE) {
            st = 0;
            ph ^= 1u;
        }
        // Another warp's wait ran out: stop too (decided for the whole warp).
        if (__any_sync(kFullMask, *reinterpret_cast<volatile int*>(&sm.abort_flag) != 0)) break;
    }
}

template <typename T, int D, int BS, int G>
__global__ void __launch_bounds__(DecodeShape<T, D, BS, G>::THREADS, 2)
decode_simt_kernel(const __grid_constant__ DecodeParams p) {
    using S = DecodeShape<T, D, BS, G>;
    extern __shared__ uint8_t smem_raw[];
    auto& sm = decode_smem<typename S::Smem>(smem_raw);
    decode_smem_init(sm, S::NSTAGE, S::NCW);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (warp < S::NCW)
        simt_consumer<T, D, BS, G>(p, sm, warp, lane);
    else if (warp == S::PRODUCER_WARP)
        decode_producer<S, BS, G, false>(p, sm, lane, nullptr, nullptr);
    else
        merge_worker<S, D, G>(p, sm, lane);
}

}  // namespace pa
