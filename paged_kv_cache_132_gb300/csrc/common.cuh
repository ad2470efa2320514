// common.cuh -- device helpers shared by the library's kernels (sm_103a).
//
// Inline PTX for the pieces of the Blackwell memory pipeline the kernels use:
// mbarrier phases with bounded waits, bulk copies global->shared completed on
// an mbarrier, and the base-2 exponential.  Nothing here traps: a wait that
// runs out reports failure to its caller, which records PA_DEVERR_TIMEOUT.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "../../include/pa.h"

namespace pa {

// ---------------------------------------------------------------------------
// element types
// ---------------------------------------------------------------------------
// Unpack one 16-byte chunk (4 x f32, or 8 x 16-bit) to fp32.
__device__ inline void unpack16(const uint4& w, float* out, float) {
    out[0] = __uint_as_float(w.x);
    out[1] = __uint_as_float(w.y);
    out[2] = __uint_as_float(w.z);
    out[3] = __uint_as_float(w.w);
}
__device__ inline void unpack16(const uint4& w, float* out, __nv_bfloat16) {
    // A bfloat16 is the high half of a binary32: shift or mask it into place.
    const uint32_t v[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        out[2 * i] = __uint_as_float(v[i] << 16);
        out[2 * i + 1] = __uint_as_float(v[i] & 0xffff0000u);
    }
}
__device__ inline void unpack16(const uint4& w, float* out, __half) {
    const uint32_t v[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __half2 h2;
        memcpy(&h2, &v[i], 4);
        float2 f = __half22float2(h2);
        out[2 * i] = f.x;
        out[2 * i + 1] = f.y;
    }
}

// ---------------------------------------------------------------------------
// math
// ---------------------------------------------------------------------------
// 2^x with the hardware's approximate base-2 exponential (ex2(-inf) = +0).
__device__ inline float exp2_approx(float x) {
    float y;
    asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ---------------------------------------------------------------------------
// shared-memory addresses, mbarriers, bulk copies
// ---------------------------------------------------------------------------
__device__ inline uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ inline void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ inline void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ inline void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ inline void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ inline bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ inline uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase of `bar` with the given parity to complete, for at most
// `limit_ns` nanoseconds of wall time.  Returns false if the limit ran out.
__device__ inline bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t start = global_timer_ns();
    while (true) {
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (global_timer_ns() - start > limit_ns) return false;
    }
}

// Bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned) from
// global memory into this CTA's shared memory; completion is counted on `bar`.
__device__ inline void bulk_copy_g2s(void* smem_dst, const void* gmem_src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(smem_dst)),
        "l"(gmem_src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// Programmatic dependent launch: let the next kernel in the stream start
// launching, and (in that kernel) wait until the previous one has completed
// and its memory is visible.  Without the launch attribute both are no-ops.
__device__ inline void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ inline void pdl_wait_prerequisites() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ inline void set_error(int* err, int bits) {
    if (err) atomicOr(err, bits);
}

}  // namespace pa
