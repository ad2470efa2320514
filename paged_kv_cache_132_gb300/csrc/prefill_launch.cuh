// prefill_launch.cuh -- launch of one prefill kernel instance: one CTA per
// (query tile, sequence, KV head), 224 threads, two CTAs per SM, launched as
// a programmatic dependent of the cache write before it.
#pragma once

#include "prefill.cuh"

namespace pa {

template <typename T, int D>
cudaError_t launch_prefill_t(const PrefillParams& p, const CUtensorMap* tq, const CUtensorMap* tk,
                             const CUtensorMap* tv, cudaStream_t stream) {
    using Shape = PrefillShape<D>;
    constexpr int kMaxDevices = 64;
    static int configured[kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (!__atomic_load_n(&configured[dev], __ATOMIC_ACQUIRE)) {
        e = cudaFuncSetAttribute(prefill_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Shape::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        __atomic_store_n(&configured[dev], 1, __ATOMIC_RELEASE);
    }
    const long long grid = (long long)p.num_seqs * p.tiles_per_seq * p.num_kv_heads;
    if (grid <= 0) return cudaSuccess;
    if (grid > 0x7fffffffLL) return cudaErrorNotSupported;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(Shape::THREADS);
    cfg.dynamicSmemBytes = Shape::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, prefill_kernel<T, D>, p, *tq, *tk, *tv);
}

}  // namespace pa
