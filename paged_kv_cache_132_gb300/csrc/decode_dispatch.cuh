// decode_dispatch.cuh -- instantiate the decode kernels for every supported
// (head_dim, block_size, group) of one element type.
#pragma once

#include "decode_mma.cuh"
#include "decode_simt.cuh"

#define PA_FOR_EACH_DECODE_SHAPE(CASE) \
    CASE(64, 8, 1) CASE(64, 8, 2) CASE(64, 8, 4) CASE(64, 8, 8)          \
    CASE(64, 16, 1) CASE(64, 16, 2) CASE(64, 16, 4) CASE(64, 16, 8)      \
    CASE(64, 32, 1) CASE(64, 32, 2) CASE(64, 32, 4) CASE(64, 32, 8)      \
    CASE(128, 8, 1) CASE(128, 8, 2) CASE(128, 8, 4) CASE(128, 8, 8)      \
    CASE(128, 16, 1) CASE(128, 16, 2) CASE(128, 16, 4) CASE(128, 16, 8)  \
    CASE(128, 32, 1) CASE(128, 32, 2) CASE(128, 32, 4) CASE(128, 32, 8)

namespace pa {

template <typename T>
cudaError_t dispatch_decode_simt(const DecodeParams& p, int head_dim, int block_size, int group, int ub,
                                 cudaStream_t stream) {
#define PA_SIMT_CASE(DD, BB, GG)                                                                   \
    if (head_dim == DD && block_size == BB && group == GG)                                        \
        return launch_persistent<DecodeShape<T, DD, BB, GG>>(decode_simt_kernel<T, DD, BB, GG>, ub, stream, p);
    PA_FOR_EACH_DECODE_SHAPE(PA_SIMT_CASE)
#undef PA_SIMT_CASE
    return cudaErrorNotSupported;
}

template <typename T>
cudaError_t dispatch_decode_mma(const DecodeParams& p, int head_dim, int block_size, int group, int ub,
                                const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t stream) {
#define PA_MMA_CASE(DD, BB, GG)                                                                     \
    if (head_dim == DD && block_size == BB && group == GG)                                         \
        return launch_persistent<DecodeShape<T, DD, BB, GG>>(decode_mma_kernel<T, DD, BB, GG>, ub, stream, p, tk, tv);
    PA_FOR_EACH_DECODE_SHAPE(PA_MMA_CASE)
#undef PA_MMA_CASE
    return cudaErrorNotSupported;
}

}  // namespace pa
