// decode_mma_bf16.cu -- tensor-core decode kernels for __nv_bfloat16 pools.
#include "decode_dispatch.cuh"

namespace pa {

cudaError_t launch_decode_mma_bf16(const DecodeParams& p, int head_dim, int block_size, int group, int ub,
                                 const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t stream) {
    return dispatch_decode_mma<__nv_bfloat16>(p, head_dim, block_size, group, ub, tk, tv, stream);
}

}  // namespace pa
