// decode_simt_f16.cu -- CUDA-core decode kernels for __half pools.
#include "decode_dispatch.cuh"

namespace pa {

cudaError_t launch_decode_simt_f16(const DecodeParams& p, int head_dim, int block_size, int group, int ub,
                                  cudaStream_t stream) {
    return dispatch_decode_simt<__half>(p, head_dim, block_size, group, ub, stream);
}

}  // namespace pa
