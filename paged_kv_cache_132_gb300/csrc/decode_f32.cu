// decode_f32.cu -- decode kernels for binary32 pools (CUDA cores).
#include "decode_dispatch.cuh"

namespace pa {

cudaError_t launch_decode_f32(const DecodeParams& p, int head_dim, int block_size, int group, int ub,
                              cudaStream_t stream) {
    return dispatch_decode_simt<float>(p, head_dim, block_size, group, ub, stream);
}

}  // namespace pa
