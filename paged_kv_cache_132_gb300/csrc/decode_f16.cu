// decode_f16.cu -- decode kernels for __half pools (one translation unit per
// element type, so that the build compiles them in parallel).
#include "decode_simt.cuh"

namespace pa {

cudaError_t launch_decode_f16(const DecodeParams& p, int head_dim, int block_size, int group, int ub,
                            cudaStream_t stream) {
    return dispatch_decode_simt<__half>(p, head_dim, block_size, group, ub, stream);
}

}  // namespace pa
