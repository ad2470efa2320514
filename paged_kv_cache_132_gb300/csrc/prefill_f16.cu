// Prefill kernels for f16 pools (head_dim 64 and 128).
#include "prefill_launch.cuh"

namespace pa {
cudaError_t launch_prefill_f16(const PrefillParams& p, int head_dim, const CUtensorMap* tq, const CUtensorMap* tk,
                               const CUtensorMap* tv, cudaStream_t stream) {
    if (head_dim == 64) return launch_prefill_t<__half, 64>(p, tq, tk, tv, stream);
    if (head_dim == 128) return launch_prefill_t<__half, 128>(p, tq, tk, tv, stream);
    return cudaErrorNotSupported;
}
}  // namespace pa
