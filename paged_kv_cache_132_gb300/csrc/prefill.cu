// prefill.cu -- dispatch of the prefill launch by pool dtype.
#include "kernels.h"
#include "../../include/pa.h"

namespace pa {

cudaError_t launch_prefill_f16(const PrefillParams& p, int head_dim, const CUtensorMap* tq, const CUtensorMap* tk,
                               const CUtensorMap* tv, cudaStream_t stream);
cudaError_t launch_prefill_bf16(const PrefillParams& p, int head_dim, const CUtensorMap* tq,
                                const CUtensorMap* tk, const CUtensorMap* tv, cudaStream_t stream);

cudaError_t launch_prefill(const PrefillParams& p, int dtype, int head_dim, const CUtensorMap* tmap_q,
                           const CUtensorMap* tmap_k, const CUtensorMap* tmap_v, cudaStream_t stream) {
    if (dtype == PA_F16) return launch_prefill_f16(p, head_dim, tmap_q, tmap_k, tmap_v, stream);
    if (dtype == PA_BF16) return launch_prefill_bf16(p, head_dim, tmap_q, tmap_k, tmap_v, stream);
    return cudaErrorNotSupported;
}

}  // namespace pa
