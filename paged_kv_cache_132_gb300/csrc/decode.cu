// decode.cu -- the planning kernel of a decode call, the workspace layout and
// the dispatch to the element-type translation units.
//
// The planning kernel turns the context lengths into the work list of
// (sequence, partition) pairs -- a sequence of n tokens has ceil(n / P)
// partitions of P tokens, at least one -- resets the work counter and the
// per-(sequence, KV head) merge counters, and records the item count.  It
// runs first in the stream, so the decode kernel finds a ready list and a
// clean workspace on every call.
#include "common.cuh"
#include "kernels.h"

namespace pa {

cudaError_t launch_decode_f32(const DecodeParams& p, int head_dim, int block_size, int group, int ub,
                              cudaStream_t stream);
cudaError_t launch_decode_simt_f16(const DecodeParams& p, int head_dim, int block_size, int group, int ub,
                                  cudaStream_t stream);
cudaError_t launch_decode_simt_bf16(const DecodeParams& p, int head_dim, int block_size, int group, int ub,
                                   cudaStream_t stream);
cudaError_t launch_decode_mma_f16(const DecodeParams& p, int head_dim, int block_size, int group, int ub,
                                 const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t stream);
cudaError_t launch_decode_mma_bf16(const DecodeParams& p, int head_dim, int block_size, int group, int ub,
                                  const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t stream);

namespace {

constexpr int kPlanThreads = 1024;

__global__ void __launch_bounds__(kPlanThreads) decode_plan_kernel(const __grid_constant__ DecodeParams p) {
    __shared__ int warp_total[32];
    __shared__ int carry;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t units = (int64_t)p.num_seqs * p.num_kv_heads;
    for (int64_t i = tid; i < units; i += kPlanThreads) p.counters[i] = 0;
    if (tid == 0) {
        carry = 0;
        *p.next_item = 0;
    }
    __syncthreads();
    for (int base = 0; base < p.num_seqs; base += kPlanThreads) {
        const int s = base + tid;
        int np = 0;
        if (s < p.num_seqs) {
            int ctx = p.context_lens[s];
            if (ctx < 0 || ctx > p.ctx_cap) {
                set_error(p.err, PA_DEVERR_CONTEXT_LEN);
                ctx = ctx < 0 ? 0 : p.ctx_cap;
            }
            np = ctx == 0 ? 1 : (ctx + p.partition_size - 1) / p.partition_size;
        }
        // Inclusive scan of np over the CTA.
        int x = np;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, off);
            if (lane >= off) x += y;
        }
        if (lane == 31) warp_total[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int t = warp_total[lane];
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, t, off);
                if (lane >= off) t += y;
            }
            warp_total[lane] = t;
        }
        __syncthreads();
        const int inclusive = x + (warp > 0 ? warp_total[warp - 1] : 0);
        const int first = carry + inclusive - np;
        for (int k = 0; k < np; ++k) p.items[first + k] = make_int2(s, k);
        __syncthreads();
        if (tid == kPlanThreads - 1) carry += inclusive;
        __syncthreads();
    }
    if (tid == 0) *p.num_items = carry * p.num_kv_heads;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace

int decode_stage_tokens(int head_dim, int elem_bytes) {
    const int row = head_dim * elem_bytes;
    const int t = 32768 / (2 * row);
    return t < 64 ? t : 64;
}

DecodeWorkspaceLayout decode_workspace_layout(int num_seqs, int num_heads, int max_parts, int head_dim) {
    DecodeWorkspaceLayout w{};
    const size_t s = (size_t)num_seqs, h = (size_t)num_heads, mp = (size_t)max_parts;
    size_t off = 0;
    w.next_item = off;
    w.num_items = off + 4;
    off = 256;
    w.items = off;
    off = align_up(off + s * mp * sizeof(int2), 256);
    w.counters = off;
    off = align_up(off + s * h * sizeof(int), 256);
    w.part_ml = off;
    off = align_up(off + s * h * mp * 2 * sizeof(float), 256);
    w.part_o = off;
    off = align_up(off + s * h * mp * (size_t)head_dim * sizeof(float), 256);
    w.total = off;
    return w;
}

cudaError_t launch_decode(const DecodeParams& p, int dtype, int head_dim, int block_size, int group,
                          int grid_items_upper_bound, DecodeVariant variant, const CUtensorMap* tmap_k,
                          const CUtensorMap* tmap_v, cudaStream_t stream) {
    const int ub = grid_items_upper_bound;
    const bool mma = variant == kDecodeMma && dtype != PA_F32 && tmap_k && tmap_v;
    decode_plan_kernel<<<1, kPlanThreads, 0, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    switch (dtype) {
        case PA_F32: return launch_decode_f32(p, head_dim, block_size, group, ub, stream);
        case PA_F16:
            return mma ? launch_decode_mma_f16(p, head_dim, block_size, group, ub, *tmap_k, *tmap_v, stream)
                       : launch_decode_simt_f16(p, head_dim, block_size, group, ub, stream);
        case PA_BF16:
            return mma ? launch_decode_mma_bf16(p, head_dim, block_size, group, ub, *tmap_k, *tmap_v, stream)
                       : launch_decode_simt_bf16(p, head_dim, block_size, group, ub, stream);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace pa
