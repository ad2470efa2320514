// decode.cu -- the planning and reduce kernels of a decode call, the
// workspace layout, and the launch sequence plan -> decode -> reduce.
//
// Planning kernel: turns the context lengths into the work list of
// (sequence, partition) pairs -- a sequence of n tokens has ceil(n / P)
// partitions of P tokens, at least one -- lists the sequences that have more
// than one partition, and resets the work counter.  It runs first in the
// stream, so every call finds a ready list and a clean workspace.
//
// Reduce kernel: the cross-partition merge of split-KV ("combine the partial
// results", "PagedAttention paper review", "How does this work?"): for each
// (sequence, query head) with partitions p = 0..P-1 holding the running max
// m_p, sum l_p and normalised output o_p,
//     M = max_p m_p,  L = sum_p l_p 2^(m_p - M),  o = sum_p (l_p 2^(m_p - M) / L) o_p.
// One warp per (sequence, query head); lanes hold 4 consecutive dims, so a
// warp-wide load of one partition's output is one contiguous 512-byte row.
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
constexpr int kReduceThreads = 256;

// Inclusive scan of x over the CTA (kPlanThreads threads); `scratch` holds
// one int per warp.
__device__ int block_inclusive_scan(int x, int* scratch) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += y;
    }
    if (lane == 31) scratch[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int t = scratch[lane];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, t, off);
            if (lane >= off) t += y;
        }
        scratch[lane] = t;
    }
    __syncthreads();
    const int r = x + (warp > 0 ? scratch[warp - 1] : 0);
    __syncthreads();
    return r;
}

__global__ void __launch_bounds__(kPlanThreads) decode_plan_kernel(const __grid_constant__ DecodeParams p) {
    __shared__ int scratch[32];
    __shared__ int carry[2];
    // The decode kernel may launch now; it waits for this grid to complete
    // before it reads the work list.
    pdl_launch_dependents();
    const int tid = threadIdx.x;
    if (tid == 0) {
        carry[0] = carry[1] = 0;
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
        const int multi = np > 1 ? 1 : 0;
        const int items_incl = block_inclusive_scan(np, scratch);
        const int multi_incl = block_inclusive_scan(multi, scratch);
        const int first = carry[0] + items_incl - np;
        for (int k = 0; k < np; ++k) p.items[first + k] = make_int2(s, k);
        if (multi) p.multi_seqs[carry[1] + multi_incl - 1] = make_int2(s, np);
        __syncthreads();
        if (tid == kPlanThreads - 1) {
            carry[0] += items_incl;
            carry[1] += multi_incl;
        }
        __syncthreads();
    }
    if (tid == 0) {
        *p.num_items = carry[0] * p.num_kv_heads;
        *p.num_multi = carry[1];
    }
    // This kernel may have been launched before the previous kernel in the
    // stream finished (it reads nothing that kernel writes); it completes only
    // after that kernel has, so the decode kernel's wait on it covers both.
    pdl_wait_prerequisites();
}

template <int D>
__global__ void __launch_bounds__(kReduceThreads, 5) decode_reduce_kernel(const __grid_constant__ DecodeParams p,
                                                                        int group) {
    constexpr int VPL = D / 32;  // dims per lane (2 or 4)
    pdl_wait_prerequisites();    // the decode kernel wrote the partials
    const float NEG_INF = __int_as_float(0xff800000);
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (kReduceThreads / 32);
    const int per_seq = p.num_kv_heads * group;
    const int64_t total = (int64_t)*p.num_multi * per_seq;
    for (int64_t w = blockIdx.x * (kReduceThreads / 32) + (threadIdx.x >> 5); w < total; w += warps) {
        const int2 sn = p.multi_seqs[w / per_seq];  // (sequence, partitions)
        const int s = sn.x, nparts = sn.y;
        const int hq = (int)(w % per_seq);  // query head h*G + g of sequence s
        const int h = hq / group, g = hq - h * group;
        const int64_t base = ((int64_t)s * p.num_kv_heads + h) * p.max_parts * group + g;
        float acc[VPL];
#pragma unroll
        for (int v = 0; v < VPL; ++v) acc[v] = 0.f;
        // Partitions in chunks of 32, lane q holding partition q's (m, l);
        // a running max M and sum L carry the merge across chunks.  The
        // outputs of a chunk's first kPre partitions are loaded together with
        // the (m, l) pairs (they do not depend on them), so that most
        // sequences (at most kPre partitions) wait for one round trip to L2,
        // not two.
        constexpr int kPre = 4;
        float M = NEG_INF, L = 0.f;
        for (int q0 = 0; q0 < nparts; q0 += 32) {
            float2 ml = make_float2(NEG_INF, 0.f);
            if (q0 + lane < nparts)
                ml = __ldcg(reinterpret_cast<const float2*>(p.part_ml + 2 * (base + (int64_t)(q0 + lane) * group)));
            float pre[kPre][VPL];
#pragma unroll
            for (int k = 0; k < kPre; ++k) {
                const float* src = p.part_o + (base + (int64_t)(q0 + k) * group) * D + lane * VPL;
                if (q0 + k < nparts) {
                    if constexpr (VPL == 4) {
                        const float4 o = __ldcg(reinterpret_cast<const float4*>(src));
                        pre[k][0] = o.x;
                        pre[k][1] = o.y;
                        pre[k][2] = o.z;
                        pre[k][3] = o.w;
                    } else {
                        const float2 o = __ldcg(reinterpret_cast<const float2*>(src));
                        pre[k][0] = o.x;
                        pre[k][1] = o.y;
                    }
                } else {
#pragma unroll
                    for (int v = 0; v < VPL; ++v) pre[k][v] = 0.f;
                }
            }
            float cm = ml.x;
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, off));
            const float newM = fmaxf(M, cm);
            const float rescale = M == NEG_INF ? 0.f : exp2_approx(M - newM);
            const float wq = ml.y > 0.f ? ml.y * exp2_approx(ml.x - newM) : 0.f;  // l_q 2^(m_q - M)
            float cl = wq;
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) cl += __shfl_xor_sync(0xffffffffu, cl, off);
            L = L * rescale + cl;
            M = newM;
#pragma unroll
            for (int v = 0; v < VPL; ++v) acc[v] *= rescale;
            const int n = min(32, nparts - q0);
#pragma unroll
            for (int k = 0; k < kPre; ++k) {
                const float wk = __shfl_sync(0xffffffffu, wq, k);  // 0 for k >= n
#pragma unroll
                for (int v = 0; v < VPL; ++v) acc[v] = fmaf(wk, pre[k][v], acc[v]);
            }
#pragma unroll 8
            for (int k = kPre; k < n; ++k) {
                const float wk = __shfl_sync(0xffffffffu, wq, k);
                const float* src = p.part_o + (base + (int64_t)(q0 + k) * group) * D + lane * VPL;
                if constexpr (VPL == 4) {
                    const float4 o = __ldcg(reinterpret_cast<const float4*>(src));
                    acc[0] = fmaf(wk, o.x, acc[0]);
                    acc[1] = fmaf(wk, o.y, acc[1]);
                    acc[2] = fmaf(wk, o.z, acc[2]);
                    acc[3] = fmaf(wk, o.w, acc[3]);
                } else {
                    const float2 o = __ldcg(reinterpret_cast<const float2*>(src));
                    acc[0] = fmaf(wk, o.x, acc[0]);
                    acc[1] = fmaf(wk, o.y, acc[1]);
                }
            }
        }
        const float invL = 1.f / L;
        const int64_t oi = ((int64_t)s * p.num_heads + (int64_t)h * group + g) * D + lane * VPL;
#pragma unroll
        for (int v = 0; v < VPL; ++v) {
            const float o = acc[v] * invL;
            if (p.out_dtype == PA_F32)
                static_cast<float*>(p.out)[oi + v] = o;
            else if (p.out_dtype == PA_F16)
                static_cast<__half*>(p.out)[oi + v] = __float2half_rn(o);
            else
                static_cast<__nv_bfloat16*>(p.out)[oi + v] = __float2bfloat16_rn(o);
        }
    }
}

cudaError_t launch_reduce(const DecodeParams& p, int head_dim, int group, int sms, cudaStream_t stream) {
    // One warp per (sequence, query head) up to the upper bound of the work;
    // the kernel strides over the real count beyond 8 CTAs per SM.
    const int64_t work = (int64_t)p.num_seqs * p.num_heads;
    int64_t ctas = (work + kReduceThreads / 32 - 1) / (kReduceThreads / 32);
    if (ctas > 8LL * sms) ctas = 8LL * sms;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)(ctas > 0 ? ctas : 1));
    cfg.blockDim = dim3(kReduceThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (head_dim == 64) return cudaLaunchKernelEx(&cfg, decode_reduce_kernel<64>, p, group);
    if (head_dim == 128) return cudaLaunchKernelEx(&cfg, decode_reduce_kernel<128>, p, group);
    return cudaErrorNotSupported;
}

int device_sm_count() {
    constexpr int kMaxDevices = 64;
    static int cached[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    int n = __atomic_load_n(&cached[dev], __ATOMIC_ACQUIRE);
    if (n == 0 && cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess)
        __atomic_store_n(&cached[dev], n, __ATOMIC_RELEASE);
    return n;
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
    w.next_item = 0;
    w.num_items = 4;
    w.num_multi = 8;
    size_t off = 256;
    w.items = off;
    off = align_up(off + s * mp * sizeof(int2), 256);
    w.multi_seqs = off;
    off = align_up(off + s * sizeof(int2), 256);
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
    cudaError_t e = cudaSuccess;
    if (p.direct_items == 0) {
        // The planning kernel may overlap the previous kernel in the stream (it
        // waits for it before completing).
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(1);
        cfg.blockDim = dim3(kPlanThreads);
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, decode_plan_kernel, p);
        if (e != cudaSuccess) return e;
    }
    switch (dtype) {
        case PA_F32: e = launch_decode_f32(p, head_dim, block_size, group, ub, stream); break;
        case PA_F16:
            e = mma ? launch_decode_mma_f16(p, head_dim, block_size, group, ub, *tmap_k, *tmap_v, stream)
                    : launch_decode_simt_f16(p, head_dim, block_size, group, ub, stream);
            break;
        case PA_BF16:
            e = mma ? launch_decode_mma_bf16(p, head_dim, block_size, group, ub, *tmap_k, *tmap_v, stream)
                    : launch_decode_simt_bf16(p, head_dim, block_size, group, ub, stream);
            break;
        default: return cudaErrorNotSupported;
    }
    if (e != cudaSuccess) return e;
    // With a single partition per sequence every output is already final.
    if (p.max_parts > 1) {
        const int sms = device_sm_count();
        if (sms <= 0) return cudaErrorInvalidDevice;
        e = launch_reduce(p, head_dim, group, sms, stream);
    }
    return e;
}

}  // namespace pa
