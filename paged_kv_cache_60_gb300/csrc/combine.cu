// LSE combine of split-KV partials.
//
// Merge rule (XQA page, section "归约怎么记"): with per-split (m_i, l_i, O~_i),
// m = max m_i, l = sum l_i e^(m_i - m), O = (1/l) sum O~_i e^(m_i - m). The
// partials here are stored normalised, as (o_i, lse_i) with lse_i = m_i + ln l_i,
// so the same merge reads lse = M + ln sum_i e^(lse_i - M), M = max lse_i, and
// out = sum_i e^(lse_i - lse) o_i. Splits are summed in index order, so the
// result is bitwise reproducible. The kernel is chained to the split-KV kernel
// with programmatic dependent launch (FlashMLA page, section "合并与性能账本").
//
// One warp per output row (query token, query head); each lane owns DV/32
// consecutive outputs.
#include <cuda_runtime.h>

#include "common.cuh"

namespace da {

constexpr float kLog2e = 1.4426950408889634f;

template <int DV>
__global__ void __launch_bounds__(128) combine_kernel(const __grid_constant__ CombineParams p) {
    const int b = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int hq = blockIdx.y * 4 + warp;
    // The scheduling words come from the metadata kernel, which completed
    // before the split-KV kernel passed its own wait (and so before this grid
    // could start): read them from L2 ahead of the wait, so that their latency
    // overlaps the split-KV kernel's tail. The partials need the wait.
    const int32_t *hd = p.meta.header;
    const int ns = __ldcg(p.meta.num_splits + b);
    const int so = __ldcg(p.meta.split_offset + b);
    const MetaHdr mh = load_meta_header_cg(hd);
    pdl_wait();
    pdl_launch_dependents();  // the next kernel may start its prologue; it waits for this grid before reading
    if (!meta_header_ok(mh, p.B, p.H_kv, p.G, p.splits, p.num_parts, p.s_q, p.window, p.topk))
        return;  // the split-KV kernel has flagged the mismatch
    if (hq >= p.rows) return;
    if (ns == 1) return;  // written directly by the split-KV kernel
    if (ns < 0 || so < 0 || so + ns > p.meta.max_splits) return;
    constexpr int PER_LANE = DV / 32;
    static_assert(DV % 64 == 0, "DV must be a multiple of 64");
    const float *lp = p.meta.lse_part + (size_t)so * p.rows + hq;
    // lane s holds split s's lse (splits beyond 32 are folded in a loop)
    float M = -INFINITY;
    for (int s = lane; s < ns; s += 32) M = fmax_nan(M, lp[(size_t)s * p.rows]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmax_nan(M, __shfl_xor_sync(0xffffffffu, M, off));
    __nv_bfloat16 *op = reinterpret_cast<__nv_bfloat16 *>(p.out) + ((size_t)b * p.rows + hq) * DV;
    float acc[PER_LANE];
#pragma unroll
    for (int k = 0; k < PER_LANE; ++k) acc[k] = 0.f;
    float lse_v = -INFINITY;
    if (M != -INFINITY) {
        float Z = 0.f;
        for (int s = lane; s < ns; s += 32) Z += ex2((lp[(size_t)s * p.rows] - M) * kLog2e);
        // fixed-order tree sum over lanes
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) Z += __shfl_xor_sync(0xffffffffu, Z, off);
        lse_v = M + logf(Z);
        for (int s0 = 0; s0 < ns; s0 += 32) {
            const int cnt = min(32, ns - s0);
            const float w_l = (lane < cnt) ? ex2((lp[(size_t)(s0 + lane) * p.rows] - lse_v) * kLog2e) : 0.f;
            const float *src0 = p.meta.o_part + (((size_t)(so + s0)) * p.rows + hq) * DV;
            const size_t sstride = (size_t)p.rows * DV;
#pragma unroll 4
            for (int s = 0; s < cnt; ++s) {
                const float w = __shfl_sync(0xffffffffu, w_l, s);
                const float *src = src0 + s * sstride;
                if constexpr (PER_LANE == 2) {
                    const float2 v = reinterpret_cast<const float2 *>(src)[lane];
                    acc[0] += w * v.x;
                    acc[1] += w * v.y;
                } else {
#pragma unroll
                    for (int k4 = 0; k4 < PER_LANE / 4; ++k4) {
                        const float4 v = reinterpret_cast<const float4 *>(src)[k4 * 32 + lane];
                        acc[k4 * 4 + 0] += w * v.x;
                        acc[k4 * 4 + 1] += w * v.y;
                        acc[k4 * 4 + 2] += w * v.z;
                        acc[k4 * 4 + 3] += w * v.w;
                    }
                }
            }
        }
    }
    if (p.sinks != nullptr) {
        // the attention sink joins the denominator once, after the splits are
        // merged (XQA page, section "一个容易漏掉的细节:attention sink")
        const float tot = log_add_exp(lse_v, p.sinks[hq % (p.rows / p.s_q)]);
        const float fac = (lse_v == -INFINITY) ? 0.f : expf(lse_v - tot);
#pragma unroll
        for (int k = 0; k < PER_LANE; ++k) acc[k] *= fac;
        lse_v = tot;
    }
    if constexpr (PER_LANE == 2) {
        reinterpret_cast<__nv_bfloat162 *>(op)[lane] = __floats2bfloat162_rn(acc[0], acc[1]);
    } else {
#pragma unroll
        for (int k4 = 0; k4 < PER_LANE / 4; ++k4) {
            uint2 w;
            w.x = pack_bf16(acc[k4 * 4 + 0], acc[k4 * 4 + 1]);
            w.y = pack_bf16(acc[k4 * 4 + 2], acc[k4 * 4 + 3]);
            reinterpret_cast<uint2 *>(op)[k4 * 32 + lane] = w;
        }
    }
    if (lane == 0) p.lse[(size_t)b * p.rows + hq] = lse_v;
}

cudaError_t launch_combine(int DV, const CombineParams &p, cudaStream_t stream, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.B, (p.rows + 3) / 4);
    cfg.blockDim = dim3(128);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    switch (DV) {
        case 64: return cudaLaunchKernelEx(&cfg, combine_kernel<64>, p);
        case 128: return cudaLaunchKernelEx(&cfg, combine_kernel<128>, p);
        case 512: return cudaLaunchKernelEx(&cfg, combine_kernel<512>, p);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace da
