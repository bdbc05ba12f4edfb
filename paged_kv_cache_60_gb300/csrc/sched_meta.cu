// Scheduling metadata kernel.
//
// FlashMLA page ("FlashMLA 注意力内核源码走读"), section "调度": a small kernel
// hands (request, KV range) work units to the SMs before the main kernel runs,
// so that every SM gets about the same amount of work and the main kernel only
// reads its assignment. Work is counted in 64-token chunks.
//   fixed mode (splits = S): the split range of FlashAttention's block.h
//     (FlashAttention tiling page, section 5.3): per = ceil(n_b / S),
//     split s = [s*per, min((s+1)*per, n_b)).
//   auto mode (splits = 0): the concatenated chunk sequence of all requests is
//     cut into num_parts intervals of per = ceil(total / num_parts) chunks.
// With a sliding window, a request's chunks start at the one holding the
// first token its first query token sees.
// One CTA of 1024 threads; block-wide scans over tiles of 1024 requests.
#include <cuda_runtime.h>

#include "common.cuh"
#include "decode_attn.h"

namespace da {

// Inclusive block scan of v (blockDim.x == 1024). Returns the inclusive value,
// and the tile total in `total`.
__device__ __forceinline__ int block_incl_scan(int v, int *warp_sums, int &total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        int n = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += n;
    }
    if (lane == 31) warp_sums[warp] = v;
    __syncthreads();
    if (warp == 0) {
        int w = warp_sums[lane];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            int n = __shfl_up_sync(0xffffffffu, w, off);
            if (lane >= off) w += n;
        }
        warp_sums[lane] = w;
    }
    __syncthreads();
    if (warp > 0) v += warp_sums[warp - 1];
    total = warp_sums[31];
    __syncthreads();
    return v;
}

constexpr int kSmemReq = 4096;  // requests whose prefix sums stay in shared memory

__global__ void __launch_bounds__(1024) sched_meta_kernel(const __grid_constant__ SchedParams p) {
    __shared__ int warp_sums[32];
    __shared__ int s_err;
    __shared__ int s_co[kSmemReq + 1];  // chunk_offset
    __shared__ int s_so[kSmemReq + 1];  // split_offset
    pdl_wait();
    pdl_launch_dependents();
    const int tid = threadIdx.x;
    const bool in_smem = p.B <= kSmemReq;
    if (tid == 0) {
        s_err = 0;
        s_co[0] = 0;
        s_so[0] = 0;
    }
    __syncthreads();
    // chunk_offset[b] from shared memory when it fits, else from global memory
    auto co = [&](int b) -> int { return in_smem ? s_co[b] : p.chunk_offset[b]; };

    // pass 1: chunks per request and their prefix sum
    int carry = 0;
    for (int base = 0; base < p.B; base += blockDim.x) {
        const int b = base + tid;
        int n = 0;
        if (b < p.B) {
            int L = p.seqlens[b];
            if (L < 0) {
                atomicOr(&s_err, DA_DEV_NEG_LEN);
                L = 0;
            }
            if (L > p.max_len) {
                atomicOr(&s_err, DA_DEV_SEQ_TOO_LONG);
                L = p.max_len;
            }
            // sparse decode: the request's topk listed positions, whatever its length
            n = chunks_of(L, p.s_q, p.window, p.topk);
        }
        int tile_total;
        const int incl = block_incl_scan(n, warp_sums, tile_total);
        if (b < p.B) {
            p.chunk_offset[b + 1] = carry + incl;
            if (in_smem) s_co[b + 1] = carry + incl;
        }
        carry += tile_total;
    }
    if (tid == 0) p.chunk_offset[0] = 0;
    const int total = carry;
    __syncthreads();
    const int per = p.splits > 0 ? 0 : max(1, (total + p.num_parts - 1) / p.num_parts);

    // pass 2: splits per request and their prefix sum
    carry = 0;
    for (int base = 0; base < p.B; base += blockDim.x) {
        const int b = base + tid;
        int ns = 0;
        if (b < p.B) {
            const int c0 = co(b), cn = co(b + 1);
            if (p.splits > 0)
                ns = p.splits;
            else if (cn > c0)
                ns = (cn - 1) / per - c0 / per + 1;
            p.num_splits[b] = ns;
        }
        int tile_total;
        const int incl = block_incl_scan(ns, warp_sums, tile_total);
        if (b < p.B) {
            p.split_offset[b + 1] = carry + incl;
            if (in_smem) s_so[b + 1] = carry + incl;
        }
        carry += tile_total;
    }
    if (tid == 0) p.split_offset[0] = 0;
    const int total_splits = carry;
    __syncthreads();
    auto so = [&](int b) -> int { return in_smem ? s_so[b] : p.split_offset[b]; };

    // pass 3: one record per part
    for (int q = tid; q < p.num_parts; q += blockDim.x) {
        int b0, s0, c0, c1;
        if (p.splits > 0) {
            b0 = q / p.splits;
            s0 = q % p.splits;
            const int cb = co(b0);
            const int n = co(b0 + 1) - cb;
            const int per_b = (n + p.splits - 1) / p.splits;
            c0 = cb + min(s0 * per_b, n);
            c1 = cb + min((s0 + 1) * per_b, n);
        } else {
            c0 = (int)min((long long)q * per, (long long)total);
            c1 = min(c0 + per, total);
            if (c0 >= total) {
                b0 = -1;
                s0 = 0;
            } else {
                // first i in [0, B] with chunk_offset[i] > c0, minus one
                int lo = 0, hi = p.B;
                while (lo < hi) {
                    const int mid = (lo + hi) >> 1;
                    if (co(mid) > c0)
                        hi = mid;
                    else
                        lo = mid + 1;
                }
                b0 = lo - 1;
                s0 = q - co(b0) / per;
            }
        }
        int4 *rec = reinterpret_cast<int4 *>(p.parts) + 2 * q;
        rec[0] = make_int4(b0, s0, c0, c1);
        if (b0 >= 0) {
            const int L0 = min(max(p.seqlens[b0], 0), p.max_len);
            rec[1] = make_int4(co(b0), L0, so(b0), p.splits > 0 ? p.splits : so(b0 + 1) - so(b0));
        } else {
            rec[1] = make_int4(0, 0, 0, 0);
        }
    }
    __syncthreads();
    if (tid == 0) {
        int32_t *h = p.meta;
        h[kHMagic] = kMetaMagic;
        h[kHB] = p.B;
        h[kHHkv] = p.H_kv;
        h[kHG] = p.G;
        h[kHSplits] = p.splits;
        h[kHNumParts] = p.num_parts;
        h[kHCpc] = p.cpc;
        h[kHChunk] = kChunk;
        h[kHTotalChunks] = total;
        h[kHTotalSplits] = total_splits;
        h[kHPer] = per;
        h[kHError] = s_err;
        h[kHErrorDetail] = 0;
        h[kHKvDtype] = p.kv_dtype;
        h[kHNumSms] = p.num_sms;
        h[kHSq] = p.s_q;
        h[kHWindow] = p.window;
        h[kHTopk] = p.topk;
        for (int k = kHTopk + 1; k < kHeaderWords; ++k) h[k] = 0;
    }
}

cudaError_t launch_sched_meta(const SchedParams &p, cudaStream_t stream, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(1024);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, sched_meta_kernel, p);
}

}  // namespace da
