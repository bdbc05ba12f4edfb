// KV append: writes each request's new token into the page slot that its
// block table gives for its position, quantising on the way.
//
// The decode kernels read a pool that already holds the step's new K/V; the
// write itself happens upstream of attention (XQA page, section
// "一次 decode step 的完整时序": the KV append is not part of XQA, the new
// token lands in the pool first and the attention kernel only reads through
// the page table). The formats are those the decode kernels read:
//   * bf16 pools: a copy of the token's H_kv * D values;
//   * e4m3 pools: code = e4m3(x / scale[h]) with one fp32 scale per KV head and
//     tensor (XQA page, section "Hopper 路径上 V 不做显式反量化", largest finite 448);
//   * the 656-byte latent token (FlashMLA page, section "数据加载"): per block
//     of 128 NoPE values, scale = max|x| / 448 (1 for an all-zero block),
//     512 codes, the four fp32 scales, then the 64 RoPE values as bf16.
// Rounding is the IEEE one everywhere: the quotient x / scale is the fp32
// division rounded to nearest (not a plain multiply by a reciprocal), the e4m3
// code the nearest finite value with ties to even, saturating at +-448; NaN
// maps to 0x7F. The quotient is computed by Markstein's correction of the
// reciprocal product where that gives the rounded quotient exactly, and by the
// division elsewhere (see quot_rn). The pool layout is [num_pages][page_size][H_kv][D] (bf16 / e4m3)
// or [num_pages][page_size][1][656].
//
// The work is a scatter of a few hundred bytes per request, HBM / latency
// bound: per thread the same 16-byte vector of K and of V (two loads, two
// 16- or 8-byte stores), coalesced along the token's contiguous H_kv * D
// values; the latent format takes one warp per token (lanes 8k..8k+7 own
// block k and reduce its max with shuffles). Every request's new row is read,
// even when its position skips it.
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "decode_attn.h"
#include "layout.h"

namespace da {
namespace {

constexpr int kThreads = 256;
constexpr int kLatentRow = 656;
constexpr int kLatentNope = 512;
constexpr int kLatentScales = 512;   // byte offset of the 4 fp32 scales
constexpr int kLatentRope = 528;     // byte offset of the 64 bf16 RoPE values
constexpr float kE4m3Max = 448.f;

__device__ __forceinline__ uint4 ld_stream_v4(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void st_v4(void *p, uint4 v) {
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ void st_v2(void *p, uint2 v) {
    asm volatile("st.global.v2.u32 [%0], {%1, %2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two fp32 values -> two e4m3 codes (lo in bits 0..7, hi in bits 8..15):
// round to nearest even, finite results saturate at +-448, NaN -> 0x7F (one
// test per pair on the common path: the sum of two values is NaN when either
// is).
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    uint32_t c = r;
    const float t = lo + hi;
    if (t != t) {
        if (lo != lo) c = (c & 0xFF00u) | 0x7Fu;
        if (hi != hi) c = (c & 0x00FFu) | 0x7F00u;
    }
    return c;
}

// The reciprocal of a scale and whether Markstein's correction applies to it:
// y = RN(1 / s) (correctly rounded), for scales in [2^-80, 2^100]: the
// reciprocal stays normal, and an input small enough for the residual below to
// underflow (|x| < 2^-100) gives |x / s| < 2^-20, which codes to a signed zero
// whatever its last bit.
struct Recip {
    float s, y;
    bool ok;
};
__device__ __forceinline__ Recip recip_of(float s) {
    const float a = fabsf(s);
    return Recip{s, __frcp_rn(s), a >= 0x1p-80f && a <= 0x1p100f};
}

// RN(x / s), the quotient rounded to nearest, by Markstein's correction
// (P. Markstein, "Computation of elementary functions on the IBM RISC
// System/6000 processor", IBM J. Res. Develop. 34 (1990)): with y = RN(1/s),
// q0 = RN(x y) is within an ulp of x / s, the residual r = x - q0 s is exact
// in one fused multiply-add, and RN(q0 + r y) is the rounded quotient, as long
// as nothing overflows or underflows on the way. That equality was checked
// exhaustively over every finite bf16 x with |x| >= 2^-100 and |x / s| in
// [2^-12, 2^10] for 5090 scales (powers of two and their neighbours,
// log-uniform 1e-4 .. 1e2, amax / 448): the range in which the e4m3 code
// depends on the quotient's value. Below it the code is a signed zero (the
// sign is taken from q0, so -0 stays -0), above it the code saturates, and a
// NaN input gives a NaN quotient, so those need no test. What does: a scale
// outside the range recip_of accepts, an infinite input, and a quotient large
// enough to overflow the residual (|x| y >= 2^100): one running max of |x| per
// group of values tells, and the IEEE division runs only where some active
// lane of the warp has such a value (the vote is over the lanes that reach it:
// requests that are skipped leave the loop first).
// Pairs of values go through the packed fp32 pipe (mul.rn / fma.rn on .f32x2:
// each lane rounds exactly as the scalar instruction does).
__device__ __forceinline__ uint64_t f2pack(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void f2unpack(uint64_t r, float &a, float &b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
template <int N>
__device__ __forceinline__ void quot_rn(const float (&x)[N], const Recip &d, float (&q)[N]) {
    static_assert(N % 2 == 0, "pairs of values");
    float mx = 0.f;
    const uint64_t y2 = f2pack(d.y, d.y), ns2 = f2pack(-d.s, -d.s);
#pragma unroll
    for (int i = 0; i < N; i += 2) {
        const uint64_t x2 = f2pack(x[i], x[i + 1]);
        uint64_t q02, r2, qq2;
        asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(q02) : "l"(x2), "l"(y2));
        asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r2) : "l"(q02), "l"(ns2), "l"(x2));
        asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(qq2) : "l"(r2), "l"(y2), "l"(q02));
        float q0a, q0b, qa, qb;
        f2unpack(q02, q0a, q0b);
        f2unpack(qq2, qa, qb);
        q[i] = copysignf(qa, q0a);
        q[i + 1] = copysignf(qb, q0b);
        mx = fmaxf(mx, fmaxf(fabsf(x[i]), fabsf(x[i + 1])));
    }
    const bool fast = d.ok && mx < INFINITY && mx * fabsf(d.y) < 0x1p100f;
    if (!__all_sync(__activemask(), fast)) {
        if (!fast) {
#pragma unroll
            for (int i = 0; i < N; ++i) q[i] = __fdiv_rn(x[i], d.s);
        }
    }
}

// RN(a / 448), the block scale of the 656-byte token, by the same correction
// with the constant y = RN(1/448); checked exhaustively against the IEEE
// division for every bf16 magnitude >= 2^-100 (the block maxima are bf16
// values). Smaller, infinite or NaN maxima take the division.
__device__ __forceinline__ float div448(float a) {
    constexpr float y = 0x1.24924ap-9f;  // RN(1 / 448)
    if (!(a >= 0x1p-100f && a < INFINITY)) return __fdiv_rn(a, kE4m3Max);
    const float q0 = a * y;
    const float r = fmaf(-q0, kE4m3Max, a);
    return fmaf(r, y, q0);
}

// Eight bf16 values (one 16-byte vector) / s -> eight e4m3 codes.
__device__ __forceinline__ uint2 quant8(uint4 x, const Recip &d) {
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
    float v[8], q[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] = bf16_lo(w[i]);
        v[2 * i + 1] = bf16_hi(w[i]);
    }
    quot_rn(v, d, q);
    uint32_t c[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) c[i] = e4m3x2(q[2 * i], q[2 * i + 1]);
    return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
}

// Shared prologue of both kernels: where request b's token goes, or -1 when
// it is skipped (negative position) or invalid (error bit set by `reporter`).
__device__ __forceinline__ int64_t slot_of(const AppendParams &p, int b, bool reporter) {
    const int t = __ldg(p.positions + b);
    if (t < 0) return -1;
    if ((int64_t)t >= (int64_t)p.max_pages * p.page_size) {
        if (reporter && p.error) atomicOr(p.error, DA_DEV_SEQ_TOO_LONG);
        return -1;
    }
    const int page = __ldg(p.block_table + (int64_t)b * p.max_pages + t / p.page_size);
    if (page < 0 || page >= p.num_pages) {
        if (reporter && p.error) atomicOr(p.error, DA_DEV_BAD_PAGE);
        return -1;
    }
    return (int64_t)page * p.page_size + t % p.page_size;
}

// bf16 / e4m3 pools. Work item = kV values (one or two 16-byte vectors of 8)
// at the same place in K and in V of one request (items of a request are
// consecutive). The row loads are issued before the position and page
// lookups, so their latencies overlap. The e4m3 build takes 16 values per item
// (D a multiple of 16): each thread then moves as many bytes per lookup chain
// as a bf16 thread, and stores its 16 codes as one 16-byte vector.
// Six blocks per SM (at most 40 registers a thread): the latency of a work
// item's chain (row loads, position and page lookups, quotients, stores)
// is hidden by more resident threads; measured faster than the four blocks
// that 52 registers allow, despite a few spilled words.
template <bool kFp8, int kV>
__global__ void __launch_bounds__(kThreads, 6) append_gqa_kernel(const AppendParams p) {
    pdl_wait();               // positions, block table and new rows may come from the previous kernel
    pdl_launch_dependents();  // the next kernel waits for this grid before it reads the pool
    constexpr int NV = kV / 8;  // 16-byte input vectors per item
    const int vpr = p.D / kV;
    const int per_req = p.H_kv * vpr;
    const int64_t total = (int64_t)p.B * per_req;
    for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x; i < total; i += (int64_t)gridDim.x * kThreads) {
        const int b = (int)(i / per_req);
        const int e = (int)(i - (int64_t)b * per_req);
        const int64_t src = (int64_t)b * p.row_stride + (int64_t)e * kV;
        uint4 xk[NV], xv[NV];
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            xk[j] = ld_stream_v4(p.k_new + src + 8 * j);
            xv[j] = ld_stream_v4(p.v_new + src + 8 * j);
        }
        const int64_t slot = slot_of(p, b, e == 0);
        if (slot < 0) continue;
        const int64_t vec = slot * per_req + e;
        if constexpr (!kFp8) {
#pragma unroll
            for (int j = 0; j < NV; ++j) {
                st_v4(p.k_pool + vec * kV * 2 + 16 * j, xk[j]);
                st_v4(p.v_pool + vec * kV * 2 + 16 * j, xv[j]);
            }
        } else {
            const int h = e / vpr;
            const Recip dk = recip_of(__ldg(p.k_scale + h)), dv = recip_of(__ldg(p.v_scale + h));
            if constexpr (NV == 2) {
                const uint2 k0 = quant8(xk[0], dk), k1 = quant8(xk[1], dk);
                const uint2 v0 = quant8(xv[0], dv), v1 = quant8(xv[1], dv);
                st_v4(p.k_pool + vec * kV, make_uint4(k0.x, k0.y, k1.x, k1.y));
                st_v4(p.v_pool + vec * kV, make_uint4(v0.x, v0.y, v1.x, v1.y));
            } else {
                st_v2(p.k_pool + vec * kV, quant8(xk[0], dk));
                st_v2(p.v_pool + vec * kV, quant8(xv[0], dv));
            }
        }
    }
}

// 656-byte latent tokens, one warp per request. Lane l holds NoPE values
// [16l, 16l+16); lanes 8k..8k+7 form block k.
struct LatentIn {
    uint4 a0, a1, rope;
};
__device__ __forceinline__ LatentIn latent_load(const AppendParams &p, int b, int lane) {
    const uint16_t *src = p.k_new + (int64_t)b * p.row_stride;
    LatentIn x;
    x.a0 = ld_stream_v4(src + lane * 16);
    x.a1 = ld_stream_v4(src + lane * 16 + 8);
    x.rope = lane < 8 ? ld_stream_v4(src + kLatentNope + lane * 8) : make_uint4(0u, 0u, 0u, 0u);
    return x;
}
// every lane of the warp calls this for the same request
__device__ __forceinline__ void latent_store(const AppendParams &p, int b, int lane, const LatentIn &x) {
    const int64_t slot = slot_of(p, b, lane == 0);  // uniform over the warp
    if (slot < 0) return;
    const uint32_t w[8] = {x.a0.x, x.a0.y, x.a0.z, x.a0.w, x.a1.x, x.a1.y, x.a1.z, x.a1.w};
    // max |x| by the magnitude bits: exact, and a NaN wins (scale 1 then)
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        m = max(m, (w[i] << 16) & 0x7FFFFFFFu);
        m = max(m, w[i] & 0x7FFF0000u);
    }
    m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
    m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
    m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 4));
    const float amax = __uint_as_float(m);
    const float scale = amax > 0.f ? div448(amax) : 1.f;
    const Recip d = recip_of(scale);
    float v[16], q[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        v[2 * i] = bf16_lo(w[i]);
        v[2 * i + 1] = bf16_hi(w[i]);
    }
    quot_rn(v, d, q);
    uint32_t c[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) c[i] = e4m3x2(q[4 * i], q[4 * i + 1]) | (e4m3x2(q[4 * i + 2], q[4 * i + 3]) << 16);
    uint8_t *row = p.k_pool + slot * kLatentRow;
    st_v4(row + lane * 16, make_uint4(c[0], c[1], c[2], c[3]));
    const float s1 = __shfl_sync(0xFFFFFFFFu, scale, 8);
    const float s2 = __shfl_sync(0xFFFFFFFFu, scale, 16);
    const float s3 = __shfl_sync(0xFFFFFFFFu, scale, 24);
    if (lane == 0)
        st_v4(row + kLatentScales,
              make_uint4(__float_as_uint(scale), __float_as_uint(s1), __float_as_uint(s2), __float_as_uint(s3)));
    if (lane < 8) st_v4(row + kLatentRope + lane * 16, x.rope);
}

__global__ void __launch_bounds__(kThreads, 6) append_mla_kernel(const AppendParams p) {
    pdl_wait();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    constexpr int kWarps = kThreads / 32;
    for (int b = blockIdx.x * kWarps + (threadIdx.x >> 5); b < p.B; b += gridDim.x * kWarps) {
        // the row loads first, then the position and page lookups
        latent_store(p, b, lane, latent_load(p, b, lane));
    }
}

}  // namespace

cudaError_t launch_append(int kv_dtype, const AppendParams &p, cudaStream_t stream, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    constexpr int64_t kMaxBlocks = 1 << 20;    // grid-stride beyond that
    if (kv_dtype == DA_KV_FP8_MLA656) {
        const int64_t blocks = (p.B + kThreads / 32 - 1) / (kThreads / 32);
        cfg.gridDim = dim3((unsigned)(blocks < kMaxBlocks ? blocks : kMaxBlocks));
        return cudaLaunchKernelEx(&cfg, append_mla_kernel, p);
    }
    const bool wide = kv_dtype == DA_KV_FP8_PER_TENSOR && p.D % 16 == 0;
    const int64_t items = (int64_t)p.B * p.H_kv * (p.D / (wide ? 16 : 8));
    const int64_t blocks = (items + kThreads - 1) / kThreads;
    cfg.gridDim = dim3((unsigned)(blocks < kMaxBlocks ? blocks : kMaxBlocks));
    if (kv_dtype == DA_KV_FP8_PER_TENSOR)
        return wide ? cudaLaunchKernelEx(&cfg, append_gqa_kernel<true, 16>, p)
                    : cudaLaunchKernelEx(&cfg, append_gqa_kernel<true, 8>, p);
    return cudaLaunchKernelEx(&cfg, append_gqa_kernel<false, 8>, p);
}

}  // namespace da
