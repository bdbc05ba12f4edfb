// Split-KV decode kernel for the 656-byte FP8 latent token (MQA: 128 query
// heads share one KV head; D_qk = 576, D_v = 512), on the 5th-generation
// tensor cores (tcgen05, accumulators in tensor memory).
//
// The token format is the FlashMLA page's ("FlashMLA 注意力内核源码走读", section
// "数据加载"): 512 e4m3 values with one fp32 scale per 128 of them, then 64
// bf16 RoPE values; K is the 576 dequantised values and V their first 512.
// Dequantisation goes to bf16 and the products run in bf16 with fp32
// accumulation, as that section describes.
//
// Work split: two CTAs per part, each owning 64 of the 128 query heads. The
// output of 128 heads x 512 values in fp32 would fill a whole SM's tensor
// memory, so it is split by head across the pair; each CTA dequantises the
// part's tokens itself (the KV bytes are read from HBM once and from L2 twice).
//
// Per 64-token chunk:
//   S  = Q K^T   M = 64 heads, N = 64 tokens, K = 576   (S in TMEM, double buffered)
//   softmax      one thread per head: running max m, sum l, exp2, P -> shared memory (bf16)
//   O^T += V^T P^T  M = 128 (four blocks of V's 512 columns), N = 64 heads, K = 64 tokens
// V^T is read straight from the dequantised K tile through an MN-major
// descriptor, so the tile is written once. The running max is re-based only
// when it grows by more than 2^8 (then O^T columns are rescaled in TMEM);
// otherwise P values stay below 256 and the sums are exact to fp32 rounding.
// (Online softmax: attention pipeline page, section 三; exp via exp2: section 一.)
//
// Roles (416 threads): warp 0 issues MMAs (one lane) and owns the TMEM
// allocation; warps 1-4 run the softmax and the epilogue (TMEM lane quadrant
// = warp % 4); warps 5-12 dequantise tokens and load Q.
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "decode_attn.h"
#include "segwalk.cuh"

namespace da {

namespace mla {
constexpr int HEADS = 64;                  // query heads per CTA
constexpr int DQK = 576, DV = 512;
constexpr int NSL = DQK / 64;              // 64-column slices of a row (9)
constexpr int SLICE = kChunk * 128;        // one slice of a 64-row tile (8 KB)
constexpr int TILE = NSL * SLICE;          // 64 rows x 576 bf16 (72 KB)
constexpr int ROW_BYTES = 656;
constexpr int OFF_Q = 0;
constexpr int OFF_K0 = TILE;
constexpr int OFF_K1 = 2 * TILE;
constexpr int OFF_P = 3 * TILE;
constexpr int OFF_MISC = OFF_P + HEADS * 128;
// misc: 14 mbarriers, tmem base, abort flag, per-head alpha / l / m
constexpr int OFF_BARS = OFF_MISC;
constexpr int OFF_TMEM = OFF_BARS + 14 * 8;
constexpr int OFF_ABORT = OFF_TMEM + 4;
constexpr int OFF_ALPHA = OFF_ABORT + 12;
constexpr int OFF_L = OFF_ALPHA + HEADS * 4;
constexpr int OFF_M = OFF_L + HEADS * 4;
constexpr int SMEM = OFF_M + HEADS * 4 + 1024;  // + alignment slack
constexpr int THREADS = 13 * 32;
constexpr int SM_WARPS = 4, DQ_WARPS = 8;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t S_COL = 0;              // two S buffers: columns 0 and 64
constexpr uint32_t O_COL = 128;            // O^T blocks j = 0..3 at 128 + 64 j
constexpr float RESCALE_LOG2 = 8.f;        // re-base the max when it grows by more than 2^8
static_assert(SMEM <= 232448, "shared memory budget");
}  // namespace mla

constexpr float kLn2Mla = 0.6931471805599453f;

__device__ __forceinline__ uint32_t swz(int row, int c16) { return (uint32_t)(row * 128 + ((c16 ^ (row & 7)) << 4)); }

// 16 e4m3 values times `scale`, as 16 bf16 (two 16-byte words).
__device__ __forceinline__ void dequant16(const uint4 v, float scale, uint4 &lo, uint4 &hi) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t h01 = e4m3x2_to_f16x2((uint16_t)(w[k] & 0xffff));
        const uint32_t h23 = e4m3x2_to_f16x2((uint16_t)(w[k] >> 16));
        const float2 f01 = __half22float2(*reinterpret_cast<const __half2 *>(&h01));
        const float2 f23 = __half22float2(*reinterpret_cast<const __half2 *>(&h23));
        o[2 * k] = pack_bf16(f01.x * scale, f01.y * scale);
        o[2 * k + 1] = pack_bf16(f23.x * scale, f23.y * scale);
    }
    lo = make_uint4(o[0], o[1], o[2], o[3]);
    hi = make_uint4(o[4], o[5], o[6], o[7]);
}

__global__ void __launch_bounds__(mla::THREADS, 1) mla_decode_kernel(const __grid_constant__ MlaParams p) {
    using namespace mla;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + OFF_BARS);
    uint64_t *kfull = bars + 0, *kempty = bars + 2, *sfull = bars + 4, *sfree = bars + 6;
    uint64_t *pfull = bars + 8, *pfree = bars + 9, *ofull = bars + 10, *ofree = bars + 11;
    uint64_t *qfull = bars + 12, *qfree = bars + 13;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + OFF_TMEM);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + OFF_ABORT);
    float *alpha_sm = reinterpret_cast<float *>(smem + OFF_ALPHA);
    float *l_sm = reinterpret_cast<float *>(smem + OFF_L);
    float *m_sm = reinterpret_cast<float *>(smem + OFF_M);
    const uint32_t q_addr = smem_u32(smem + OFF_Q);
    const uint32_t k_addr[2] = {smem_u32(smem + OFF_K0), smem_u32(smem + OFF_K1)};
    const uint32_t p_addr = smem_u32(smem + OFF_P);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int part = blockIdx.x, hh = blockIdx.y;  // head half: heads [64 hh, 64 hh + 64)

    if (threadIdx.x == 0) {
        mbar_init(&kfull[0], DQ_WARPS);
        mbar_init(&kfull[1], DQ_WARPS);
        mbar_init(&kempty[0], 1);
        mbar_init(&kempty[1], 1);
        mbar_init(&sfull[0], 1);
        mbar_init(&sfull[1], 1);
        mbar_init(&sfree[0], SM_WARPS);
        mbar_init(&sfree[1], SM_WARPS);
        mbar_init(pfull, SM_WARPS);
        mbar_init(pfree, 1);
        mbar_init(ofull, 1);
        mbar_init(ofree, SM_WARPS);
        mbar_init(qfull, DQ_WARPS);
        mbar_init(qfree, 1);
        *abort_flag = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    if (warp == 0) tmem_alloc(tmem_slot, TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();
    pdl_launch_dependents();

    const int4 rec0 = p.meta.parts[2 * part];
    const int4 rec1 = p.meta.parts[2 * part + 1];
    const int32_t *hd = p.meta.header;
    const bool meta_ok = hd[kHMagic] == kMetaMagic && hd[kHB] == p.B && hd[kHHkv] == 1 && hd[kHG] == p.H_q &&
                         hd[kHSplits] == p.splits && hd[kHNumParts] == p.num_parts && (int)gridDim.x == p.num_parts;
    const int max_len = p.max_pages * p.page_size;

    if (!meta_ok) {
        if (threadIdx.x == 0) atomicOr(&p.meta.header[kHError], DA_DEV_META_MISMATCH);
    } else if (warp == 0) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            // Two cursors walk the same chunk sequence: one issues S = Q K^T,
            // the other O^T += V^T P^T. Whichever is ready goes first (the
            // product for P first, since the next chunk's tile waits on it);
            // the barriers keep S at most two chunks ahead.
            constexpr uint32_t IDESC_QK = umma_idesc_bf16(64, 64, 0, 0);
            constexpr uint32_t IDESC_PV = umma_idesc_bf16(128, 64, 1, 0);
            SegWalker wq = make_walker(p.meta, rec0, rec1, p.B, p.seqlens, max_len);
            SegWalker wp = wq;
            auto next_seg = [](SegWalker &w, int &n) -> bool {
                Seg g;
                while (w.next(g)) {
                    n = g.lc1 - g.lc0;
                    if (n > 0) return true;
                }
                return false;
            };
            int nq = 0, np = 0;
            bool q_more = next_seg(wq, nq), p_more = next_seg(wp, np);
            int qc = 0, pc = 0, qcur = 0, pcur = 0, qseg = 0, pseg = 0;
            bool ok = true;
            uint64_t t_idle = 0;
            uint32_t spins = 0;
            while (q_more || p_more) {
                bool issued = false;
                if (p_more && pcur < qcur && mbar_test(pfull, pcur & 1) &&
                    (pc != 0 || pseg == 0 || mbar_test(ofree, (pseg - 1) & 1))) {
                    const int kb = pcur & 1;
                    tc_fence_after();
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
#pragma unroll
                        for (int kt = 0; kt < kChunk / 16; ++kt) {
                            const uint64_t a = umma_desc(k_addr[kb] + 2 * j * SLICE + kt * 2048, SLICE, 1024);
                            const uint64_t b = umma_desc(p_addr + kt * 32, 16, 1024);
                            umma_bf16(tmem + O_COL + 64 * j, a, b, IDESC_PV, !(pc == 0 && kt == 0));
                        }
                    }
                    umma_commit(&kempty[kb]);
                    umma_commit(pfree);
                    if (pc == np - 1) umma_commit(ofull);
                    ++pcur;
                    if (++pc == np) {
                        pc = 0;
                        ++pseg;
                        p_more = next_seg(wp, np);
                    }
                    issued = true;
                } else if (q_more && (qc != 0 || mbar_test(qfull, qseg & 1)) &&
                           mbar_test(&kfull[qcur & 1], (qcur >> 1) & 1) &&
                           mbar_test(&sfree[qcur & 1], ((qcur >> 1) & 1) ^ 1)) {
                    const int kb = qcur & 1;
                    tc_fence_after();
#pragma unroll 4
                    for (int ks = 0; ks < DQK / 16; ++ks) {
                        const uint32_t off = (ks >> 2) * SLICE + (ks & 3) * 32;
                        umma_bf16(tmem + S_COL + 64 * kb, umma_desc(q_addr + off, 16, 1024),
                                  umma_desc(k_addr[kb] + off, 16, 1024), IDESC_QK, ks > 0);
                    }
                    umma_commit(&sfull[kb]);
                    if (qc == nq - 1) umma_commit(qfree);  // Q may be replaced once these complete
                    ++qcur;
                    if (++qc == nq) {
                        qc = 0;
                        ++qseg;
                        q_more = next_seg(wq, nq);
                    }
                    issued = true;
                }
                if (issued) {
                    spins = 0;
                } else if ((++spins & 63) == 0) {
                    const uint64_t now = global_ns();
                    if (spins == 64) t_idle = now;
                    if (*abort_flag || now - t_idle > p.wait_limit_ns) {
                        ok = false;
                        break;
                    }
                }
            }
            if (!ok) {
                atomicOr(&p.meta.header[kHError], DA_DEV_TIMEOUT);
                *abort_flag = 1;
            }
            // every product issued here has completed before the TMEM goes away
            umma_commit(qfree);
            mbar_wait_timed(qfree, (qseg & 1), 100000000ull);
        }
    } else if (warp >= 5) {
        // ------------------------------------------------------------ dequantise K/V tokens, load Q
        // Warp dw owns tokens 8 dw .. 8 dw + 7 of every chunk. Per token, lane l
        // reads NoPE bytes 16 l .. 16 l + 15 (one 512-byte coalesced load per
        // warp), lanes 0-7 the RoPE part and lanes 0-3 the four scales; all
        // loads of a chunk are in flight while the warp waits for its buffer.
        const int dt = threadIdx.x - 5 * 32;  // 0 .. 255
        const int dw = warp - 5;
        SegWalker wk = make_walker(p.meta, rec0, rec1, p.B, p.seqlens, max_len);
        Seg sg;
        int ic = 0, seg = 0;
        bool ok = true;
        while (ok && wk.next(sg)) {
            const int n = sg.lc1 - sg.lc0;
            if (n == 0) continue;
            // Q rows of this CTA's 64 heads, as the A operand (K-major, 128-byte swizzle)
            if (!(ok = mbar_wait_warp(qfree, (seg & 1) ^ 1, abort_flag, p.wait_limit_ns))) break;
            {
                const uint4 *qsrc = reinterpret_cast<const uint4 *>(reinterpret_cast<const __nv_bfloat16 *>(p.q) +
                                                                    ((size_t)sg.b * p.H_q + hh * HEADS) * DQK);
                for (int e = dt; e < HEADS * (DQK / 8); e += DQ_WARPS * 32) {
                    const int h = e / (DQK / 8), c = e % (DQK / 8);
                    *reinterpret_cast<uint4 *>(smem + OFF_Q + (c >> 3) * SLICE + swz(h, c & 7)) = qsrc[e];
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(qfull);
            const int32_t *bt_row = p.block_table + (size_t)sg.b * p.max_pages;
            for (int c = 0; c < n && ok; ++c) {
                const int cur = ic + c, kb = cur & 1;
                const int t0 = (sg.lc0 + c) * kChunk + 8 * dw;  // first of this warp's 8 tokens
                // the 8 tokens lie in one page (page sizes are multiples of 8)
                const uint8_t *rows = nullptr;
                if (t0 < sg.L) {
                    const int pg = bt_row[t0 / p.page_size];
                    if (pg < 0 || pg >= p.num_pages) {
                        if (lane == 0) {
                            atomicOr(&p.meta.header[kHError], DA_DEV_BAD_PAGE);
                            p.meta.header[kHErrorDetail] = pg;
                        }
                    } else {
                        rows = p.pool + ((size_t)pg * p.page_size + t0 % p.page_size) * ROW_BYTES;
                    }
                }
                const int nv = rows ? min(8, sg.L - t0) : 0;  // valid tokens of the 8
                uint4 nope[8], rope[8];
                float sc[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    nope[i] = make_uint4(0u, 0u, 0u, 0u);
                    rope[i] = nope[i];
                    sc[i] = 0.f;
                    if (i < nv) {
                        const uint8_t *r = rows + i * ROW_BYTES;
                        nope[i] = ldg_stream16(r + 16 * lane);
                        if (lane < 8) rope[i] = ldg_stream16(r + 528 + 16 * lane);
                        if (lane < 4) sc[i] = ldg_stream4f(r + 512 + 4 * lane);
                    }
                }
                if (!(ok = mbar_wait_warp(&kempty[kb], ((cur >> 1) & 1) ^ 1, abort_flag, p.wait_limit_ns))) break;
                uint8_t *kt = smem + (kb ? OFF_K1 : OFF_K0);
                // lane l's 16 values go to slice l / 4, 16-byte chunks 2 (l % 4) and 2 (l % 4) + 1;
                // half the lanes store their upper chunk first so each store touches all banks
                const int sl = lane >> 2, cA = 2 * (lane & 3) + ((lane >> 2) & 1), cB = cA ^ 1;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int tok = 8 * dw + i;
                    const float scale = __shfl_sync(0xffffffffu, sc[i], lane >> 3);
                    uint4 lo, hi;
                    dequant16(nope[i], scale, lo, hi);
                    const bool swap = (lane >> 2) & 1;
                    *reinterpret_cast<uint4 *>(kt + sl * SLICE + swz(tok, cA)) = swap ? hi : lo;
                    *reinterpret_cast<uint4 *>(kt + sl * SLICE + swz(tok, cB)) = swap ? lo : hi;
                    if (lane < 8) *reinterpret_cast<uint4 *>(kt + 8 * SLICE + swz(tok, lane)) = rope[i];
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&kfull[kb]);
            }
            ic += n;
            ++seg;
        }
        if (!ok && lane == 0) {
            atomicOr(&p.meta.header[kHError], DA_DEV_TIMEOUT);
            *abort_flag = 1;
        }
    } else {
        // ------------------------------------------------------------ softmax and epilogue (warps 1-4)
        const int quad = warp & 3;                 // TMEM lanes [32 quad, 32 quad + 32)
        const int head = quad * 16 + lane;         // owned head (lanes 0-15)
        const bool owner = lane < 16;
        const int sid = threadIdx.x - 32;          // 0 .. 127
        const float sl2 = p.scale_log2;
        SegWalker wk = make_walker(p.meta, rec0, rec1, p.B, p.seqlens, max_len);
        Seg sg;
        int ic = 0, seg = 0;
        bool ok = true;
        while (wk.next(sg)) {
            const int n = sg.lc1 - sg.lc0;
            const bool direct = sg.ns == 1;
            const int split = sg.so + sg.s;
            const bool split_ok = direct || (split >= 0 && split < p.meta.max_splits);
            if (n == 0) {
                // no tokens: output 0, lse -inf
                for (int e = sid; e < HEADS * DV; e += 128) {
                    const size_t hq = (size_t)hh * HEADS + e / DV;
                    if (direct)
                        reinterpret_cast<__nv_bfloat16 *>(p.out)[((size_t)sg.b * p.H_q + hq) * DV + e % DV] =
                            __float2bfloat16_rn(0.f);
                    else if (split_ok)
                        p.meta.o_part[((size_t)split * p.H_q + hq) * DV + e % DV] = 0.f;
                }
                if (sid < HEADS) {
                    const size_t hq = (size_t)hh * HEADS + sid;
                    if (direct)
                        p.lse[(size_t)sg.b * p.H_q + hq] = -INFINITY;
                    else if (split_ok)
                        p.meta.lse_part[(size_t)split * p.H_q + hq] = -INFINITY;
                }
                continue;
            }
            float m_used = -INFINITY, l = 0.f;
            for (int c = 0; c < n; ++c) {
                const int cur = ic + c, sb = cur & 1;
                bool w_ok = mbar_wait_warp(&sfull[sb], (cur >> 1) & 1, abort_flag, p.wait_limit_ns);
                tc_fence_after();
                float s[64];
                {
                    uint32_t r[64];
                    tmem_ld64_sync(tmem + ((uint32_t)(32 * quad) << 16) + S_COL + 64 * sb, r);
#pragma unroll
                    for (int e = 0; e < 64; ++e) s[e] = __uint_as_float(r[e]);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sfree[sb]);
                const int nvalid = sg.L - (sg.lc0 + c) * kChunk;
                float mx = -INFINITY;
#pragma unroll
                for (int e = 0; e < 64; ++e) {
                    s[e] = (e < nvalid) ? s[e] * sl2 : -INFINITY;
                    mx = fmaxf(mx, s[e]);
                }
                // P's buffer and O^T are free once the previous chunk's PV has completed
                if (cur > 0) w_ok = w_ok && mbar_wait_warp(pfree, (cur - 1) & 1, abort_flag, p.wait_limit_ns);
                const float m_new = fmaxf(m_used, mx);
                const bool need = owner && c > 0 && (m_new > m_used + RESCALE_LOG2);
                if (c == 0) m_used = m_new;
                // both decisions are taken by all four warps together
                if (named_barrier_or(1, 128, !w_ok || *abort_flag != 0)) {
                    if (lane == 0) {
                        atomicOr(&p.meta.header[kHError], DA_DEV_TIMEOUT);
                        *abort_flag = 1;
                    }
                    ok = false;
                    break;
                }
                if (named_barrier_or(1, 128, need)) {
                    {
                        const float alpha = need ? ex2(m_used - m_new) : 1.f;
                        if (need) {
                            m_used = m_new;
                            l *= alpha;
                        }
                        if (owner) alpha_sm[head] = alpha;
                        named_barrier_sync(1, 128);
                        // rescale every O^T row this thread holds (row = d_v, column = head)
#pragma unroll 1
                        for (int j = 0; j < 4; ++j) {
#pragma unroll 1
                            for (int k = 0; k < 4; ++k) {
                                uint32_t r[16];
                                const uint32_t ta = tmem + ((uint32_t)(32 * quad) << 16) + O_COL + 64 * j + 16 * k;
                                tmem_ld16_sync(ta, r);
#pragma unroll
                                for (int e = 0; e < 16; ++e)
                                    r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha_sm[16 * k + e]);
                                tmem_st16(ta, r);
                            }
                        }
                        tmem_wait_st();
                        tc_fence_before();
                        named_barrier_sync(1, 128);
                    }
                }
                // P row of this head: 64 tokens, bf16, K-major B operand with 128-byte swizzle
                float ps = 0.f;
                uint32_t pk[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const float p0 = ex2(s[2 * e] - m_used), p1 = ex2(s[2 * e + 1] - m_used);
                    ps += p0 + p1;
                    pk[e] = pack_bf16(p0, p1);
                }
                l += ps;
                if (owner) {
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        *reinterpret_cast<uint4 *>(smem + OFF_P + swz(head, k)) =
                            make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(pfull);
            }
            if (!ok) break;
            // ---- epilogue: O = O^T / l
            const bool o_ok = !named_barrier_or(1, 128, !mbar_wait_warp(ofull, seg & 1, abort_flag, p.wait_limit_ns));
            tc_fence_after();
            if (owner) {
                l_sm[head] = l;
                m_sm[head] = m_used;
            }
            named_barrier_sync(1, 128);
            if (o_ok) {
#pragma unroll 1
                for (int j = 0; j < 4; ++j) {
                    const int d = 128 * j + 32 * quad + lane;
#pragma unroll 1
                    for (int k = 0; k < 4; ++k) {
                        uint32_t r[16];
                        tmem_ld16_sync(tmem + ((uint32_t)(32 * quad) << 16) + O_COL + 64 * j + 16 * k, r);
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const int h = 16 * k + e;
                            const float lh = l_sm[h];
                            const float o = lh > 0.f ? __uint_as_float(r[e]) / lh : 0.f;
                            const size_t hq = (size_t)hh * HEADS + h;
                            if (direct)
                                reinterpret_cast<__nv_bfloat16 *>(p.out)[((size_t)sg.b * p.H_q + hq) * DV + d] =
                                    __float2bfloat16_rn(o);
                            else if (split_ok)
                                p.meta.o_part[((size_t)split * p.H_q + hq) * DV + d] = o;
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(ofree);
            if (owner) {
                const float v = l > 0.f ? (m_used + log2f(l)) * kLn2Mla : -INFINITY;
                const size_t hq = (size_t)hh * HEADS + head;
                if (direct)
                    p.lse[(size_t)sg.b * p.H_q + hq] = v;
                else if (split_ok)
                    p.meta.lse_part[(size_t)split * p.H_q + hq] = v;
            }
            named_barrier_sync(1, 128);
            if (!o_ok) {
                if (lane == 0) {
                    atomicOr(&p.meta.header[kHError], DA_DEV_TIMEOUT);
                    *abort_flag = 1;
                }
                break;
            }
            ic += n;
            ++seg;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, TMEM_COLS);
}

int mla_ctas_per_part() { return 2; }
bool mla_kernel_available() { return true; }

cudaError_t launch_mla(const MlaParams &p, cudaStream_t stream, bool pdl) {
    cudaError_t e = cudaFuncSetAttribute(mla_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, mla::SMEM);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.num_parts, 2);
    cfg.blockDim = dim3(mla::THREADS);
    cfg.dynamicSmemBytes = mla::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, mla_decode_kernel, p);
}

}  // namespace da
