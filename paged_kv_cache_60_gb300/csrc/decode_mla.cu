// Split-KV decode kernel for the 656-byte FP8 latent token (MQA: 128 query
// heads share one KV head; D_qk = 576, D_v = 512), on the 5th-generation
// tensor cores (tcgen05, accumulators and one operand in tensor memory).
//
// The token format is the FlashMLA page's ("FlashMLA 注意力内核源码走读", section
// "数据加载"): 512 e4m3 values with one fp32 scale per 128 of them, then 64
// bf16 RoPE values; K is the 576 dequantised values and V their first 512.
// Dequantisation goes to bf16 (exact e4m3 value in fp32, times the scale, ->
// bf16) and the products run in bf16 with fp32 accumulation, as that section
// describes.
//
// Work split: a cluster of two CTAs (two SMs) per part. Both hold all 128
// query heads, so every MMA has 128 rows (one per head). CTA r holds dims
// [256 r, 256 r + 320) of each latent row:
//   S_r = Q[:, 288 r : 288 r + 288] K[:, same]^T   M = 128 heads, N = 64 tokens, 18 MMAs,
//                                                 Q read from tensor memory
//   the two partial S are swapped through L2 (a slot per CTA in the
//   scheduling-metadata buffer, signalled through the cluster's mbarriers) and
//   added (fp32 addition commutes, so both CTAs hold the same S bit for bit and
//   take the same softmax decisions without further exchange);
//   O[:, 256 r : 256 r + 256] += P V               M = 128 heads, N = 256 dims, 4 MMAs,
//                                                 P read from tensor memory
// So each CTA dequantises 320 of the 576 values of a token, and O (128 heads x
// 512 fp32) is split by value dim across the pair's tensor memories.
//
// Softmax (one thread per head, which also owns that head's row of S, P and
// O in tensor memory): running max m, sum l, exp2; the max is re-based only
// when it grows by more than 2^8 (then the thread rescales its O row);
// otherwise P values stay below 256. (Online softmax: attention pipeline page,
// section 三; exp via exp2: section 一.)
//
// Roles (416 threads): warp 0 issues MMAs (one lane) and owns the TMEM
// allocation; warps 1-4 load Q, run the softmax and the epilogue (TMEM lane
// quadrant = warp % 4); warps 5-12 dequantise tokens into a four-deep ring.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>

#include "common.cuh"
#include "decode_attn.h"
#include "segwalk.cuh"

namespace da {

namespace mla {
constexpr int HQ = 128;                    // query heads, all of them in each CTA
constexpr int DQK = 576, DV = 512;
constexpr int WIN = 320;                   // dims of a latent row held by one CTA: [256 r, 256 r + 320)
constexpr int WSL = WIN / 64;              // 64-dim slices of the window (5)
constexpr int UNITS = WIN / 16;            // 16-value units per token row (20)
constexpr int KSTEPS = 18;                 // 288 contraction dims per CTA, 16 per MMA
constexpr int KSLICE = kChunk * 128;       // one slice of a 64-token tile (8 KB)
constexpr int KTILE = WSL * KSLICE;        // 40 KB
constexpr int NK = 4;                      // depth of the dequantised-tile ring
constexpr int ROW_BYTES = 656;
constexpr int OFF_K = 0;                   // NK tiles
constexpr int OFF_MISC = NK * KTILE;
// misc: mbarriers, tmem base, abort flag
constexpr int NBARS = 2 * NK + 10;
constexpr int OFF_BARS = OFF_MISC;
constexpr int OFF_TMEM = OFF_BARS + NBARS * 8;
constexpr int OFF_ABORT = OFF_TMEM + 4;
constexpr int SMEM = OFF_ABORT + 12 + 1024;  // + alignment slack
constexpr int THREADS = 13 * 32;
constexpr int SM_THREADS = 128, DQ_WARPS = 8;
// tensor memory (512 columns x 128 lanes; lane = head)
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t O_COL = 0;              // O: 256 fp32 value dims
constexpr uint32_t S_COL = 256;            // S: 64 fp32 tokens
constexpr uint32_t Q_COL = 320;            // Q: 288 bf16 dims, two per column (144 columns)
constexpr uint32_t P_COL = 464;            // P: 64 bf16 tokens, two per column (32 columns)
constexpr float RESCALE_LOG2 = 8.f;        // re-base the max when it grows by more than 2^8
static_assert(SMEM <= 232448, "shared memory budget");
static_assert(P_COL + 32 <= TMEM_COLS, "tensor memory budget");
static_assert(KTILE % 1024 == 0, "1024-byte aligned operand tiles");
}  // namespace mla

constexpr float kLn2Mla = 0.6931471805599453f;

__device__ __forceinline__ uint32_t swz(int row, int c16) { return (uint32_t)(row * 128 + ((c16 ^ (row & 7)) << 4)); }

// Exact e4m3 -> fp32 without the conversion pipe: the sign, exponent and
// mantissa bits of the code are moved to the fp32 sign, the low exponent bits
// and the top mantissa bits, which gives the value times 2^-120 (a subnormal
// fp32 for e4m3 subnormals); one multiply by 2^120 (no flush to zero) makes it
// exact. The NaN codes (0x7f, 0xff) decode to +-480 here; the tokens a decode
// step reads never hold them.
__device__ __forceinline__ float e4m3_from_bits(uint32_t fbits) {
    float r;
    asm("mul.rn.f32 %0, %1, 0f7B800000;" : "=f"(r) : "f"(__uint_as_float(fbits)));  // x 2^120
    return r;
}
__device__ __forceinline__ float mul_rn(float a, float b) {
    float r;
    asm("mul.rn.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

// 16 e4m3 values times `scale` (fp32 product, then bf16 round to nearest even),
// as 16 bf16 (two 16-byte words).
__device__ __forceinline__ void dequant16(const uint4 v, float scale, uint4 &lo, uint4 &hi) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t x = w[k];
        const float f0 = e4m3_from_bits(((x << 20) & 0x07f00000u) | ((x << 24) & 0x80000000u));
        const float f1 = e4m3_from_bits(((x << 12) & 0x07f00000u) | ((x << 16) & 0x80000000u));
        const float f2 = e4m3_from_bits(((x << 4) & 0x07f00000u) | ((x << 8) & 0x80000000u));
        const float f3 = e4m3_from_bits(((x >> 4) & 0x07f00000u) | (x & 0x80000000u));
        o[2 * k] = pack_bf16(mul_rn(f0, scale), mul_rn(f1, scale));
        o[2 * k + 1] = pack_bf16(mul_rn(f2, scale), mul_rn(f3, scale));
    }
    lo = make_uint4(o[0], o[1], o[2], o[3]);
    hi = make_uint4(o[4], o[5], o[6], o[7]);
}


// SPARSE: top-k decode (the tokens are the positions p.indices lists; p.topk > 0)
template <bool SPARSE>
__global__ void __launch_bounds__(mla::THREADS, 1) mla_decode_kernel(const __grid_constant__ MlaParams p) {
    using namespace mla;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + OFF_BARS);
    uint64_t *kfull = bars, *kempty = bars + NK;
    uint64_t *sfull = bars + 2 * NK, *sfree = sfull + 1, *pfull = sfull + 2, *pfree = sfull + 3;
    uint64_t *ofull = sfull + 4, *ofree = sfull + 5, *qfull = sfull + 6, *qfree = sfull + 7;
    uint64_t *xfull = sfull + 8, *xfree = sfull + 9;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + OFF_TMEM);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + OFF_ABORT);
    const uint32_t k_base = smem_u32(smem + OFF_K);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int part = blockIdx.x;
    const uint32_t rank = cluster_ctarank();  // 0 or 1: which window of the latent row
    const uint32_t peer = rank ^ 1u;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NK; ++i) {
            mbar_init(&kfull[i], DQ_WARPS);
            mbar_init(&kempty[i], 1);
        }
        mbar_init(sfull, 1);
        mbar_init(sfree, SM_THREADS / 32);
        mbar_init(pfull, SM_THREADS / 32);
        mbar_init(pfree, 1);
        mbar_init(ofull, 1);
        mbar_init(ofree, SM_THREADS / 32);
        mbar_init(qfull, SM_THREADS / 32);
        mbar_init(qfree, 1);
        mbar_init(xfull, SM_THREADS / 32);  // the peer's four softmax warps
        mbar_init(xfree, SM_THREADS / 32);
        *abort_flag = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    if (warp == 0) tmem_alloc(tmem_slot, TMEM_COLS);
    tc_fence_before();
    cluster_sync_all();  // the peer's barriers exist before any remote arrival
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();
    pdl_launch_dependents();

    const int4 rec0 = p.meta.parts[2 * part];
    const int4 rec1 = p.meta.parts[2 * part + 1];
    const int32_t *hd = p.meta.header;
    const bool meta_ok = meta_header_ok(load_meta_header(hd), p.B, 1, p.H_q, p.splits, p.num_parts, 1, 0,
                                        p.topk) &
                         ((int)gridDim.x == p.num_parts);
    const int max_len = p.max_pages * p.page_size;

    if (!meta_ok) {
        if (threadIdx.x == 0 && rank == 0) atomicOr(&p.meta.header[kHError], DA_DEV_META_MISMATCH);
    } else if (warp == 0) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            // Two cursors walk the same chunk sequence: one issues S = Q K^T,
            // the other O += P V. The product for P goes first when it is
            // ready (the softmax of the next chunk waits on it); S is issued
            // in two halves so that a P that becomes ready meanwhile is not
            // queued behind a whole S.
            constexpr uint32_t IDESC_QK = umma_idesc_bf16(128, 64, 0, 0);
            constexpr uint32_t IDESC_PV = umma_idesc_bf16(128, 256, 0, 1);
            const int ks0 = 2 * (int)rank;  // first 16-dim step of this CTA's 288 contraction dims in its window
            SegWalker wq = make_walker(p.meta, rec0, rec1, p.B, p.seqlens, max_len, 1, 0, p.topk);
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
            int qhalf = 0;  // 0: next S starts fresh; 1: its first half is issued
            int qdone = 0;  // chunks whose S is fully issued
            bool ok = true;
            uint64_t t_idle = 0;
            uint32_t spins = 0;
            while (q_more || p_more) {
                bool issued = false;
                if (p_more && pcur < qdone && mbar_test(pfull, pcur & 1) &&
                    (pc != 0 || pseg == 0 || mbar_test(ofree, (pseg - 1) & 1))) {
                    const uint32_t kb = k_base + (pcur % NK) * KTILE;
                    tc_fence_after();
#pragma unroll
                    for (int kt = 0; kt < kChunk / 16; ++kt)
                        umma_bf16_tmem_a(tmem + O_COL, tmem + P_COL + 8 * kt, umma_desc(kb + kt * 2048, KSLICE, 1024),
                                         IDESC_PV, !(pc == 0 && kt == 0));
                    umma_commit(&kempty[pcur % NK]);
                    umma_commit(pfree);
                    if (pc == np - 1) umma_commit(ofull);
                    ++pcur;
                    if (++pc == np) {
                        pc = 0;
                        ++pseg;
                        p_more = next_seg(wp, np);
                    }
                    issued = true;
                } else if (q_more && (qhalf == 1 ||
                                      ((qc != 0 || mbar_test(qfull, qseg & 1)) &&
                                       mbar_test(&kfull[qcur % NK], (qcur / NK) & 1) &&
                                       mbar_test(sfree, (qcur & 1) ^ 1)))) {
                    const uint32_t kb = k_base + (qcur % NK) * KTILE;
                    if (qhalf == 0) tc_fence_after();
                    const int i0 = qhalf * (KSTEPS / 2);
#pragma unroll
                    for (int i = i0; i < i0 + KSTEPS / 2; ++i) {
                        const int ks = ks0 + i;
                        umma_bf16_tmem_a(tmem + S_COL, tmem + Q_COL + 8 * i,
                                         umma_desc(kb + (ks >> 2) * KSLICE + (ks & 3) * 32, 16, 1024), IDESC_QK, i > 0);
                    }
                    if (qhalf == 0) {
                        qhalf = 1;
                    } else {
                        qhalf = 0;
                        umma_commit(sfull);
                        if (qc == nq - 1) umma_commit(qfree);  // Q may be replaced once these complete
                        qdone = ++qcur;
                        if (++qc == nq) {
                            qc = 0;
                            ++qseg;
                            q_more = next_seg(wq, nq);
                        }
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
        // ------------------------------------------------------------ dequantise this CTA's window
        // A token row of the window is 20 units of 16 values. Thread dt takes
        // units dt + 256 i (i < 5) of the chunk's 64 x 20, so a warp's loads
        // cover contiguous bytes of one or two rows. Rank 0's units are NoPE
        // bytes 16 g; rank 1's are NoPE bytes 256 + 16 g (g < 16) and the 64
        // RoPE values (g >= 16, 32 bytes each). All loads of a chunk are in
        // flight while the warp waits for its tile of the ring.
        const int dt = threadIdx.x - 5 * 32;  // 0 .. 255
        SegWalker wk = make_walker(p.meta, rec0, rec1, p.B, p.seqlens, max_len, 1, 0, p.topk);
        Seg sg;
        int ic = 0;
        bool ok = true;
        while (ok && wk.next(sg)) {
            const int n = sg.lc1 - sg.lc0;
            const int32_t *bt_row = p.block_table + (size_t)sg.b * p.max_pages;
            const int32_t *idx_row = p.indices + (size_t)sg.b * p.topk;  // sparse decode only
            // sparse decode: the positions listed in this thread's slots, loaded one
            // chunk ahead so that only the block-table and row loads sit on the chain
            int tnext[5];
            if (SPARSE) {
#pragma unroll
                for (int i = 0; i < 5; ++i) {
                    const int slot = sg.lc0 * kChunk + (dt + 256 * i) / UNITS;
                    tnext[i] = (n > 0 && slot < p.topk) ? idx_row[slot] : -1;
                }
            }
            for (int c = 0; c < n && ok; ++c) {
                const int cur = ic + c, kb = cur % NK;
                const int tbase = (sg.lc0 + c) * kChunk;
                int tcur[5];
                if (SPARSE) {
#pragma unroll
                    for (int i = 0; i < 5; ++i) {
                        tcur[i] = tnext[i];
                        const int slot = tbase + kChunk + (dt + 256 * i) / UNITS;
                        tnext[i] = (c + 1 < n && slot < p.topk) ? idx_row[slot] : -1;
                    }
                }
                uint4 ra[5], rb[5];
                float sc[5];
#pragma unroll
                for (int i = 0; i < 5; ++i) {
                    const int u = dt + 256 * i, tok = u / UNITS, g = u % UNITS;
                    // dense: token tbase + tok; sparse: the position listed in slot tbase + tok
                    // (slots past topk and positions outside [0, L) are skipped: a zero row)
                    int t = tbase + tok;
                    if (SPARSE) t = tcur[i];
                    const bool valid = t >= 0 && t < sg.L;
                    ra[i] = make_uint4(0u, 0u, 0u, 0u);
                    rb[i] = ra[i];
                    sc[i] = 0.f;
#ifdef DA_PAGE_TRACE
                    if (p.page_trace && rank == 0 && g == 0 && cur < p.page_trace_cap)
                        p.page_trace[((size_t)part * p.page_trace_cap + cur) * kChunk + tok] =
                            valid ? bt_row[t / p.page_size] * p.page_size + t % p.page_size : -2;
#endif
                    if (valid) {
                        const int pg = bt_row[t / p.page_size];
                        if (pg < 0 || pg >= p.num_pages) {
                            atomicOr(&p.meta.header[kHError], DA_DEV_BAD_PAGE);
                            p.meta.header[kHErrorDetail] = pg;
                        } else {
                            const uint8_t *row = p.pool + ((size_t)pg * p.page_size + t % p.page_size) * ROW_BYTES;
                            if (rank == 1 && g >= 16) {
                                ra[i] = ldg_stream16(row + 528 + 32 * (g - 16));
                                rb[i] = ldg_stream16(row + 528 + 32 * (g - 16) + 16);
                            } else {
                                const int byte = 256 * (int)rank + 16 * g;
                                ra[i] = ldg_stream16(row + byte);
                                sc[i] = ldg_stream4f(row + 512 + 4 * (byte >> 7));
                            }
                        }
                    }
                }
                if (!(ok = mbar_wait_warp(&kempty[kb], ((cur / NK) & 1) ^ 1, abort_flag, p.wait_limit_ns))) break;
                uint8_t *kt = smem + OFF_K + kb * KTILE;
#pragma unroll
                for (int i = 0; i < 5; ++i) {
                    const int u = dt + 256 * i, tok = u / UNITS, g = u % UNITS;
                    uint4 lo = ra[i], hi = rb[i];
                    if (!(rank == 1 && g >= 16)) dequant16(ra[i], sc[i], lo, hi);
                    // window dims 16 g .. 16 g + 15: slice g / 4, chunks 2 (g % 4) and + 1; every
                    // other group of four units stores its upper chunk first (fewer bank conflicts)
                    const int sl = g >> 2, c0 = 2 * (g & 3);
                    const bool swap = (g >> 2) & 1;
                    *reinterpret_cast<uint4 *>(kt + sl * KSLICE + swz(tok, c0 + (swap ? 1 : 0))) = swap ? hi : lo;
                    *reinterpret_cast<uint4 *>(kt + sl * KSLICE + swz(tok, c0 + (swap ? 0 : 1))) = swap ? lo : hi;
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&kfull[kb]);
            }
            ic += n;
        }
        if (!ok && lane == 0) {
            atomicOr(&p.meta.header[kHError], DA_DEV_TIMEOUT);
            *abort_flag = 1;
        }
    } else {
        // ------------------------------------------------------------ Q load, softmax, epilogue (warps 1-4)
        const int quad = warp & 3;
        const int head = quad * 32 + lane;         // this thread's row of S, P, O and Q in tensor memory
        const int sid = threadIdx.x - 32;          // 0 .. 127
        const uint32_t trow = tmem + ((uint32_t)(32 * quad) << 16);
        const float sl2 = p.scale_log2;
        // partial scores travel through L2: this CTA's slot and the peer's, laid out
        // [16-byte column i][head] so that a warp's stores and loads are coalesced
        float4 *x_mine = reinterpret_cast<float4 *>(p.meta.xchg) + ((size_t)part * 2 + rank) * 16 * HQ + head;
        const float4 *x_other = reinterpret_cast<const float4 *>(p.meta.xchg) + ((size_t)part * 2 + peer) * 16 * HQ + head;
        const uint32_t xfull_peer = mapa_shared(smem_u32(xfull), peer);
        const uint32_t xfree_peer = mapa_shared(smem_u32(xfree), peer);
        const int d_base = 256 * (int)rank;        // value dims held by this CTA: [d_base, d_base + 256)
        SegWalker wk = make_walker(p.meta, rec0, rec1, p.B, p.seqlens, max_len, 1, 0, p.topk);
        Seg sg;
        int ic = 0, seg = 0;
        bool ok = true;
        while (ok && wk.next(sg)) {
            const int n = sg.lc1 - sg.lc0;
            const bool direct = sg.ns == 1;
            const int split = sg.so + sg.s;
            const bool split_ok = direct || (split >= 0 && split < p.meta.max_splits);
            __nv_bfloat16 *out_row =
                reinterpret_cast<__nv_bfloat16 *>(p.out) + ((size_t)sg.b * p.H_q + head) * DV + d_base;
            float *part_row = p.meta.o_part + ((size_t)split * p.H_q + head) * DV + d_base;
            if (n == 0) {
                // no tokens: output 0 for this CTA's value dims, lse -inf (rank 0)
                for (int k = 0; k < 32; ++k) {
                    if (direct)
                        reinterpret_cast<uint4 *>(out_row)[k] = make_uint4(0u, 0u, 0u, 0u);
                    else if (split_ok)
                        reinterpret_cast<float4 *>(part_row)[2 * k] = reinterpret_cast<float4 *>(part_row)[2 * k + 1] =
                            make_float4(0.f, 0.f, 0.f, 0.f);
                }
                if (rank == 0) {
                    if (direct)
                        p.lse[(size_t)sg.b * p.H_q + head] = -INFINITY;
                    else if (split_ok)
                        p.meta.lse_part[(size_t)split * p.H_q + head] = -INFINITY;
                }
                continue;
            }
            // this head's q, dims [288 r, 288 r + 288), into tensor memory as the A operand of S
            if (!(ok = mbar_wait_warp(qfree, (seg & 1) ^ 1, abort_flag, p.wait_limit_ns))) break;
            {
                const uint4 *qs = reinterpret_cast<const uint4 *>(reinterpret_cast<const __nv_bfloat16 *>(p.q) +
                                                                 ((size_t)sg.b * HQ + head) * DQK + 288 * rank);
#pragma unroll 1
                for (int j = 0; j < 9; ++j) {  // 32 dims = 16 columns per store
                    uint32_t r[16];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint4 v = qs[4 * j + k];
                        r[4 * k] = v.x;
                        r[4 * k + 1] = v.y;
                        r[4 * k + 2] = v.z;
                        r[4 * k + 3] = v.w;
                    }
                    tmem_st16(trow + Q_COL + 16 * j, r);
                }
                tmem_wait_st();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(qfull);
            float m_used = -INFINITY, l = 0.f;
            for (int c = 0; c < n; ++c) {
                const int cur = ic + c;
                const int cbase = (sg.lc0 + c) * kChunk;
                // sparse decode: this chunk's listed positions (slots lane, lane + 32),
                // loaded before the waits so that their latency overlaps them
                int t0 = -1, t1 = -1;
                if (SPARSE) {
                    const int32_t *ir = p.indices + (size_t)sg.b * p.topk + cbase;
                    if (cbase + lane < p.topk) t0 = ir[lane];
                    if (cbase + lane + 32 < p.topk) t1 = ir[lane + 32];
                }
                bool w_ok = mbar_wait_warp(sfull, cur & 1, abort_flag, p.wait_limit_ns);
                tc_fence_after();
                float s[64];
                {
                    uint32_t r[64];
                    tmem_ld64_sync(trow + S_COL, r);
#pragma unroll
                    for (int e = 0; e < 64; ++e) s[e] = __uint_as_float(r[e]);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(sfree);
                // swap partial rows with the peer: ours into its buffer once it has
                // consumed the previous one, then add the peer's into ours
                if (cur > 0) w_ok = w_ok && mbar_wait_warp(xfree, (cur - 1) & 1, abort_flag, p.wait_limit_ns);
                if (w_ok) {
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        x_mine[i * HQ] = make_float4(s[4 * i], s[4 * i + 1], s[4 * i + 2], s[4 * i + 3]);
                    fence_acq_rel_cluster();  // each lane's stores, before the warp's release below
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster(xfull_peer);
                }
                w_ok = w_ok && mbar_wait_warp_cluster(xfull, cur & 1, abort_flag, p.wait_limit_ns);
                if (w_ok) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float4 v = __ldcg(x_other + i * HQ);
                        s[4 * i] += v.x;
                        s[4 * i + 1] += v.y;
                        s[4 * i + 2] += v.z;
                        s[4 * i + 3] += v.w;
                    }
                    // the sums above consumed every load, so the peer may overwrite the buffer
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster_relaxed(xfree_peer);
                }
                float mx = -INFINITY;
                if (SPARSE) {
                    // sparse: slot e counts when it lies before topk and lists a position in
                    // [0, L); the warp's ballots give the 64 bits (vm0: slots 0-31, vm1: 32-63)
                    const uint32_t vm0 = __ballot_sync(0xffffffffu, t0 >= 0 && t0 < sg.L);
                    const uint32_t vm1 = __ballot_sync(0xffffffffu, t1 >= 0 && t1 < sg.L);
#pragma unroll
                    for (int e = 0; e < 64; ++e) {
                        const bool v = ((e < 32 ? vm0 >> e : vm1 >> (e - 32)) & 1u) != 0u;
                        s[e] = v ? s[e] * sl2 : -INFINITY;
                        mx = fmaxf(mx, s[e]);
                    }
                } else {
                    const int nvalid = sg.L - cbase;  // >= 1: tokens of this chunk in the sequence
#pragma unroll
                    for (int e = 0; e < 64; ++e) {
                        s[e] = (e < nvalid) ? s[e] * sl2 : -INFINITY;
                        mx = fmaxf(mx, s[e]);
                    }
                }
                // P's columns and O are free once the previous chunk's PV has completed
                if (cur > 0) w_ok = w_ok && mbar_wait_warp(pfree, (cur - 1) & 1, abort_flag, p.wait_limit_ns);
                if (__any_sync(0xffffffffu, !w_ok || *abort_flag != 0)) {
                    if (lane == 0) {
                        atomicOr(&p.meta.header[kHError], DA_DEV_TIMEOUT);
                        *abort_flag = 1;
                    }
                    ok = false;
                    break;
                }
                tc_fence_after();
                const float m_new = fmaxf(m_used, mx);
                const bool need = c > 0 && (m_new > m_used + RESCALE_LOG2);
                if (c == 0) m_used = m_new;
                if (__any_sync(0xffffffffu, need)) {
                    // re-base: scale this head's O row (tensor-memory loads and stores are warp-wide)
                    const float alpha = need ? ex2(m_used - m_new) : 1.f;
                    if (need) {
                        m_used = m_new;
                        l *= alpha;
                    }
#pragma unroll 1
                    for (int k = 0; k < 16; ++k) {
                        uint32_t r[16];
                        tmem_ld16_sync(trow + O_COL + 16 * k, r);
#pragma unroll
                        for (int e = 0; e < 16; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
                        tmem_st16(trow + O_COL + 16 * k, r);
                    }
                }
                // P row of this head: 64 tokens as bf16 pairs, the A operand of O += P V
                // (while no token has counted yet, m_used is -inf: exponents from 0 give P = 0)
                const float base = (SPARSE && m_used == -INFINITY) ? 0.f : m_used;
                float ps = 0.f;
                uint32_t pk[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const float p0 = ex2(s[2 * e] - base), p1 = ex2(s[2 * e + 1] - base);
                    ps += p0 + p1;
                    pk[e] = pack_bf16(p0, p1);
                }
                l += ps;
                {
                    uint32_t r0[16], r1[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        r0[e] = pk[e];
                        r1[e] = pk[16 + e];
                    }
                    tmem_st16(trow + P_COL, r0);
                    tmem_st16(trow + P_COL + 16, r1);
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(pfull);
            }
            if (!ok) break;
            // ---- epilogue: O / l for this CTA's 256 value dims of this head
            const bool o_ok = mbar_wait_warp(ofull, seg & 1, abort_flag, p.wait_limit_ns);
            tc_fence_after();
            if (o_ok) {
                const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
                for (int k = 0; k < 16; ++k) {
                    uint32_t r[16];
                    tmem_ld16_sync(trow + O_COL + 16 * k, r);
                    if (direct) {
                        uint32_t b[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            b[e] = pack_bf16(__uint_as_float(r[2 * e]) * inv, __uint_as_float(r[2 * e + 1]) * inv);
                        reinterpret_cast<uint4 *>(out_row)[2 * k] = make_uint4(b[0], b[1], b[2], b[3]);
                        reinterpret_cast<uint4 *>(out_row)[2 * k + 1] = make_uint4(b[4], b[5], b[6], b[7]);
                    } else if (split_ok) {
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            reinterpret_cast<float4 *>(part_row)[4 * k + e] =
                                make_float4(__uint_as_float(r[4 * e]) * inv, __uint_as_float(r[4 * e + 1]) * inv,
                                            __uint_as_float(r[4 * e + 2]) * inv, __uint_as_float(r[4 * e + 3]) * inv);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(ofree);
            if (rank == 0) {
                const float v = l > 0.f ? (m_used + log2f(l)) * kLn2Mla : -INFINITY;
                if (direct)
                    p.lse[(size_t)sg.b * p.H_q + head] = v;
                else if (split_ok)
                    p.meta.lse_part[(size_t)split * p.H_q + head] = v;
            }
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
    cluster_sync_all();  // the peer has finished writing into this CTA's shared memory
}

int mla_ctas_per_part() { return 2; }
bool mla_kernel_available() { return true; }

// Parts that can run at once: clusters of two CTAs, one CTA per SM.
int mla_max_parts() {
    static std::atomic<int> cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (const int c = cached[dev].load(std::memory_order_relaxed)) return c;
    if (cudaFuncSetAttribute(mla_decode_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, mla::SMEM) !=
        cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1024, 2);
    cfg.blockDim = dim3(mla::THREADS);
    cfg.dynamicSmemBytes = mla::SMEM;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 2;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, mla_decode_kernel<false>, &cfg) != cudaSuccess) return 0;
    cached[dev].store(n, std::memory_order_relaxed);
    return n;
}

cudaError_t launch_mla(const MlaParams &p, cudaStream_t stream, bool pdl) {
    auto kern = p.topk > 0 ? mla_decode_kernel<true> : mla_decode_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, mla::SMEM);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.num_parts, 2);
    cfg.blockDim = dim3(mla::THREADS);
    cfg.dynamicSmemBytes = mla::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 2;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace da
