// Split-KV decode kernel for the 656-byte FP8 latent token (MQA: 128 query
// heads share one KV head; D_qk = 576, D_v = 512), on the 5th-generation
// tensor cores (tcgen05, accumulators and one operand in tensor memory).
//
// The token format is the FlashMLA page's ("FlashMLA 注意力内核源码走读", section
// "数据加载"): 512 e4m3 values with one fp32 scale per 128 of them, then 64
// bf16 RoPE values; K is the 576 dequantised values and V their first 512.
// Dequantisation goes to bf16 (exact e4m3 value times the scale in fp32, ->
// bf16) and the products run in bf16 with fp32 accumulation, as that section
// describes.
//
// Work split: every part (a range of 64-token chunks) runs on 2 * s_q CTAs
// that never communicate: CTA (j, r) serves query token j (draft j of s_q)
// and value dims [256 r, 256 r + 256). Each computes the whole score matrix
// of its draft,
//   S = Q K^T      M = 128 heads, N = 64 tokens, K = 576 dims: 36 MMAs, q dims
//                  [0, 320) read from tensor memory, [320, 576) from shared memory
// so every MMA has 128 rows (one per head), runs the online softmax on it, and
// accumulates its half of the output,
//   O[:, 256 r : 256 r + 256] += P V     M = 128, N = 256, K = 64 tokens: 4 MMAs,
//                                        P read from tensor memory.
// O (128 heads x 512 fp32) fills a whole SM's tensor memory, hence the split
// by value dim; the QK^T work is done by both CTAs of a pair, which trades
// tensor time for the 32 KB of partial scores per chunk that a split of the
// contraction dims would have to exchange. The two CTAs read the same rows;
// the second read is served by L2.
//
// Softmax (one thread per head, which also owns that head's row of S, P and
// O in tensor memory): running max m, sum l, exp2; the max is re-based only
// when it grows by more than 2^8 (then the thread rescales its O row);
// otherwise P values stay below 256. (Online softmax: attention pipeline page,
// section 三; exp via exp2: section 一.)
//
// Roles (416 threads): warp 0 issues MMAs (one lane) and owns the tensor
// memory; warps 1-4 load q, run the softmax and the epilogue (tensor-memory
// lane quadrant = warp % 4); warps 5-12 dequantise tokens into two rings of
// two slots: the value slices of this CTA (freed when P V has read them) and
// the other five slices (freed as soon as Q K^T has read them). The MMAs
// run in the order QK(c), PV(c - 1), QK(c + 1), ..., and QK(c) reads the
// five K-only slices first, so the value slot of chunk c + 1 has the time of
// those MMAs to be refilled.
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "decode_attn.h"
#include "segwalk.cuh"

namespace da {

namespace mla {
constexpr int HQ = 128;                     // query heads of one query token
constexpr int DQK = 576, DV = 512;
constexpr int NSL = 9;                      // 64-dim slices of a latent row: 8 NoPE + 1 RoPE
constexpr int SLICE = kChunk * 128;         // one slice of a 64-token tile (128-byte swizzle): 8 KB
constexpr int QSLICE = HQ * 128;            // one slice of q for the 128 heads: 16 KB
constexpr int VSL = 4;                      // slices of the value dims one CTA accumulates
constexpr int KSL = NSL - VSL;              // the other five, read by Q K^T only
constexpr int VSLOT = VSL * SLICE;          // 32 KB
constexpr int KSLOT = KSL * SLICE;          // 40 KB
constexpr int NR = 2;                       // slots per ring
constexpr int QTM = 5;                      // q slices in tensor memory: dims [0, 320)
constexpr int QSM = NSL - QTM;              // q slices in shared memory: dims [320, 576)
constexpr int KU = 24;                      // 16-byte units of a row that only Q K^T reads: 16 NoPE + 8 RoPE
constexpr int VU = 16;                      // NoPE units of the value dims of one CTA
constexpr int DQ_WARPS = 8, DQ_THREADS = DQ_WARPS * 32;
constexpr int KUPT = kChunk * KU / DQ_THREADS;  // K-only units per dequantising thread and chunk: 6
constexpr int VUPT = kChunk * VU / DQ_THREADS;  // value units per dequantising thread and chunk: 4
constexpr int SM_WARPS = 4;
constexpr int THREADS = (1 + SM_WARPS + DQ_WARPS) * 32;
constexpr int ROW_BYTES = 656;
constexpr int OFF_Q = 0;
constexpr int OFF_V = OFF_Q + QSM * QSLICE;
constexpr int OFF_K = OFF_V + NR * VSLOT;
constexpr int OFF_BARS = OFF_K + NR * KSLOT;
constexpr int NBARS = 4 * NR + 10;
constexpr int OFF_TMEM = OFF_BARS + NBARS * 8;
constexpr int OFF_ABORT = OFF_TMEM + 4;
constexpr int SMEM = OFF_ABORT + 12 + 1024;  // + alignment slack
// tensor memory (512 columns x 128 lanes; lane = head)
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t O_COL = 0;               // O: 256 fp32 value dims
constexpr uint32_t S_COL = 256;             // S: 64 fp32 tokens
constexpr uint32_t P_COL = 320;             // P: 64 bf16 tokens, two per column (32 columns)
constexpr uint32_t Q_COL = 352;             // q dims [0, 320): two bf16 per column (160 columns)
constexpr float RESCALE_LOG2 = 8.f;         // re-base the max when it grows by more than 2^8
static_assert(KUPT * DQ_THREADS == kChunk * KU && VUPT * DQ_THREADS == kChunk * VU, "units per chunk");
static_assert(Q_COL + QTM * 32 == TMEM_COLS, "tensor memory budget");
static_assert(SMEM <= 232448, "shared memory budget");
static_assert(OFF_V % 1024 == 0 && OFF_K % 1024 == 0 && VSLOT % 1024 == 0 && KSLOT % 1024 == 0,
              "1024-byte aligned operand tiles");
}  // namespace mla

constexpr float kLn2Mla = 0.6931471805599453f;

__device__ __forceinline__ uint32_t swz(int row, int c16) { return (uint32_t)(row * 128 + ((c16 ^ (row & 7)) << 4)); }

__device__ __forceinline__ float mul_rn(float a, float b) {
    float r;
    asm("mul.rn.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

// Exact e4m3 -> fp32 without the conversion pipe, for the code in bits
// [24, 32) of x: an arithmetic shift by 4 puts its exponent and mantissa on
// fp32 bits 20-26 and copies its sign onto bits 27-31; the mask keeps bits
// 20-26 and the sign at bit 31. The pattern is the code's value times
// 2^-120 (an fp32 subnormal for e4m3 subnormals). The NaN codes (0x7f, 0xff)
// read as +-480 here; the tokens a decode step reads never hold them.
__device__ __forceinline__ float e4m3_top_scaled(uint32_t x) {
    return __uint_as_float((uint32_t)((int32_t)x >> 4) & 0x87F00000u);
}

// 16 e4m3 values times `scale` (one fp32 rounding of the exact product, then
// bf16 round to nearest even), as 16 bf16 (two 16-byte words). For scales
// below 2^8 the 2^120 that the bit moves leave out is folded into the scale
// (scale * 2^120 is exact), so one multiply gives RN(e4m3 * scale); larger or
// non-finite scales take a second, exact multiply by 2^120 first.
__device__ __forceinline__ void dequant16(const uint4 v, float scale, uint4 &lo, uint4 &hi) {
    const float two120 = __uint_as_float(0x7B800000u);
    const bool folded = scale < 256.f;
    const float m = folded ? mul_rn(scale, two120) : scale;
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float f[16];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t x = w[k];
        f[4 * k] = e4m3_top_scaled(x << 24);
        f[4 * k + 1] = e4m3_top_scaled(x << 16);
        f[4 * k + 2] = e4m3_top_scaled(x << 8);
        f[4 * k + 3] = e4m3_top_scaled(x);
    }
    if (folded) {
#pragma unroll
        for (int e = 0; e < 16; ++e) f[e] = mul_rn(f[e], m);
    } else {
#pragma unroll
        for (int e = 0; e < 16; ++e) f[e] = mul_rn(mul_rn(f[e], two120), m);
    }
    lo = make_uint4(pack_bf16(f[0], f[1]), pack_bf16(f[2], f[3]), pack_bf16(f[4], f[5]), pack_bf16(f[6], f[7]));
    hi = make_uint4(pack_bf16(f[8], f[9]), pack_bf16(f[10], f[11]), pack_bf16(f[12], f[13]),
                    pack_bf16(f[14], f[15]));
}

// Slice s of a latent row in this CTA's rings: the value slot holds slices
// [4 r, 4 r + 4), the K-only slot the other five in increasing order.
__device__ __forceinline__ bool is_v_slice(int s, int r) { return (s >> 2) == r && s < 8; }
__device__ __forceinline__ int k_slot_index(int s, int r) { return r == 0 ? s - 4 : (s < 4 ? s : 4); }

// S = Q K^T for one chunk on CTA rank R: the five K-only slices first, then the
// four value slices (q slices below QTM from tensor memory, the others from
// shared memory); KONLY selects the K-only or the value group.
template <int R, bool KONLY>
__device__ __forceinline__ void mla_issue_qk(uint32_t tmem, uint64_t dq0, uint64_t dslot) {
    using namespace mla;
    constexpr uint32_t IDESC_QK = umma_idesc_bf16(128, 64, 0, 0);
#pragma unroll
    for (int k = 0; k < (KONLY ? KSL : VSL); ++k) {
        const int s = KONLY ? (R == 0 ? 4 + k : (k < 4 ? k : 8)) : 4 * R + k;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint64_t db = dslot + (uint64_t)((k * SLICE + 32 * i) >> 4);
            const bool acc = !(KONLY && k == 0 && i == 0);
            if (s < QTM)
                umma_bf16_tmem_a_w(tmem + S_COL, tmem + Q_COL + 32 * s + 8 * i, db, IDESC_QK, acc);
            else
                umma_bf16_ss_w(tmem + S_COL, dq0 + (uint64_t)(((s - QTM) * QSLICE + 32 * i) >> 4), db, IDESC_QK,
                               acc);
        }
    }
}

// The MMA warp of the latent-token kernel: per chunk c, S = Q K^T, then
// O += P V of chunk c - 1 (P of chunk c - 1 is ready by then, and these MMAs
// fill the time in which the softmax reads S of chunk c); a segment's last
// P V goes before the next segment's Q K^T.
template <int R>
__device__ __noinline__ void mla_issue(const MlaParams &p, uint8_t *smem, uint32_t tmem, int4 rec0, int4 rec1,
                                       int max_len, volatile int *abort_flag) {
    using namespace mla;
    constexpr uint32_t IDESC_PV = umma_idesc_bf16(128, 256, 0, 1);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + OFF_BARS);
    uint64_t *kfull = bars, *kempty = bars + NR, *vfull = bars + 2 * NR, *vempty = bars + 3 * NR;
    uint64_t *sfull = bars + 4 * NR, *sfree = sfull + 1, *pfull = sfull + 2, *pfree = sfull + 3;
    uint64_t *ofull = sfull + 4, *ofree = sfull + 5, *qfull = sfull + 6, *qfree = sfull + 7;
    uint64_t *drain = sfull + 8;
    // descriptors of the operand tiles, advanced by constant offsets
    const uint64_t dq0 = umma_desc(smem_u32(smem + OFF_Q), 16, 1024);
    const uint64_t dk0 = umma_desc(smem_u32(smem + OFF_K), 16, 1024);
    const uint64_t dv0 = umma_desc(smem_u32(smem + OFF_V), 16, 1024);
    const uint64_t dpv0 = umma_desc(smem_u32(smem + OFF_V), SLICE, 1024);
    SegWalker wk = make_walker(p.meta, rec0, rec1, p.B, p.seqlens, max_len, p.s_q, 0, p.topk);
    Seg sg;
    bool ok = true;
    int cur = 0, nseg = 0;
    int pend = -1, pend_first = 0, pend_last = 0, pend_seg = 0;
    auto wait = [&](uint64_t *bar, uint32_t par) -> bool {
        return ok && (ok = mbar_wait_warp(bar, par, abort_flag, p.wait_limit_ns));
    };
    // O[:, value dims] += P(x) V(x)
    auto issue_pv = [&](int x, bool first, bool last, int seg) {
        if (!wait(pfull, x & 1)) return;
        if (first && !wait(ofree, (seg & 1) ^ 1)) return;
        tc_fence_after();
        const uint64_t dv = dpv0 + (uint64_t)(((x % NR) * VSLOT) >> 4);
#pragma unroll
        for (int kt = 0; kt < kChunk / 16; ++kt)
            umma_bf16_tmem_a_w(tmem + O_COL, tmem + P_COL + 8 * kt, dv + (uint64_t)((kt * 2048) >> 4), IDESC_PV,
                               !(first && kt == 0));
        umma_commit_w(&vempty[x % NR]);
        umma_commit_w(pfree);
        if (last) umma_commit_w(ofull);
    };
    while (ok && wk.next(sg)) {
        const int n = sg.lc1 - sg.lc0;
        if (n == 0) continue;
        for (int c = 0; c < n && ok; ++c, ++cur) {
            const int slot = cur % NR;
            const uint32_t par = (cur / NR) & 1;
            if (c == 0 && !wait(qfull, nseg & 1)) break;
            if (!wait(&kfull[slot], par) || !wait(sfree, (cur & 1) ^ 1)) break;
            tc_fence_after();
            mla_issue_qk<R, true>(tmem, dq0, dk0 + (uint64_t)((slot * KSLOT) >> 4));
            if (!wait(&vfull[slot], par)) break;
            tc_fence_after();
            mla_issue_qk<R, false>(tmem, dq0, dv0 + (uint64_t)((slot * VSLOT) >> 4));
            umma_commit_w(sfull);
            umma_commit_w(&kempty[slot]);
            if (c == n - 1) umma_commit_w(qfree);  // q may be replaced once these complete
            if (pend >= 0) issue_pv(pend, pend_first, pend_last, pend_seg);
            pend = cur;
            pend_first = c == 0;
            pend_last = c == n - 1;
            pend_seg = nseg;
            if (c == n - 1 && ok) {
                issue_pv(pend, pend_first, pend_last, pend_seg);
                pend = -1;
            }
        }
        ++nseg;
    }
    if (!ok && (threadIdx.x & 31) == 0) {
        atomicOr(&p.meta.header[kHError], DA_DEV_TIMEOUT);
        *abort_flag = 1;
    }
    // every product issued here has completed before the tensor memory goes away
    umma_commit_w(drain);
    mbar_wait_timed(drain, 0, 100000000ull);
}

// SPARSE: top-k decode (the tokens are the positions p.indices lists; p.topk > 0)
template <bool SPARSE>
__global__ void __launch_bounds__(mla::THREADS, 1) mla_decode_kernel(const __grid_constant__ MlaParams p) {
    using namespace mla;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + OFF_BARS);
    uint64_t *kfull = bars, *kempty = bars + NR, *vfull = bars + 2 * NR, *vempty = bars + 3 * NR;
    uint64_t *sfull = bars + 4 * NR, *sfree = sfull + 1, *pfull = sfull + 2, *pfree = sfull + 3;
    uint64_t *ofull = sfull + 4, *ofree = sfull + 5, *qfull = sfull + 6, *qfree = sfull + 7;
    uint64_t *drain = sfull + 8, *stall = sfull + 9;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + OFF_TMEM);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + OFF_ABORT);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int part = blockIdx.x;
    const int r = blockIdx.y & 1;               // value dims [256 r, 256 r + 256)
    const int draft = blockIdx.y >> 1;          // query token j of s_q

    if (threadIdx.x == 0) {
        for (int i = 0; i < NR; ++i) {
            mbar_init(&kfull[i], DQ_WARPS);
            mbar_init(&vfull[i], DQ_WARPS);
            mbar_init(&kempty[i], 1);
            mbar_init(&vempty[i], 1);
        }
        mbar_init(sfull, 1);
        mbar_init(sfree, SM_WARPS);
        mbar_init(pfull, SM_WARPS);
        mbar_init(pfree, 1);
        mbar_init(ofull, 1);
        mbar_init(ofree, SM_WARPS);
        mbar_init(qfull, SM_WARPS);
        mbar_init(qfree, 1);
        mbar_init(drain, 1);
        mbar_init(stall, 1);
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
    const bool meta_ok = meta_header_ok(load_meta_header(p.meta.header), p.B, 1, p.H_q, p.splits, p.num_parts,
                                        p.s_q, 0, p.topk) &
                         ((int)gridDim.x == p.num_parts) & ((int)gridDim.y == 2 * p.s_q);
    const int max_len = p.max_pages * p.page_size;

    if (!meta_ok) {
        if (threadIdx.x == 0 && blockIdx.y == 0) atomicOr(&p.meta.header[kHError], DA_DEV_META_MISMATCH);
    } else if (warp == 0) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp walks the schedule and waits; one elected lane issues
        // each MMA and commit (the descriptors stay warp-uniform).
        if (r == 0)
            mla_issue<0>(p, smem, tmem, rec0, rec1, max_len, abort_flag);
        else
            mla_issue<1>(p, smem, tmem, rec0, rec1, max_len, abort_flag);
    } else if (warp >= 1 + SM_WARPS) {
        // ------------------------------------------------------------ dequantise whole rows
        // A row is 40 units of 16 bytes: 32 of NoPE codes (16 values, the scale of
        // their 128-value block), 8 of RoPE values (8 bf16, copied as stored). Per
        // chunk, the 24 units per row that only Q K^T reads (16 NoPE, 8 RoPE) are
        // loaded, converted and stored first; then the 16 units of this CTA's
        // value dims. Thread dt takes units dt + 256 i of each kind, so a warp's
        // loads cover contiguous bytes of one or two rows.
        const int dt = threadIdx.x - (1 + SM_WARPS) * 32;  // 0 .. 255
        SegWalker wk = make_walker(p.meta, rec0, rec1, p.B, p.seqlens, max_len, p.s_q, 0, p.topk);
        Seg sg;
        int cur = 0;
        bool ok = true;
        uint8_t *const vring = smem + OFF_V;
        uint8_t *const kring = smem + OFF_K;
        while (ok && wk.next(sg)) {
            const int n = sg.lc1 - sg.lc0;
            const int32_t *bt_row = p.block_table + (size_t)sg.b * p.max_pages;
            const int32_t *idx_row = p.indices + (size_t)sg.b * p.topk;  // sparse decode only
            // one unit: its 16 bytes of the row of position t (zero when t is outside
            // the sequence or its page outside the pool) and, for NoPE, its scale
            auto load_unit = [&](int t, int g, uint4 &v, float &sc) {
                v = make_uint4(0u, 0u, 0u, 0u);
                sc = 0.f;
                if (t < 0 || t >= sg.L) return;
                const int pg = bt_row[t / p.page_size];
                if (pg < 0 || pg >= p.num_pages) {
                    atomicOr(&p.meta.header[kHError], DA_DEV_BAD_PAGE);
                    p.meta.header[kHErrorDetail] = pg;
                    return;
                }
                const uint8_t *row = p.pool + ((size_t)pg * p.page_size + t % p.page_size) * ROW_BYTES;
                if (g >= 32) {
                    v = ldg_stream16(row + 528 + 16 * (g - 32));
                } else {
                    v = ldg_stream16(row + 16 * g);
                    sc = ldg_stream4f(row + 512 + 4 * (g >> 3));
                }
            };
            // converts (NoPE) or copies (RoPE) one unit into its slice of a tile
            auto store_unit = [&](uint8_t *slice, int tok, int g, const uint4 v, float sc) {
                if (g >= 32) {  // 16-byte chunk g - 32 of slice 8, as stored
                    *reinterpret_cast<uint4 *>(slice + swz(tok, g - 32)) = v;
                    return;
                }
                uint4 lo, hi;
                dequant16(v, sc, lo, hi);
                // 16-byte chunks c0, c0 + 1 of the slice's row; odd slices store the
                // upper chunk first (fewer bank conflicts across the warp)
                const int c0 = 2 * (g & 3);
                const bool swap = (g >> 2) & 1;
                *reinterpret_cast<uint4 *>(slice + swz(tok, c0 + (swap ? 1 : 0))) = swap ? hi : lo;
                *reinterpret_cast<uint4 *>(slice + swz(tok, c0 + (swap ? 0 : 1))) = swap ? lo : hi;
            };
            for (int c = 0; c < n && ok; ++c, ++cur) {
                const int slot = cur % NR;
                const uint32_t par = ((cur / NR) & 1) ^ 1;
                const int tbase = (sg.lc0 + c) * kChunk;
                // dense: token tbase + tok; sparse: the position listed in slot tbase + tok
                // (slots past topk and positions outside [0, L) are skipped: a zero row)
                auto position = [&](int tok) -> int {
                    if (!SPARSE) return tbase + tok;
                    return tbase + tok < p.topk ? idx_row[tbase + tok] : -1;
                };
                {
                    uint4 v[KUPT];
                    float sc[KUPT];
#pragma unroll
                    for (int i = 0; i < KUPT; ++i) {
                        const int u = dt + DQ_THREADS * i, tok = u / KU, kg = u % KU;
                        const int g = kg < 16 ? 16 * (1 - r) + kg : 16 + kg;
                        const int t = position(tok);
#ifdef DA_PAGE_TRACE
                        if (p.page_trace && blockIdx.y == 0 && kg == 0 && cur < p.page_trace_cap)
                            p.page_trace[((size_t)part * p.page_trace_cap + cur) * kChunk + tok] =
                                (t >= 0 && t < sg.L) ? bt_row[t / p.page_size] * p.page_size + t % p.page_size : -2;
#endif
                        load_unit(t, g, v[i], sc[i]);
                    }
                    // the K-only slots are free once Q K^T of the chunk two back has read them
                    if (!(ok = mbar_wait_warp(&kempty[slot], par, abort_flag, p.wait_limit_ns))) break;
#pragma unroll
                    for (int i = 0; i < KUPT; ++i) {
                        const int u = dt + DQ_THREADS * i, tok = u / KU, kg = u % KU;
                        const int g = kg < 16 ? 16 * (1 - r) + kg : 16 + kg;
                        const int s = g < 32 ? g >> 2 : 8;
                        store_unit(kring + slot * KSLOT + k_slot_index(s, r) * SLICE, tok, g, v[i], sc[i]);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&kfull[slot]);
                }
                {
                    uint4 v[VUPT];
                    float sc[VUPT];
#pragma unroll
                    for (int i = 0; i < VUPT; ++i) {
                        const int u = dt + DQ_THREADS * i, tok = u / VU;
                        load_unit(position(tok), 16 * r + u % VU, v[i], sc[i]);
                    }
                    // the value slots once P V of that chunk has read them
                    if (!(ok = mbar_wait_warp(&vempty[slot], par, abort_flag, p.wait_limit_ns))) break;
#pragma unroll
                    for (int i = 0; i < VUPT; ++i) {
                        const int u = dt + DQ_THREADS * i, tok = u / VU, g = 16 * r + u % VU;
                        store_unit(vring + slot * VSLOT + ((g >> 2) - 4 * r) * SLICE, tok, g, v[i], sc[i]);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&vfull[slot]);
                }
            }
        }
        if (!ok && lane == 0) {
            atomicOr(&p.meta.header[kHError], DA_DEV_TIMEOUT);
            *abort_flag = 1;
        }
    } else {
        // ------------------------------------------------------------ q load, softmax, epilogue (warps 1-4)
        const int quad = warp & 3;
        const int head = quad * 32 + lane;         // this thread's row of S, P, O and q in tensor memory
        const uint32_t trow = tmem + ((uint32_t)(32 * quad) << 16);
        const float sl2 = p.scale_log2;
        const int rows = p.s_q * HQ;               // output rows of a request: [query token][head]
        const int d_base = 256 * r;                // value dims of this CTA
        bool ok = true;
        if (p.debug_stall) {
            // test build only: a wait that nothing completes runs out
            ok = mbar_wait_warp(stall, 0, abort_flag, p.wait_limit_ns);
            if (!ok && lane == 0) {
                atomicOr(&p.meta.header[kHError], DA_DEV_TIMEOUT);
                *abort_flag = 1;
            }
        }
        SegWalker wk = make_walker(p.meta, rec0, rec1, p.B, p.seqlens, max_len, p.s_q, 0, p.topk);
        Seg sg;
        int cur = 0, nseg = 0;
        while (ok && wk.next(sg)) {
            const int n = sg.lc1 - sg.lc0;
            const bool direct = sg.ns == 1;
            const int split = sg.so + sg.s;
            const bool split_ok = direct || (split >= 0 && split < p.meta.max_splits);
            const size_t orow = direct ? (size_t)sg.b * rows + draft * HQ + head
                                       : (size_t)split * rows + draft * HQ + head;
            __nv_bfloat16 *out_row = reinterpret_cast<__nv_bfloat16 *>(p.out) + orow * DV + d_base;
            float *part_row = p.meta.o_part + orow * DV + d_base;
            float *lse_dst = direct ? p.lse + orow : p.meta.lse_part + orow;
            if (n == 0) {
                // no tokens: output 0 for this CTA's value dims, lse -inf (r = 0)
                for (int k = 0; k < 32; ++k) {
                    if (direct)
                        reinterpret_cast<uint4 *>(out_row)[k] = make_uint4(0u, 0u, 0u, 0u);
                    else if (split_ok)
                        reinterpret_cast<float4 *>(part_row)[2 * k] = reinterpret_cast<float4 *>(part_row)[2 * k + 1] =
                            make_float4(0.f, 0.f, 0.f, 0.f);
                }
                if (r == 0 && (direct || split_ok)) *lse_dst = -INFINITY;
                continue;
            }
            // this head's q row of query token `draft`: dims [0, 320) into tensor memory
            // (the A operand of its first five slices), dims [320, 576) into shared memory
            if (!(ok = mbar_wait_warp(qfree, (nseg & 1) ^ 1, abort_flag, p.wait_limit_ns))) break;
            {
                const uint4 *qs = reinterpret_cast<const uint4 *>(reinterpret_cast<const __nv_bfloat16 *>(p.q) +
                                                                 ((size_t)sg.b * rows + draft * HQ + head) * DQK);
#pragma unroll 1
                for (int j = 0; j < 10; ++j) {  // 32 dims = 16 columns per store
                    uint32_t rr[16];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint4 v = qs[4 * j + k];
                        rr[4 * k] = v.x;
                        rr[4 * k + 1] = v.y;
                        rr[4 * k + 2] = v.z;
                        rr[4 * k + 3] = v.w;
                    }
                    tmem_st16(trow + Q_COL + 16 * j, rr);
                }
#pragma unroll 4
                for (int k = 0; k < QSM * 8; ++k)  // 16-byte chunk k % 8 of slice k / 8
                    *reinterpret_cast<uint4 *>(smem + OFF_Q + (k >> 3) * QSLICE + swz(head, k & 7)) = qs[40 + k];
                tmem_wait_st();
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(qfull);
            // tokens this query token sees: draft j of s_q sits at position L - s_q + j
            const int L_vis = sg.L - p.s_q + 1 + draft;
            float m_used = -INFINITY, l = 0.f;
            for (int c = 0; c < n; ++c, ++cur) {
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
                    uint32_t rr[64];
                    tmem_ld64_sync(trow + S_COL, rr);
#pragma unroll
                    for (int e = 0; e < 64; ++e) s[e] = __uint_as_float(rr[e]);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(sfree);
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
                    const int nvalid = L_vis - cbase;  // tokens of this chunk the query token sees
#pragma unroll
                    for (int e = 0; e < 64; ++e) {
                        s[e] = (e < nvalid) ? s[e] * sl2 : -INFINITY;
                        mx = fmaxf(mx, s[e]);
                    }
                }
                // P's columns and O are free once the previous chunk's P V has completed
                w_ok = w_ok && mbar_wait_warp(pfree, (cur & 1) ^ 1, abort_flag, p.wait_limit_ns);
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
                        uint32_t rr[16];
                        tmem_ld16_sync(trow + O_COL + 16 * k, rr);
#pragma unroll
                        for (int e = 0; e < 16; ++e) rr[e] = __float_as_uint(__uint_as_float(rr[e]) * alpha);
                        tmem_st16(trow + O_COL + 16 * k, rr);
                    }
                }
                // P row of this head: 64 tokens as bf16 pairs, the A operand of O += P V
                // (while no token has counted yet, m_used is -inf: exponents from 0 give P = 0)
                const float base = m_used == -INFINITY ? 0.f : m_used;
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
            const bool o_ok = mbar_wait_warp(ofull, nseg & 1, abort_flag, p.wait_limit_ns);
            tc_fence_after();
            if (o_ok) {
                const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
                for (int k = 0; k < 16; ++k) {
                    uint32_t rr[16];
                    tmem_ld16_sync(trow + O_COL + 16 * k, rr);
                    if (direct) {
                        uint32_t b[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            b[e] = pack_bf16(__uint_as_float(rr[2 * e]) * inv, __uint_as_float(rr[2 * e + 1]) * inv);
                        reinterpret_cast<uint4 *>(out_row)[2 * k] = make_uint4(b[0], b[1], b[2], b[3]);
                        reinterpret_cast<uint4 *>(out_row)[2 * k + 1] = make_uint4(b[4], b[5], b[6], b[7]);
                    } else if (split_ok) {
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            reinterpret_cast<float4 *>(part_row)[4 * k + e] =
                                make_float4(__uint_as_float(rr[4 * e]) * inv, __uint_as_float(rr[4 * e + 1]) * inv,
                                            __uint_as_float(rr[4 * e + 2]) * inv, __uint_as_float(rr[4 * e + 3]) * inv);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(ofree);
            if (r == 0 && (direct || split_ok)) *lse_dst = l > 0.f ? (m_used + log2f(l)) * kLn2Mla : -INFINITY;
            if (!o_ok) {
                if (lane == 0) {
                    atomicOr(&p.meta.header[kHError], DA_DEV_TIMEOUT);
                    *abort_flag = 1;
                }
                break;
            }
            ++nseg;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, TMEM_COLS);
}

// CTAs per part: one pair (value-dim halves) per query token.
int mla_ctas_per_part(int s_q) { return 2 * s_q; }
bool mla_kernel_available() { return true; }

cudaError_t launch_mla(const MlaParams &p, cudaStream_t stream, bool pdl) {
    auto kern = p.topk > 0 ? mla_decode_kernel<true> : mla_decode_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, mla::SMEM);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.num_parts, 2 * p.s_q);
    cfg.blockDim = dim3(mla::THREADS);
    cfg.dynamicSmemBytes = mla::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace da
