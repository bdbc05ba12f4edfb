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

#include <atomic>

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
constexpr int QTM = 5;                      // q slices in tensor memory (rank 0: dims [0, 320); rank 1: [256, 576))
constexpr int QSM = NSL - QTM;              // q slices in shared memory (rank 0: [320, 576); rank 1: [0, 256))
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
constexpr uint32_t Q_COL = 352;             // q slices in tensor memory: two bf16 per column (160 columns)
constexpr float RESCALE_LOG2 = 8.f;         // re-base the max when it grows by more than 2^8
static_assert(KUPT * DQ_THREADS == kChunk * KU && VUPT * DQ_THREADS == kChunk * VU, "units per chunk");
static_assert(Q_COL + QTM * 32 == TMEM_COLS, "tensor memory budget");
static_assert(SMEM <= 232448, "shared memory budget");
static_assert(OFF_V % 1024 == 0 && OFF_K % 1024 == 0 && VSLOT % 1024 == 0 && KSLOT % 1024 == 0,
              "1024-byte aligned operand tiles");
}  // namespace mla

constexpr float kLn2Mla = 0.6931471805599453f;

__device__ __forceinline__ uint32_t swz(int row, int c16) { return (uint32_t)(row * 128 + ((c16 ^ (row & 7)) << 4)); }

__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ float mul_rn(float a, float b) {
    float r;
    asm("mul.rn.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

// 16 e4m3 values times `scale`, as 16 bf16 (two 16-byte words): each code goes
// to f16 by the hardware pair conversion (exact: every e4m3 value, NaN
// included, is an f16 value), then to fp32 (exact), is multiplied by the scale
// in fp32 (one rounding of the exact product) and rounded to bf16 (nearest
// even) -- the FlashMLA page's chain (section 计算环节一: FP8 -> half -> float32,
// times the scale, -> bfloat16).
__device__ __forceinline__ void dequant16(const uint4 v, float scale, uint4 &lo, uint4 &hi) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t h01 = e4m3x2_to_f16x2((uint16_t)(w[k] & 0xFFFFu));
        const uint32_t h23 = e4m3x2_to_f16x2((uint16_t)(w[k] >> 16));
        const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&h01));
        const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&h23));
        o[2 * k] = pack_bf16(mul_rn(a.x, scale), mul_rn(a.y, scale));
        o[2 * k + 1] = pack_bf16(mul_rn(b.x, scale), mul_rn(b.y, scale));
    }
    lo = make_uint4(o[0], o[1], o[2], o[3]);
    hi = make_uint4(o[4], o[5], o[6], o[7]);
}

// Slice s of a latent row in this CTA's rings: the value slot holds slices
// [4 r, 4 r + 4), the K-only slot the other five in increasing order.
__device__ __forceinline__ int k_slot_index(int s, int r) { return r == 0 ? s - 4 : (s < 4 ? s : 4); }

// S = Q K^T for one chunk on CTA rank R: the five K-only slices first, then the
// four value slices (the q slices of this rank's value dims and one more from
// tensor memory, the others from
// shared memory); KONLY selects the K-only or the value group.
template <int R, bool KONLY>
__device__ __forceinline__ void mla_issue_qk(uint32_t tmem, uint64_t dq0, uint64_t dslot) {
    using namespace mla;
    constexpr uint32_t IDESC_QK = umma_idesc_bf16(128, 64, 0, 0);
#pragma unroll 1
    for (int k = 0; k < (KONLY ? KSL : VSL); ++k) {
        const int s = KONLY ? (R == 0 ? 4 + k : (k < 4 ? k : 8)) : 4 * R + k;
        const uint64_t db = dslot + (uint64_t)((k * SLICE) >> 4);
        // a 16-dim step advances both descriptors by 32 bytes (2 units of 16 bytes)
        // rank 0 keeps q slices 0-4 in tensor memory, rank 1 slices 4-8: either way
        // the value slices, whose MMAs wait on the last tile of a chunk, read q
        // from tensor memory
        if (R == 0 ? s < QTM : s >= NSL - QTM) {
            const uint32_t a = tmem + Q_COL + 32 * (R == 0 ? s : s - (NSL - QTM));
#pragma unroll
            for (int i = 0; i < 4; ++i)
                umma_bf16_tmem_a_w(tmem + S_COL, a + 8 * i, db + 2 * i, IDESC_QK, !(KONLY && k == 0 && i == 0));
        } else {
            const uint64_t da = dq0 + (uint64_t)(((R == 0 ? s - QTM : s) * QSLICE) >> 4);
#pragma unroll
            for (int i = 0; i < 4; ++i)
                umma_bf16_ss_w(tmem + S_COL, da + 2 * i, db + 2 * i, IDESC_QK, !(KONLY && k == 0 && i == 0));
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
        return ok && (ok = mbar_wait_warp_ool(bar, par, abort_flag, p.wait_limit_ns));
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
            umma_commit_w(&kempty[slot]);  // the K-only slot is free once these have read it
            if (!wait(&vfull[slot], par)) break;
            tc_fence_after();
            mla_issue_qk<R, false>(tmem, dq0, dv0 + (uint64_t)((slot * VSLOT) >> 4));
            umma_commit_w(sfull);
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
        // their 128-value block), 8 of RoPE values (8 bf16, copied as stored).
        // Thread dt owns NoPE column gk = 16 (1 - r) + dt % 16 (read by Q K^T only)
        // and gv = 16 r + dt % 16 (a value column) of tokens dt / 16 + 16 i (i < 4),
        // and RoPE unit 32 + dt % 8 of tokens dt / 8 + 32 j (j < 2): per chunk four
        // K-only NoPE units, four value units and two RoPE units, the same kind of
        // work on every lane. A warp's loads cover 256 contiguous bytes of two rows.
        // Within a segment the work is software-pipelined: the block-table lookups
        // of chunk c + 2, the loads of the value units of chunk c before its K-only
        // units are converted, and the loads of
        // the K-only units of chunk c + 1 before the value units of c are.
        const int dt = threadIdx.x - (1 + SM_WARPS) * 32;  // 0 .. 255
        const int gk = 16 * (1 - r) + (dt & 15), gv = 16 * r + (dt & 15), gr = dt & 7;
        const bool pf_lane = (dt & 15) == 0;               // these 16 threads cover the 64 rows of a chunk (page trace)
        auto tok_of = [&](int k) { return k < 4 ? (dt >> 4) + 16 * k : (dt >> 3) + 32 * (k - 4); };
        // Where this thread's units land in a slot: token rows dt / 16 + 16 i share
        // their swizzle (token & 7), so the offsets of the two 16-byte chunks of a
        // NoPE unit are fixed per thread (+ 2048 i for unit i); odd slices store the
        // upper chunk first (fewer bank conflicts).
        auto nope_off = [&](int g, int base, int half) -> uint32_t {
            const int tok = dt >> 4, c0 = 2 * (g & 3), swap = (g >> 2) & 1;
            return base + swz(tok, c0 + (half ^ swap));
        };
        const uint32_t k_lo = nope_off(gk, OFF_K + k_slot_index(gk >> 2, r) * SLICE, 0);
        const uint32_t k_hi = nope_off(gk, OFF_K + k_slot_index(gk >> 2, r) * SLICE, 1);
        const uint32_t v_lo = nope_off(gv, OFF_V + ((gv >> 2) - 4 * r) * SLICE, 0);
        const uint32_t v_hi = nope_off(gv, OFF_V + ((gv >> 2) - 4 * r) * SLICE, 1);
        const uint32_t r_off = OFF_K + k_slot_index(8, r) * SLICE + swz(dt >> 3, gr);  // + 4096 j
        const bool kswap = (gk >> 2) & 1, vswap = (gv >> 2) & 1;
        // 16 e4m3 codes -> 16 bf16, the first store at byte offset o_1 of shared
        // memory (chunk c0 + swap), the second at o_2; with swap the upper 8 codes
        // are converted into the first word
        auto store_nope = [&](uint32_t o_1, uint32_t o_2, bool swap, uint4 v, float sc) {
            if (swap) v = make_uint4(v.z, v.w, v.x, v.y);
            uint4 w1, w2;
            dequant16(v, sc, w1, w2);
            *reinterpret_cast<uint4 *>(smem + o_1) = w1;
            *reinterpret_cast<uint4 *>(smem + o_2) = w2;
        };
        auto load_nope = [&](int row, int g, uint4 &v, float &sc) {
            v = make_uint4(0u, 0u, 0u, 0u);
            sc = 0.f;
            if (row < 0) return;
            const uint8_t *base = p.pool + (size_t)row * ROW_BYTES;
            v = ldg_stream16(base + 16 * g);
            sc = ldg_stream4f(base + 512 + 4 * (g >> 3));
        };
        auto load_rope = [&](int row) -> uint4 {
            return row < 0 ? make_uint4(0u, 0u, 0u, 0u) : ldg_stream16(p.pool + (size_t)row * ROW_BYTES + 528 + 16 * gr);
        };
        SegWalker wk = make_walker(p.meta, rec0, rec1, p.B, p.seqlens, max_len, p.s_q, 0, p.topk);
        Seg sg;
        int cur = 0;
        bool ok = true;
        while (ok && wk.next(sg)) {
            const int n = sg.lc1 - sg.lc0;
            if (n == 0) continue;
            const int32_t *bt_row = p.block_table + (size_t)sg.b * p.max_pages;
            const int32_t *idx_row = p.indices + (size_t)sg.b * p.topk;  // sparse decode only
            // position of token `tok` of local chunk cc: dense, the token itself; sparse,
            // the position listed in that slot; -1 past the segment, past topk or
            // outside [0, L) (a zero row)
            auto position = [&](int cc, int tok) -> int {
                if (cc >= n) return -1;
                const int s = (sg.lc0 + cc) * kChunk + tok;
                int t = s;
                if (SPARSE) t = s < p.topk ? idx_row[s] : -1;
                return (t >= 0 && t < sg.L) ? t : -1;
            };
            auto page_index = [&](int t) -> int { return p.log2_page >= 0 ? t >> p.log2_page : t / p.page_size; };
            // Dense decode reads the block table through a window of 64 entries,
            // [wbase, wbase + 64), two per lane (wcur: wbase + lane, wnext: wbase + 32 +
            // lane), loaded a window ahead: page lookups are warp shuffles, without the
            // latency of a load (the table's lines leave L2 between uses under the row
            // stream). Entries past the request's pages are not read (-1).
            const int npg = (sg.L + p.page_size - 1) / p.page_size;
            auto bt_load = [&](int i) -> int { return i < npg ? bt_row[i] : -1; };
            int wbase = 0, wcur = -1, wnext = -1;
            if (!SPARSE) {
                wbase = page_index(sg.lc0 * kChunk) & ~31;
                wcur = bt_load(wbase + lane);
                wnext = bt_load(wbase + 32 + lane);
            }
            // slides the window on until index lo lies in its first half (every lane)
            auto advance = [&](int lo) {
                while (lo >= wbase + 32) {
                    wbase += 32;
                    wcur = wnext;
                    wnext = bt_load(wbase + 32 + lane);
                }
            };
            // page of position t (every lane of the warp calls it: shuffles)
            auto page_of = [&](int t) -> int {
                if (SPARSE) return t < 0 ? -1 : bt_row[page_index(t)];
                const int i = t < 0 ? wbase : page_index(t);
                const int a = __shfl_sync(0xffffffffu, wcur, (i - wbase) & 31);
                const int b = __shfl_sync(0xffffffffu, wnext, (i - wbase) & 31);
                return t < 0 ? -1 : (i - wbase < 32 ? a : b);
            };
            // pool row of position t on page pg, or -1 (a page outside the pool sets the error bit)
            auto row_of = [&](int t, int pg) -> int {
                if (t < 0) return -1;
                if (pg < 0 || pg >= p.num_pages) {
                    atomicOr(&p.meta.header[kHError], DA_DEV_BAD_PAGE);
                    p.meta.header[kHErrorDetail] = pg;
                    return -1;
                }
                return pg * p.page_size + (p.log2_page >= 0 ? t & (p.page_size - 1) : t % p.page_size);
            };
            // rows of this thread's tokens in local chunk cc, dense decode with pages
            // of at least one chunk: one page per chunk, no memory latency
            auto chunk_rows_dense = [&](int cc, int rows[6]) {
                const int t0 = (sg.lc0 + cc) * kChunk;
                const bool in = cc < n;
                const int pg = page_of(in ? t0 : -1);
                const bool pg_ok = pg >= 0 && pg < p.num_pages;
                if (in && !pg_ok) {
                    atomicOr(&p.meta.header[kHError], DA_DEV_BAD_PAGE);
                    p.meta.header[kHErrorDetail] = pg;
                }
                const int rb = pg * p.page_size + (p.log2_page >= 0 ? t0 & (p.page_size - 1) : t0 % p.page_size);
#pragma unroll
                for (int k = 0; k < 6; ++k)
                    rows[k] = (in && pg_ok && t0 + tok_of(k) < sg.L) ? rb + tok_of(k) : -1;
            };
            const bool one_page = !SPARSE && p.page_size >= kChunk;
            // Sparse decode: lane l of a warp looks up one of the 16 distinct tokens
            // the warp's lanes need (lanes l and l + 16 the same one) and the rows
            // reach the lanes that need them by shuffles: one position, page and row
            // per lane and chunk, not six (215 vs 277 us per top-k 2048 call). Dense
            // decode with pages shorter than a chunk keeps one lookup per token and
            // thread (its pages come from the block-table window by shuffles anyway;
            // the shared form there cost the dense build 7 % on one-page chunks).
            const int lk = lane & 15, dw = dt >> 5;
            const int wtok = lk < 8 ? 2 * dw + (lk & 1) + 16 * (lk >> 1) : 4 * dw + ((lk - 8) & 3) + 32 * ((lk - 8) >> 2);
            auto src_of = [&](int k) { return k < 4 ? 2 * k + (lane >> 4) : 8 + ((lane >> 3) & 3) + 4 * (k - 4); };
            auto spread = [&](int r, int(&rows)[6]) {
#pragma unroll
                for (int k = 0; k < 6; ++k) rows[k] = __shfl_sync(0xffffffffu, r, src_of(k));
            };
#ifdef DA_PAGE_TRACE
            // test build: the trace value of this lane's token, handed to the lanes that record it
            auto trace_spread = [&](int t, int pg, int idx) {
                const int tv = t >= 0 ? pg * p.page_size + t % p.page_size : -2;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int v = __shfl_sync(0xffffffffu, tv, src_of(k));
                    if (p.page_trace && blockIdx.y == 0 && pf_lane && idx < p.page_trace_cap)
                        p.page_trace[((size_t)part * p.page_trace_cap + idx) * kChunk + tok_of(k)] = v;
                }
            };
#endif
            int pos2 = -1, pos2a[6], row0[6], row1[6];  // positions in chunk c + 2: this lane's (sparse), per token (dense)
            // prologue: rows of chunks 0 and 1, positions of chunk 2
            if (one_page) {
                chunk_rows_dense(0, row0);
                chunk_rows_dense(1, row1);
#ifdef DA_PAGE_TRACE
                if (p.page_trace && blockIdx.y == 0 && pf_lane) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        if (cur < p.page_trace_cap)
                            p.page_trace[((size_t)part * p.page_trace_cap + cur) * kChunk + tok_of(k)] =
                                row0[k] >= 0 ? row0[k] : -2;
                        if (n > 1 && cur + 1 < p.page_trace_cap)
                            p.page_trace[((size_t)part * p.page_trace_cap + cur + 1) * kChunk + tok_of(k)] =
                                row1[k] >= 0 ? row1[k] : -2;
                    }
                }
#endif
            } else if (SPARSE) {
                const int t0 = position(0, wtok), t1 = position(1, wtok);
                const int pg0 = page_of(t0), pg1 = page_of(t1);
                spread(row_of(t0, pg0), row0);
                spread(row_of(t1, pg1), row1);
                pos2 = position(2, wtok);
#ifdef DA_PAGE_TRACE
                trace_spread(t0, pg0, cur);
                if (n > 1) trace_spread(t1, pg1, cur + 1);
#endif
            } else
#pragma unroll
            for (int k = 0; k < 6; ++k) {
                const int t0 = position(0, tok_of(k)), t1 = position(1, tok_of(k));
                const int pg0 = page_of(t0), pg1 = page_of(t1);
                row0[k] = row_of(t0, pg0);
                row1[k] = row_of(t1, pg1);
                pos2a[k] = position(2, tok_of(k));
#ifdef DA_PAGE_TRACE
                if (p.page_trace && blockIdx.y == 0 && pf_lane && k < 4) {
                    if (cur < p.page_trace_cap)
                        p.page_trace[((size_t)part * p.page_trace_cap + cur) * kChunk + tok_of(k)] =
                            t0 >= 0 ? pg0 * p.page_size + t0 % p.page_size : -2;
                    if (n > 1 && cur + 1 < p.page_trace_cap)
                        p.page_trace[((size_t)part * p.page_trace_cap + cur + 1) * kChunk + tok_of(k)] =
                            t1 >= 0 ? pg1 * p.page_size + t1 % p.page_size : -2;
                }
#endif
            }
            uint4 kn[4], kr[2];
            float ksc[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) load_nope(row0[i], gk, kn[i], ksc[i]);
#pragma unroll
            for (int j = 0; j < 2; ++j) kr[j] = load_rope(row0[4 + j]);
            for (int c = 0; c < n && ok; ++c, ++cur) {
                const int slot = cur % NR;
                const uint32_t par = ((cur / NR) & 1) ^ 1;
                // a. block-table lookups of chunk c + 2
                if (!SPARSE && c + 2 < n) advance(page_index((sg.lc0 + c + 2) * kChunk));
                int pg2 = -1, pg2a[6];
                if (!one_page) {
                    if (SPARSE) {
                        pg2 = page_of(pos2);
                    } else {
#pragma unroll
                        for (int k = 0; k < 6; ++k) pg2a[k] = page_of(pos2a[k]);
                    }
                }
                // b. loads of the value units of chunk c
                uint4 vn[4];
                float vsc[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) load_nope(row0[i], gv, vn[i], vsc[i]);
                // c. the K-only units of chunk c, once Q K^T of the chunk two back has
                // read the slot
                if (!(ok = mbar_wait_warp_ool(&kempty[slot], par, abort_flag, p.wait_limit_ns))) break;
                const uint32_t ks = slot * KSLOT;
#pragma unroll
                for (int i = 0; i < 4; ++i) store_nope(k_lo + ks + 2048 * i, k_hi + ks + 2048 * i, kswap, kn[i], ksc[i]);
#pragma unroll
                for (int j = 0; j < 2; ++j) *reinterpret_cast<uint4 *>(smem + r_off + ks + 4096 * j) = kr[j];
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&kfull[slot]);
                // d. rows of chunk c + 2 (into L2 now), positions of chunk c + 3
                int row2[6];
                if (one_page) {
                    chunk_rows_dense(c + 2, row2);
#ifdef DA_PAGE_TRACE
                    if (p.page_trace && blockIdx.y == 0 && pf_lane && c + 2 < n && cur + 2 < p.page_trace_cap) {
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            p.page_trace[((size_t)part * p.page_trace_cap + cur + 2) * kChunk + tok_of(k)] =
                                row2[k] >= 0 ? row2[k] : -2;
                    }
#endif
                } else if (SPARSE) {
                    spread(row_of(pos2, pg2), row2);
#ifdef DA_PAGE_TRACE
                    if (c + 2 < n) trace_spread(pos2, pg2, cur + 2);
#endif
                } else
#pragma unroll
                for (int k = 0; k < 6; ++k) {
                    row2[k] = row_of(pos2a[k], pg2a[k]);
#ifdef DA_PAGE_TRACE
                    if (p.page_trace && blockIdx.y == 0 && pf_lane && k < 4 && c + 2 < n && cur + 2 < p.page_trace_cap)
                        p.page_trace[((size_t)part * p.page_trace_cap + cur + 2) * kChunk + tok_of(k)] =
                            pos2a[k] >= 0 ? pg2a[k] * p.page_size + pos2a[k] % p.page_size : -2;
#endif
                }
                if (!one_page) {
                    if (SPARSE) {
                        pos2 = position(c + 3, wtok);
                    } else {
#pragma unroll
                        for (int k = 0; k < 6; ++k) pos2a[k] = position(c + 3, tok_of(k));
                    }
                }
                // e. loads of the K-only units of chunk c + 1
#pragma unroll
                for (int i = 0; i < 4; ++i) load_nope(row1[i], gk, kn[i], ksc[i]);
#pragma unroll
                for (int j = 0; j < 2; ++j) kr[j] = load_rope(row1[4 + j]);
                // f. the value units of chunk c, once P V of the chunk two back has read the slot
                if (!(ok = mbar_wait_warp_ool(&vempty[slot], par, abort_flag, p.wait_limit_ns))) break;
                const uint32_t vs = slot * VSLOT;
#pragma unroll
                for (int i = 0; i < 4; ++i) store_nope(v_lo + vs + 2048 * i, v_hi + vs + 2048 * i, vswap, vn[i], vsc[i]);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&vfull[slot]);
#pragma unroll
                for (int k = 0; k < 6; ++k) {
                    row0[k] = row1[k];
                    row1[k] = row2[k];
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
            ok = mbar_wait_warp_ool(stall, 0, abort_flag, p.wait_limit_ns);
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
            // this head's q row of query token `draft`: five slices into tensor memory
            // (rank 0: dims [0, 320), rank 1: [256, 576)), the other four into shared
            // memory (rank 0: [320, 576), rank 1: [0, 256)); qs counts 16-byte chunks
            if (!(ok = mbar_wait_warp_ool(qfree, (nseg & 1) ^ 1, abort_flag, p.wait_limit_ns))) break;
            {
                const uint4 *qs = reinterpret_cast<const uint4 *>(reinterpret_cast<const __nv_bfloat16 *>(p.q) +
                                                                 ((size_t)sg.b * rows + draft * HQ + head) * DQK);
                const int tm0 = r == 0 ? 0 : 32, sm0 = r == 0 ? 40 : 0;
#pragma unroll 1
                for (int j = 0; j < 10; ++j) {  // 32 dims = 16 columns per store
                    uint32_t rr[16];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint4 v = qs[tm0 + 4 * j + k];
                        rr[4 * k] = v.x;
                        rr[4 * k + 1] = v.y;
                        rr[4 * k + 2] = v.z;
                        rr[4 * k + 3] = v.w;
                    }
                    tmem_st16(trow + Q_COL + 16 * j, rr);
                }
#pragma unroll 4
                for (int k = 0; k < QSM * 8; ++k)  // 16-byte chunk k % 8 of slice k / 8
                    *reinterpret_cast<uint4 *>(smem + OFF_Q + (k >> 3) * QSLICE + swz(head, k & 7)) = qs[sm0 + k];
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
                bool w_ok = mbar_wait_warp_ool(sfull, cur & 1, abort_flag, p.wait_limit_ns);
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
                // raw scores of the tokens this query token does not see become -inf
                if (SPARSE) {
                    // sparse: slot e counts when it lies before topk and lists a position in
                    // [0, L); the warp's ballots give the 64 bits (vm0: slots 0-31, vm1: 32-63)
                    const uint32_t vm0 = __ballot_sync(0xffffffffu, t0 >= 0 && t0 < sg.L);
                    const uint32_t vm1 = __ballot_sync(0xffffffffu, t1 >= 0 && t1 < sg.L);
#pragma unroll
                    for (int e = 0; e < 64; ++e)
                        if (!(((e < 32 ? vm0 >> e : vm1 >> (e - 32)) & 1u))) s[e] = -INFINITY;
                } else {
                    const int nvalid = L_vis - cbase;  // tokens of this chunk the query token sees
                    if (nvalid < kChunk) {             // the same for every thread of the CTA
#pragma unroll
                        for (int e = 0; e < 64; ++e)
                            if (e >= nvalid) s[e] = -INFINITY;
                    }
                }
                // sl2 = sigma log2(e) > 0: the max of the scaled scores is sl2 times the raw max
                float m1[22];
#pragma unroll
                for (int e = 0; e < 21; ++e) m1[e] = fmax3(s[3 * e], s[3 * e + 1], s[3 * e + 2]);
                m1[21] = s[63];
                float m2[8];
#pragma unroll
                for (int e = 0; e < 7; ++e) m2[e] = fmax3(m1[3 * e], m1[3 * e + 1], m1[3 * e + 2]);
                m2[7] = m1[21];
                const float mx = fmax3(fmax3(m2[0], m2[1], m2[2]), fmax3(m2[3], m2[4], m2[5]), fmaxf(m2[6], m2[7])) * sl2;
                // P's columns and O are free once the previous chunk's P V has completed
                w_ok = w_ok && mbar_wait_warp_ool(pfree, (cur & 1) ^ 1, abort_flag, p.wait_limit_ns);
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
                    const float p0 = ex2(fmaf(s[2 * e], sl2, -base)), p1 = ex2(fmaf(s[2 * e + 1], sl2, -base));
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
            const bool o_ok = mbar_wait_warp_ool(ofull, nseg & 1, abort_flag, p.wait_limit_ns);
            tc_fence_after();
            if (o_ok) {
                // (a NaN sum -- a NaN code in a row -- stays NaN rather than reading as empty)
                const float inv = !(l <= 0.f) ? 1.f / l : 0.f;
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
            if (r == 0 && (direct || split_ok)) *lse_dst = !(l <= 0.f) ? (m_used + log2f(l)) * kLn2Mla : -INFINITY;
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

// CTAs per part: one pair (value-dim halves) per query token. They form one
// thread-block cluster, so they run on one GPC, in front of one L2 partition:
// the rows the first CTA reads from HBM are L2 hits for the others.
int mla_ctas_per_part(int s_q) { return 2 * s_q; }
bool mla_kernel_available() { return true; }

// Parts that can run at once: clusters of 2 s_q CTAs, one CTA per SM.
int mla_max_parts(int s_q) {
    static std::atomic<int> cached[64][kMaxSqMla + 1];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64 || s_q < 1 || s_q > kMaxSqMla) return 0;
    if (const int c = cached[dev][s_q].load(std::memory_order_relaxed)) return c;
    if (cudaFuncSetAttribute(mla_decode_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, mla::SMEM) !=
        cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1024, 2 * s_q);
    cfg.blockDim = dim3(mla::THREADS);
    cfg.dynamicSmemBytes = mla::SMEM;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 2 * s_q;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, mla_decode_kernel<false>, &cfg) != cudaSuccess) return 0;
    cached[dev][s_q].store(n, std::memory_order_relaxed);
    return n;
}

cudaError_t launch_mla(const MlaParams &p, cudaStream_t stream, bool pdl) {
    auto kern = p.topk > 0 ? mla_decode_kernel<true> : mla_decode_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, mla::SMEM);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.num_parts, 2 * p.s_q);
    cfg.blockDim = dim3(mla::THREADS);
    cfg.dynamicSmemBytes = mla::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 2 * p.s_q;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace da
