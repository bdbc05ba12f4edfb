// Split-KV decode kernel for grouped-query attention with G = 8 query heads
// per KV head (bf16 KV with D = 64 / 128, e4m3 KV with D = 128).
//
// One CTA per (part, KV head). A part is a list of (request, chunk range)
// segments from the scheduling metadata; a chunk is 64 tokens.
//
// Data path (XQA page "TensorRT-LLM 源码完全拆解(二十九)"):
//  * page gather: one 4-D tensor map describes the whole pool
//    [num_pages][P][H_kv][D]; the page id is the outermost TMA coordinate
//    (section "Hopper:一次 TMA 只搬一个页"). Page ids are read by the producer
//    warp 32 at a time, one per lane, and broadcast with shuffles, ahead of use.
//  * K/V streaming: a producer warp fills an NS-stage ring of shared-memory
//    stages (K tile + V tile of one chunk) with TMA; full/empty mbarriers hand
//    stages to the consumer warps. Loads carry an L2 evict-first hint
//    (FlashMLA page, section "数据加载": KV is streamed once).
//  * the G query rows of one KV head stay in registers for the whole part, so
//    each KV byte is read from HBM once per group (XQA page, section
//    "GQA 的组内复用").
//  * products: the KV tile sits on the M side of a 16x8x16 warp MMA and the
//    G = 8 query heads on the N side -- the SWAP_AB orientation of the XQA page
//    (section "SWAP_AB:把 K 放在 A 位"): S^T = K Q^T, O^T += V^T P^T. With G = 8
//    the N = 8 side is exactly filled. P goes from the S accumulator to the PV
//    operand through movmatrix (8x8 transpose in registers).
//  * online softmax (attention pipeline page, section 三): running max m,
//    running sum l, rescale alpha = 2^(m_old - m_new), exponentials by exp2
//    with log2(e) folded into the score scale (same page, section 一).
//  * FP8 KV: e4m3 stays e4m3 in shared memory and is widened to f16 in
//    registers right before the MMA (XQA page, section "为什么不在搬入 SMEM 时就转换"),
//    two values per cvt; the per-tensor scales are folded into the score scale
//    (k_scale) and into the output (v_scale) (same page, section
//    "Hopper 路径上 V 不做显式反量化").
//  * several query tokens per request (linear speculative-decoding
//    verification, XQA page, section "投机解码:XQA 的第二个工作负载"): the
//    s_q draft tokens' G heads become NQ n8 tiles on the N side, so every K/V
//    fragment loaded from shared memory feeds NQ MMAs (three or four tokens:
//    two warps share each chunk, two tokens each); draft token j sees the
//    tokens [0, L - s_q + j] (a chain: each draft token sees the ones before it).
//  * every consumer warp takes whole chunks (round robin) as four independent
//    16-token tiles, so its MMA chains and shuffle reductions interleave, and
//    keeps its own (m, l, O) state; at the end of a segment the warps' states are merged
//    through shared memory in a fixed order, and the segment's result is
//    written either as the final bf16 output (request has one split) or as a
//    float32 partial plus its lse for the combine kernel.
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "decode_attn.h"
#include "segwalk.cuh"

namespace da {

constexpr float kLn2 = 0.6931471805599453f;

template <int D, bool FP8, int NQ, int WPC>
struct GqaCfg {
    static constexpr int G = 8;
    static constexpr int ES = FP8 ? 1 : 2;
    static constexpr int ROW = D * ES;       // bytes of one token's head
    static constexpr int NX = ROW / 128;     // 128-byte halves of a row
    static constexpr int TILE = kChunk * ROW;
    static constexpr int STAGE = 2 * TILE;   // K and V of one chunk
    // consumer warps and ring stages. A chunk goes to a group of WPC warps
    // (round robin over the NG groups; each warp of the group holds NQ of the
    // query tokens). NS is a multiple of NG so that stage s is always consumed
    // by group s % NG: a warp then waits on the phases of a stage one after
    // the other, and never on a phase two ahead of the barrier's current one
    // (whose parity would alias an already completed phase).
    // With several query tokens (NQ > 1) a warp holds NQ times the state and
    // the kernel runs one CTA per SM: 6 or 7 consumer warps keep at most two
    // warps on each SM sub-partition, so a thread may use up to 255 registers.
    static constexpr int NCW = WPC == 4 ? 8
                               : WPC > 1 ? 6 : (NQ > 1 ? (D == 128 && !FP8 ? 6 : 7) : (FP8 ? 10 : (D == 64 ? 5 : 6)));
    static constexpr int NG = NCW / WPC;
    // The D = 64 build for three or four query tokens runs two CTAs per SM
    // (four stages each, at most 96 registers a thread): its MMA -> softmax ->
    // MMA chain is latency-bound, and a second CTA's chunks fill the gaps
    // (69.9 vs 80.5 us per call on the four-token workload).
    static constexpr bool TWO_PER_SM = D == 64 && !FP8 && WPC == 4;
    static constexpr int NS = TWO_PER_SM ? 4 : (NCW == 5 ? 5 : NCW);
    static_assert(NCW % WPC == 0 && NS % NG == 0, "stage ownership must be fixed per warp group");
    static constexpr int THREADS = (NCW + 1) * 32;
    static constexpr int MT = D / 16;
    static constexpr int KS = D / 16;
    static constexpr int UPAD = D + 4;
    static constexpr int OFF_U = NS * STAGE;
    static constexpr int OFF_M = OFF_U + NCW * G * UPAD * 4;
    static constexpr int OFF_L = OFF_M + NCW * G * 4;
    static constexpr int OFF_W = OFF_L + NCW * G * 4;
    static constexpr int OFF_FIN = OFF_W + NCW * G * 4;
    static constexpr int OFF_BAR = (OFF_FIN + 4 * G * 4 + 7) / 8 * 8;
    static constexpr int OFF_FLAG = OFF_BAR + 2 * NS * 8;
    static constexpr int SMEM = OFF_FLAG + 16 + 1024;  // + alignment slack
    static constexpr int MIN_BLOCKS = ((D == 64 && !FP8 && NQ == 1 && WPC == 1) || TWO_PER_SM) ? 2 : 1;
    static_assert(ROW % 128 == 0, "rows must be whole 128-byte boxes");
    static_assert(!FP8 || NX == 1, "fp8 path expects one 128-byte box per row");
};

// Split merge inside a cluster (fixed split count S <= 8): the S CTAs of a
// (request, KV head) form one thread-block cluster; each has left its split's
// normalised partial (o, lse) for every row in its own shared memory. After
// a cluster barrier (arrive releases this CTA's partial, wait acquires the
// others'; a CTA's threads reaching it have also started, so no earlier
// barrier is needed before reading another CTA's memory), CTA rank r merges
// dims [floor(r D / S), floor((r + 1) D / S)) of every row from distributed
// shared memory by the rule of the combine kernel (lse = M + ln sum
// e^(lse_s - M), out = sum e^(lse_s - lse) o_s, splits in index order), adds
// the attention sink and writes out and lse. A second cluster barrier keeps
// every CTA resident until all have finished reading its memory. Called by
// the consumer warps only; the producer warp has exited by then (the barrier
// does not wait for exited threads).
struct MergeArgs {
    void *out;
    float *lse;
    const float *sinks;
    int s_q, H_q, S;
};

// Out of line (its registers stay out of the main loop's allocation); the
// kernel parameters it needs come by value.
template <int D>
__device__ __noinline__ void cluster_merge(const MergeArgs p, float *xo, float *xl, int b, int h, bool aborted) {
    constexpr int G = 8;
    constexpr float kLog2e = 1.4426950408889634f;
    const int nthr = blockDim.x - 32;  // consumer threads
    const int ctid = threadIdx.x;
    const int S = p.S;
    const int rows_cta = p.s_q * G;
    const uint32_t rank = cluster_ctarank();
    const int d0 = (int)rank * D / S, dpc = ((int)rank + 1) * D / S - d0;  // this CTA's dims
    // whole warps the merge needs; the others leave now (their writes are
    // ordered before the remaining threads' release by the CTA barrier that
    // ended the segment, and exited threads do not hold up the cluster barrier)
    const int keep = min(nthr, (rows_cta * dpc + 31) / 32 * 32);
    if (aborted || b < 0) {
        // no valid partial: weight 0 for every row
        for (int r = ctid; r < rows_cta; r += nthr) xl[r] = -INFINITY;
    }
    if (ctid >= keep) return;
    __syncwarp();          // the cluster barrier instructions below are warp-aligned
    cluster_arrive_all();  // this thread's share of the partial is written (release)
    cluster_wait_all();    // every split's partial is visible (acquire)
    if (b >= 0) {
        const uint32_t xo_s = smem_u32(xo), xl_s = smem_u32(xl);
        const size_t rows = (size_t)p.s_q * p.H_q;
        for (int idx = ctid; idx < rows_cta * dpc; idx += keep) {
            const int r = idx / dpc, d = d0 + idx % dpc;
            // every split's lse and value in one round of loads
            float ls[8], ov[8];
            float M = -INFINITY;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                ls[q] = q < S ? ld_cluster_f32(mapa_shared(xl_s + 4u * r, (uint32_t)q)) : -INFINITY;
                ov[q] = q < S ? ld_cluster_f32(mapa_shared(xo_s + 4u * ((uint32_t)r * D + d), (uint32_t)q)) : 0.f;
            }
#pragma unroll
            for (int q = 0; q < 8; ++q) M = fmax_nan(M, ls[q]);
            float acc = 0.f, lse_v = -INFINITY;
            if (M != -INFINITY) {
                float Z = 0.f;
#pragma unroll
                for (int q = 0; q < 8; ++q) Z += ls[q] == -INFINITY ? 0.f : ex2((ls[q] - M) * kLog2e);
                lse_v = M + logf(Z);
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    if (ls[q] == -INFINITY) continue;  // empty split, or a slot past S (its value unused)
                    acc += ex2((ls[q] - lse_v) * kLog2e) * ov[q];
                }
            }
            const int jj = r / G, g = r % G;
            if (p.sinks != nullptr) {
                const float tot = log_add_exp(lse_v, p.sinks[h * G + g]);
                acc *= (lse_v == -INFINITY) ? 0.f : expf(lse_v - tot);
                lse_v = tot;
            }
            const size_t orow = (size_t)b * rows + (size_t)jj * p.H_q + (size_t)h * G + g;
            reinterpret_cast<__nv_bfloat16 *>(p.out)[orow * D + d] = __float2bfloat16_rn(acc);
            if (rank == 0 && idx % dpc == 0) p.lse[orow] = lse_v;
        }
    }
    // this thread's loads from the other splits are done; wait until every
    // split is done with this one's memory before it exits
    __syncwarp();
    cluster_arrive_all();
    cluster_wait_all();
}

// NQ x WPC: query tokens per request the kernel is compiled for (s_q <=
// NQ * WPC; warp w of a chunk's group holds tokens [(w % WPC) NQ, (w % WPC + 1)
// NQ), and tokens j >= s_q are zero rows that are never written). WIN: built
// with sliding window support (without it, p.window must be 0).
template <int D, bool FP8, int NQ, int WPC, bool WIN>
__global__ void __launch_bounds__(GqaCfg<D, FP8, NQ, WPC>::THREADS, GqaCfg<D, FP8, NQ, WPC>::MIN_BLOCKS)
    gqa_decode_kernel(const __grid_constant__ CUtensorMap tm_kv, const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ GqaParams p) {
    using C = GqaCfg<D, FP8, NQ, WPC>;
    // 256-byte rows land half-major in the builds with a window or several
    // query tokens (the host builds the tensor maps to match: p.half_major)
    constexpr bool HM = WIN && C::NX > 1;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float *sm_u = reinterpret_cast<float *>(smem + C::OFF_U);
    float *sm_m = reinterpret_cast<float *>(smem + C::OFF_M);
    float *sm_l = reinterpret_cast<float *>(smem + C::OFF_L);
    float *sm_w = reinterpret_cast<float *>(smem + C::OFF_W);
    float *sm_fin = reinterpret_cast<float *>(smem + C::OFF_FIN);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    uint64_t *empty = full + C::NS;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_FLAG);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int part = blockIdx.x, h = blockIdx.y;

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::NS; ++i) {
            mbar_init(&full[i], p.boxes_per_chunk);  // one arrival per producer lane
            mbar_init(&empty[i], WPC);  // every warp of the chunk's group
        }
        *abort_flag = 0;
#ifdef DA_PAGE_TRACE
        mbar_init(reinterpret_cast<uint64_t *>(smem + C::OFF_FLAG + 8), 1);  // never arrived at
#endif
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    if (warp == C::NCW && lane == 0) {
        prefetch_tmap(&tm_kv);
        if (!p.kv_combined) prefetch_tmap(&tm_v);
    }
    __syncthreads();
    pdl_wait();
    pdl_launch_dependents();

    // the part record and the header are independent loads: issue both, then check
    const int4 rec0 = p.meta.parts[2 * part];
    const int4 rec1 = p.meta.parts[2 * part + 1];
    {
        const int32_t *hd = p.meta.header;
        const bool ok = meta_header_ok(load_meta_header(hd), p.B, p.H_kv, p.G, p.splits, p.num_parts, p.s_q,
                                       p.window, 0) &
                        ((int)gridDim.x == p.num_parts);
        if (!ok) {
            if (threadIdx.x == 0) atomicOr(&p.meta.header[kHError], DA_DEV_META_MISMATCH);
            return;
        }
    }
    const int max_len = p.max_pages * p.page_size;
    // parts beyond the header's count are never read: the check above ties gridDim.x to it

    if (warp == C::NCW) {
        // ------------------------------------------------------------ producer
        // Lane j < boxes_per_chunk owns box j of every chunk: one TMA per page
        // brings that page's K and V rows of head h (both pools, both 128-byte
        // halves of a row, through one 5-D tensor map; when the two pools are
        // too far apart for one map, two 4-D maps and two copies). Each lane keeps the
        // page ids of its next four chunks in registers, loaded four chunks
        // ahead, arrives on the chunk's full barrier with its own byte count
        // and issues its own copy -- no shuffles, no load latency in the loop.
        const int nb = p.boxes_per_chunk, bt = p.box_tokens, P = p.page_size;
        if (lane >= nb) return;
        const uint64_t pol = policy_evict_first();
        const uint32_t box_bytes = 2u * bt * C::NX * 128u;
        SegWalker wk = make_walker(p.meta, rec0, rec1, p.B, p.seqlens, max_len, p.s_q, WIN ? p.window : 0, 0);
        int i = 0;
        bool aborted = false;
        Seg sg;
        while (!aborted && wk.next(sg)) {
            const int lc0 = sg.lc0, lc1 = sg.lc1, L = sg.L;
            if (lc0 == lc1) continue;
            const int32_t *bt_row = p.block_table + (size_t)sg.b * p.max_pages;
            // local chunk lc is the request's chunk fc + lc (fc > 0 only with a sliding window)
            const int start = WIN ? window_start(L, p.s_q, p.window) : 0;
            const int fc = start / kChunk;
            // page id of this lane's box in chunk lc, or -2 when the box lies past
            // the sequence or wholly before the window (its page is not read)
            auto id_of = [&](int lc) -> int {
                const int tok = (fc + lc) * kChunk + lane * bt;
                return (lc < lc1 && tok < L && tok + bt > start) ? bt_row[tok / P] : -2;
            };
            int ring[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) ring[k] = id_of(lc0 + k);
            for (int lc = lc0; lc < lc1 && !aborted; lc += 4) {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    if (lc + k >= lc1) break;
                    int pg = ring[k];
                    ring[k] = id_of(lc + k + 4);
                    const int stage = i % C::NS;
                    if (!mbar_wait_bounded(&empty[stage], ((i / C::NS) & 1) ^ 1, abort_flag, p.wait_limit_ns)) {
                        atomicOr(&p.meta.header[kHError], DA_DEV_TIMEOUT);
                        *abort_flag = 1;
                        aborted = true;
                        break;
                    }
                    if (pg != -2 && (pg < 0 || pg >= p.num_pages)) {
                        atomicOr(&p.meta.header[kHError], DA_DEV_BAD_PAGE);
                        p.meta.header[kHErrorDetail] = pg;
                        pg = -2;  // skipped: its rows keep stale bytes
                    }
#ifdef DA_PAGE_TRACE
                    if (p.page_trace && i < p.page_trace_cap) {
                        const int tok = (fc + lc + k) * kChunk + lane * bt;
                        const size_t unit = (size_t)blockIdx.x * gridDim.y + blockIdx.y;
                        p.page_trace[(unit * p.page_trace_cap + i) * nb + lane] =
                            pg == -2 ? -2 : pg * P + ((P > kChunk) ? (tok % P) : 0);
                    }
#endif
                    mbar_arrive_expect_tx(&full[stage], pg == -2 ? 0u : box_bytes);
                    if (pg != -2) {
                        const int tok = (fc + lc + k) * kChunk + lane * bt;
                        const int in_page = (P > kChunk) ? (tok % P) : 0;
                        uint8_t *st = smem + (size_t)stage * C::STAGE + lane * box_bytes;
                        if (p.kv_combined) {
                            if constexpr (HM)
                                tma_load_5d(st, &tm_kv, &full[stage], 0, pg * P + in_page, 0, h, 0, pol);
                            else
                                tma_load_5d(st, &tm_kv, &full[stage], 0, 0, h, pg * P + in_page, 0, pol);
                        } else {  // K map in tm_kv, V map in tm_v, same box image
                            if constexpr (HM) {
                                tma_load_4d(st, &tm_kv, &full[stage], 0, pg * P + in_page, 0, h, pol);
                                tma_load_4d(st + box_bytes / 2, &tm_v, &full[stage], 0, pg * P + in_page, 0, h, pol);
                            } else {
                                tma_load_4d(st, &tm_kv, &full[stage], 0, 0, h, pg * P + in_page, pol);
                                tma_load_4d(st + box_bytes / 2, &tm_v, &full[stage], 0, 0, h, pg * P + in_page, pol);
                            }
                        }
                    }
                    ++i;
                }
            }
        }
        if (aborted) {
            // let copies already in flight land before the CTA exits (ignoring the abort flag)
            for (int k = max(0, i - C::NS); k < i; ++k) mbar_wait_timed(&full[k % C::NS], (k / C::NS) & 1, 100000000ull);
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int r8 = lane >> 2, c4 = lane & 3;
    const int grp = warp / WPC, jo = (warp % WPC) * NQ;  // this warp's group and first query token
    const int lrow = lane & 7, lmat = lane >> 3;
    const int ctid = threadIdx.x;  // 0 .. NCW*32-1
    const float kscale = FP8 ? p.k_scale[h] : 1.f;
    const float vscale = FP8 ? p.v_scale[h] : 1.f;
    const float sl2 = p.scale_log2 * kscale;
    // Stage layout: box j (tokens [j*bt, (j+1)*bt)) at j*box_bytes holds one
    // pool's rows, then the other's (p.kv_swap tells which pool comes first).
    // With bt >= 8 every box and half starts on a 1024-byte boundary. Rows of
    // 256 bytes (NX = 2) are laid out token-major, [token][half][128 B], in the
    // lean one-token build: each row is one 256-byte read, and the 128-byte
    // swizzle key of token t, half x is (2t + x) & 7 (a 2-way bank conflict on
    // ldmatrix, which that HBM-bound build does not feel); and half-major,
    // [half][token][128 B], in the builds with several query tokens or a
    // window, which do more arithmetic per byte: key t & 7, no conflict.
    // With NX = 1 the two are the same.
    const int bt = p.box_tokens, lbt = p.log2_box_tokens;
    const uint32_t half_bytes = (uint32_t)bt * C::NX * 128u;   // one pool's part of a box
    const uint32_t xstride = HM ? (uint32_t)bt * 128u : 128u;  // half 0 -> half 1 of a row
    const uint32_t k_half = p.kv_swap ? half_bytes : 0u, v_half = p.kv_swap ? 0u : half_bytes;
    auto row_of = [&](int tok) -> uint32_t {  // half 0 of token tok's row
        return HM ? (uint32_t)((tok >> lbt) * 2 * bt * C::NX + (tok & (bt - 1))) * 128u
                  : (uint32_t)((tok >> lbt) * 2 * bt + (tok & (bt - 1))) * (C::NX * 128u);
    };
    auto key_of = [&](int tok, int x) -> int { return HM ? (tok & 7) : ((tok * C::NX + x) & 7); };
    // tokens this lane addresses in ldmatrix: tile t, 8-row half sel
    uint32_t rk[4], rv[4];
    int keyk[4], keyv[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        const int tk = 16 * t + lrow + (lmat & 1) * 8;                      // K rows (QK), V rows (fp8 PV)
        const int tv = FP8 ? tk : 16 * t + lrow + (lmat >> 1) * 8;          // V rows (bf16 PV)
        rk[t] = row_of(tk) + k_half;
        rv[t] = row_of(tv) + v_half;
        keyk[t] = key_of(tk, 0);  // the key of half x is key_of(t, x): + x when token-major
        keyv[t] = key_of(tv, 0);
    }

    SegWalker wk = make_walker(p.meta, rec0, rec1, p.B, p.seqlens, max_len, p.s_q, WIN ? p.window : 0, 0);
    int i = 0;
    Seg sg;
    int merge_b = -1;  // cluster merge: the request of this CTA's (single) segment
    // cluster merge: this split's normalised partial [rows][D] and lse [rows],
    // rows = s_q * G, in the stage memory (idle once the segment is done)
    float *xo = reinterpret_cast<float *>(smem);
    float *xl = xo + (size_t)p.s_q * C::G * D;
    while (wk.next(sg)) {
        const int sb = sg.b, ss = sg.s, lc0 = sg.lc0, lc1 = sg.lc1, L = sg.L;
        merge_b = sb;
        // query fragments (B operand, n = query head r8 of this group), one
        // n8 tile per query token of the request; q is [B][s_q][H_q][D]
        uint32_t qf[C::KS][NQ][2];
#pragma unroll
        for (int j = 0; j < NQ; ++j) {
            if (jo + j >= p.s_q) {
#pragma unroll
                for (int ks = 0; ks < C::KS; ++ks) qf[ks][j][0] = qf[ks][j][1] = 0u;
                continue;
            }
            const size_t qrow = (((size_t)sb * p.s_q + jo + j) * p.H_q + (size_t)h * C::G + r8) * D;
            if constexpr (!FP8) {
                const uint32_t *q32 = reinterpret_cast<const uint32_t *>(
                    reinterpret_cast<const __nv_bfloat16 *>(p.q) + qrow);
#pragma unroll
                for (int ks = 0; ks < C::KS; ++ks) {
                    qf[ks][j][0] = q32[ks * 8 + c4];
                    qf[ks][j][1] = q32[ks * 8 + 4 + c4];
                }
            } else {
                const __nv_bfloat16 *qb = reinterpret_cast<const __nv_bfloat16 *>(p.q) + qrow;
#pragma unroll
                for (int ks = 0; ks < C::KS; ++ks) {
                    const uint2 v = *reinterpret_cast<const uint2 *>(qb + ks * 16 + c4 * 4);
                    const __nv_bfloat162 lo = *reinterpret_cast<const __nv_bfloat162 *>(&v.x);
                    const __nv_bfloat162 hi = *reinterpret_cast<const __nv_bfloat162 *>(&v.y);
                    qf[ks][j][0] = pack_f16(__low2float(lo), __high2float(lo));
                    qf[ks][j][1] = pack_f16(__low2float(hi), __high2float(hi));
                }
            }
        }
        // draft token j sees the first L - s_q + 1 + j tokens (the last `window`
        // of them with a sliding window); local chunk lc is the request's chunk fc + lc
        const int L_first = L - p.s_q + 1;
        const int start = WIN ? window_start(L, p.s_q, p.window) : 0;
        const int fc = start / kChunk;
        float m0[NQ], m1[NQ], l0[NQ], l1[NQ];
        float acc[C::MT][NQ][4];
#pragma unroll
        for (int j = 0; j < NQ; ++j) {
            m0[j] = m1[j] = -INFINITY;
            l0[j] = l1[j] = 0.f;
#pragma unroll
            for (int mt = 0; mt < C::MT; ++mt) acc[mt][j][0] = acc[mt][j][1] = acc[mt][j][2] = acc[mt][j][3] = 0.f;
        }

        for (int lc = lc0; lc < lc1; ++lc, ++i) {
            if ((i % C::NG) != grp) continue;  // one warp group per chunk, round robin
            const int stage = i % C::NS;
#ifdef DA_PAGE_TRACE
            // test build: a wait on a barrier that nothing completes runs out
            if (p.debug_stall &&
                !mbar_wait_warp(reinterpret_cast<uint64_t *>(smem + C::OFF_FLAG + 8), 0, abort_flag, p.wait_limit_ns)) {
                if (lane == 0) {
                    atomicOr(&p.meta.header[kHError], DA_DEV_TIMEOUT);
                    *abort_flag = 1;
                }
                break;
            }
#endif
            if (!mbar_wait_warp(&full[stage], (i / C::NS) & 1, abort_flag, p.wait_limit_ns)) {
                if (lane == 0) {
                    atomicOr(&p.meta.header[kHError], DA_DEV_TIMEOUT);
                    *abort_flag = 1;
                }
                break;
            }
            const int cbase = (fc + lc) * kChunk;  // first token of this chunk
            const int nvalid = L - cbase;          // >= 1: tokens of this chunk the last draft token sees
            const int nskip = WIN ? start - cbase : 0;  // > 0: rows before the window (first chunk only)
            uint8_t *stage_ptr = smem + (size_t)stage * C::STAGE;
            const uint32_t s_base = smem_u32(stage_ptr);
            const bool tail = nvalid < kChunk;
            if (tail || nskip > 0) {
                // rows past the sequence end or before the window hold stale or
                // poisoned bytes (or were not loaded): zero them in V so that
                // 0-weight tokens contribute exactly 0 (S is masked below)
                auto zero_v = [&](int a0, int a1) {
                    for (int e = lane; e < (a1 - a0) * C::NX * 8; e += 32) {
                        const int tok = a0 + e / (C::NX * 8), c16 = e % (C::NX * 8);
                        uint4 *vr = reinterpret_cast<uint4 *>(stage_ptr + row_of(tok) + v_half + (c16 >> 3) * xstride);
                        vr[c16 & 7] = make_uint4(0u, 0u, 0u, 0u);
                    }
                };
                if (nskip > 0) zero_v(0, nskip);     // nskip <= nvalid: the ranges do not overlap
                if (tail) zero_v(nvalid, kChunk);
                __syncwarp();
            }
            // ---- S^T = K Q^T for four independent 16-token tiles
            float sacc[4][NQ][4];
#pragma unroll
            for (int t = 0; t < 4; ++t)
#pragma unroll
                for (int j = 0; j < NQ; ++j) sacc[t][j][0] = sacc[t][j][1] = sacc[t][j][2] = sacc[t][j][3] = 0.f;
            if constexpr (!FP8) {
#pragma unroll
                for (int ks = 0; ks < C::KS; ++ks) {
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        const int d = ks * 16 + (lmat >> 1) * 8;
                        const int x = d >> 6;
                        const uint32_t addr =
                            s_base + rk[t] + x * xstride + ((((d & 63) >> 3) ^ (keyk[t] + (HM ? 0 : x))) << 4);
                        uint32_t a[4];
                        ldsm_x4(addr, a[0], a[1], a[2], a[3]);
#pragma unroll
                        for (int j = 0; j < NQ; ++j) mma_bf16(sacc[t][j], a, qf[ks][j][0], qf[ks][j][1]);
                    }
                }
            } else {
#pragma unroll
                for (int kk = 0; kk < D / 32; ++kk) {
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        const int chunk16 = kk * 2 + (lmat >> 1);
                        const uint32_t addr = s_base + rk[t] + ((chunk16 ^ keyk[t]) << 4);
                        uint32_t R[4];
                        ldsm_x4(addr, R[0], R[1], R[2], R[3]);
#pragma unroll
                        for (int hf = 0; hf < 2; ++hf) {
                            const uint32_t ra = R[hf * 2], rb = R[hf * 2 + 1];
                            uint32_t a[4];
                            a[0] = e4m3x2_to_f16x2((uint16_t)(ra & 0xffff));
                            a[1] = e4m3x2_to_f16x2((uint16_t)(rb & 0xffff));
                            a[2] = e4m3x2_to_f16x2((uint16_t)(ra >> 16));
                            a[3] = e4m3x2_to_f16x2((uint16_t)(rb >> 16));
#pragma unroll
                            for (int j = 0; j < NQ; ++j)
                                mma_f16(sacc[t][j], a, qf[kk * 2 + hf][j][0], qf[kk * 2 + hf][j][1]);
                        }
                    }
                }
            }
            // ---- online softmax over the chunk's 64 tokens (rows 16t + r8, 16t + r8 + 8)
            uint32_t pb[4][NQ][2];
#pragma unroll
            for (int j = 0; j < NQ; ++j) {
                const int nv = (NQ * WPC == 1) ? nvalid : L_first + jo + j - cbase;
                // with a window, draft jo + j sees tokens from L_first + jo + j - window on
                const int lv = (WIN && p.window > 0) ? L_first + jo + j - p.window - cbase : -1;
                float sv[4][4];
                float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const int ra = 16 * t + r8, rb = ra + 8;
                    const bool va = ra < nv && ra >= lv, vb = rb < nv && rb >= lv;
                    sv[t][0] = va ? sacc[t][j][0] * sl2 : -INFINITY;
                    sv[t][1] = va ? sacc[t][j][1] * sl2 : -INFINITY;
                    sv[t][2] = vb ? sacc[t][j][2] * sl2 : -INFINITY;
                    sv[t][3] = vb ? sacc[t][j][3] * sl2 : -INFINITY;
                    mx0 = fmaxf(mx0, fmaxf(sv[t][0], sv[t][2]));
                    mx1 = fmaxf(mx1, fmaxf(sv[t][1], sv[t][3]));
                }
                const float mn0 = fmaxf(m0[j], warp_max_xor_4_8_16(mx0));
                const float mn1 = fmaxf(m1[j], warp_max_xor_4_8_16(mx1));
                // an earlier draft token may have seen no token yet: keep the
                // exponent base finite so that 2^(-inf - base) = 0, not NaN
                const float bs0 = (NQ * WPC > 1 && mn0 == -INFINITY) ? 0.f : mn0;
                const float bs1 = (NQ * WPC > 1 && mn1 == -INFINITY) ? 0.f : mn1;
                const float al0 = ex2(m0[j] - bs0), al1 = ex2(m1[j] - bs1);
                float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const float p0 = ex2(sv[t][0] - bs0), p1 = ex2(sv[t][1] - bs1);
                    const float p2 = ex2(sv[t][2] - bs0), p3 = ex2(sv[t][3] - bs1);
                    ps0 += p0 + p2;
                    ps1 += p1 + p3;
                    if constexpr (!FP8) {
                        pb[t][j][0] = movmatrix_t(pack_bf16(p0, p1));
                        pb[t][j][1] = movmatrix_t(pack_bf16(p2, p3));
                    } else {
                        pb[t][j][0] = movmatrix_t(pack_f16(p0, p1));
                        pb[t][j][1] = movmatrix_t(pack_f16(p2, p3));
                    }
                }
                l0[j] = l0[j] * al0 + ps0;
                l1[j] = l1[j] * al1 + ps1;
                m0[j] = mn0;
                m1[j] = mn1;
#pragma unroll
                for (int mt = 0; mt < C::MT; ++mt) {
                    acc[mt][j][0] *= al0;
                    acc[mt][j][1] *= al1;
                    acc[mt][j][2] *= al0;
                    acc[mt][j][3] *= al1;
                }
            }
            // ---- O^T += V^T P^T
            if constexpr (!FP8) {
#pragma unroll
                for (int mt = 0; mt < C::MT; ++mt) {
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        const int d = mt * 16 + (lmat & 1) * 8;
                        const int x = d >> 6;
                        const uint32_t addr =
                            s_base + rv[t] + x * xstride + ((((d & 63) >> 3) ^ (keyv[t] + (HM ? 0 : x))) << 4);
                        uint32_t a[4];
                        ldsm_x4_t(addr, a[0], a[1], a[2], a[3]);
#pragma unroll
                        for (int j = 0; j < NQ; ++j) mma_bf16(acc[mt][j], a, pb[t][j][0], pb[t][j][1]);
                    }
                }
            } else {
#pragma unroll
                for (int kk = 0; kk < D / 32; ++kk) {
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        const int chunk16 = kk * 2 + (lmat >> 1);
                        const uint32_t addr = s_base + rv[t] + ((chunk16 ^ keyv[t]) << 4);
                        uint32_t R[4];
                        ldsm_x4_t(addr, R[0], R[1], R[2], R[3]);
#pragma unroll
                        for (int hf = 0; hf < 2; ++hf) {
                            // bytes of R: [v(t,d), v(t,d+1), v(t+1,d), v(t+1,d+1)] -> token pairs per d
                            const uint32_t u = prmt(R[hf * 2], 0u, 0x3120u);
                            const uint32_t w = prmt(R[hf * 2 + 1], 0u, 0x3120u);
                            uint32_t a[4];
                            a[0] = e4m3x2_to_f16x2((uint16_t)(u & 0xffff));
                            a[1] = e4m3x2_to_f16x2((uint16_t)(u >> 16));
                            a[2] = e4m3x2_to_f16x2((uint16_t)(w & 0xffff));
                            a[3] = e4m3x2_to_f16x2((uint16_t)(w >> 16));
#pragma unroll
                            for (int j = 0; j < NQ; ++j) mma_f16(acc[kk * 2 + hf][j], a, pb[t][j][0], pb[t][j][1]);
                        }
                    }
                }
            }
            if (tail || nskip > 0) fence_proxy_async_smem();  // generic writes above, TMA writes next
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[stage]);
        }

        // ---------------------------------------------------------- merge warps
        // one pass per query token of the request (the scratch holds one);
        // token jj = ow * NQ + jl lives in tile jl of the warps with warp % WPC == ow
        const bool direct = sg.ns == 1;
        const int split = sg.so + ss;
        const bool split_ok = direct || (split >= 0 && split < p.meta.max_splits);
        const size_t rows = (size_t)p.s_q * p.H_q;  // output rows per request: [s_q][H_q]
        int pass = 0;
#pragma unroll
        for (int jl = 0; jl < NQ; ++jl) {
#pragma unroll
            for (int ow = 0; ow < WPC; ++ow) {
                const int jj = ow * NQ + jl;
                if (jj >= p.s_q) continue;
                if (pass++ > 0) named_barrier_sync(1, C::NCW * 32);  // the previous pass has read the scratch
                if (warp % WPC == ow) {
                    const float lj0 = warp_sum_xor_4_8_16(l0[jl]);
                    const float lj1 = warp_sum_xor_4_8_16(l1[jl]);
                    if (lane < 4) {
                        sm_m[warp * C::G + 2 * c4] = m0[jl];
                        sm_m[warp * C::G + 2 * c4 + 1] = m1[jl];
                        sm_l[warp * C::G + 2 * c4] = lj0;
                        sm_l[warp * C::G + 2 * c4 + 1] = lj1;
                    }
                    float *uw = sm_u + (size_t)warp * C::G * C::UPAD;
#pragma unroll
                    for (int mt = 0; mt < C::MT; ++mt) {
                        // accumulator rows -> head-dim index
                        const int dA = FP8 ? mt * 16 + 2 * r8 : mt * 16 + r8;
                        const int dB = FP8 ? dA + 1 : dA + 8;
                        uw[(2 * c4) * C::UPAD + dA] = acc[mt][jl][0];
                        uw[(2 * c4 + 1) * C::UPAD + dA] = acc[mt][jl][1];
                        uw[(2 * c4) * C::UPAD + dB] = acc[mt][jl][2];
                        uw[(2 * c4 + 1) * C::UPAD + dB] = acc[mt][jl][3];
                    }
                }
                named_barrier_sync(1, C::NCW * 32);
                if (ctid < C::G) {
                    const int g = ctid;
                    float M = -INFINITY;
                    for (int w = ow; w < C::NCW; w += WPC) M = fmaxf(M, sm_m[w * C::G + g]);
                    float Ls = 0.f;
                    for (int w = ow; w < C::NCW; w += WPC) {
                        const float mw = sm_m[w * C::G + g];
                        const float wt = (mw == -INFINITY) ? 0.f : ex2(mw - M);
                        sm_w[w * C::G + g] = wt;
                        Ls += wt * sm_l[w * C::G + g];
                    }
                    // lse over the tokens; a request with a single split gets its
                    // attention sink here (the combine adds it to the others)
                    // (a NaN sum -- a NaN code in a row -- stays NaN rather than reading as empty)
                    float lse_v = !(Ls <= 0.f) ? (M + log2f(Ls)) * kLn2 : -INFINITY, fac = 1.f;
                    if (direct && p.sinks != nullptr) {
                        const float tot = log_add_exp(lse_v, p.sinks[h * C::G + g]);
                        fac = (lse_v == -INFINITY) ? 0.f : expf(lse_v - tot);
                        lse_v = tot;
                    }
                    sm_fin[g] = !(Ls <= 0.f) ? vscale * fac / Ls : 0.f;  // out = u * this
                    sm_fin[2 * C::G + g] = lse_v;
                }
                named_barrier_sync(1, C::NCW * 32);
                const size_t row0 = (size_t)jj * p.H_q + (size_t)h * C::G;  // row of head g = row0 + g
                // four consecutive dims per thread and step
                for (int idx = ctid; idx < C::G * (D / 4); idx += C::NCW * 32) {
                    const int g = idx / (D / 4), d = (idx % (D / 4)) * 4;
                    float4 u = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int w = ow; w < C::NCW; w += WPC) {
                        const float wt = sm_w[w * C::G + g];
                        const float4 v = *reinterpret_cast<const float4 *>(sm_u + ((size_t)w * C::G + g) * C::UPAD + d);
                        u.x += wt * v.x;
                        u.y += wt * v.y;
                        u.z += wt * v.z;
                        u.w += wt * v.w;
                    }
                    const float f = sm_fin[g];
                    const float4 o = make_float4(u.x * f, u.y * f, u.z * f, u.w * f);
                    if (direct)
                        *reinterpret_cast<uint2 *>(reinterpret_cast<__nv_bfloat16 *>(p.out) +
                                                   ((size_t)sb * rows + row0 + g) * D + d) =
                            make_uint2(pack_bf16(o.x, o.y), pack_bf16(o.z, o.w));
                    else if (p.cluster_merge)
                        *reinterpret_cast<float4 *>(xo + (size_t)(jj * C::G + g) * D + d) = o;
                    else if (split_ok)
                        *reinterpret_cast<float4 *>(p.meta.o_part + ((size_t)split * rows + row0 + g) * D + d) = o;
                }
                if (ctid < C::G) {
                    const int g = ctid;
                    const float v = sm_fin[2 * C::G + g];
                    if (direct)
                        p.lse[(size_t)sb * rows + row0 + g] = v;
                    else if (p.cluster_merge)
                        xl[jj * C::G + g] = v;
                    else if (split_ok)
                        p.meta.lse_part[(size_t)split * rows + row0 + g] = v;
                }
            }
        }
        if (named_barrier_or(1, C::NCW * 32, *abort_flag != 0)) break;
    }
    if (p.cluster_merge)
        cluster_merge<D>(MergeArgs{p.out, p.lse, p.sinks, p.s_q, p.H_q, p.splits}, xo, xl, merge_b, h,
                         *abort_flag != 0);
}

template <int D, bool FP8, int NQ, int WPC, bool WIN>
static cudaError_t launch_one(const CUtensorMap &tkv, const CUtensorMap &tv, const GqaParams &p, cudaStream_t stream,
                              bool pdl) {
    using C = GqaCfg<D, FP8, NQ, WPC>;
    auto kern = gqa_decode_kernel<D, FP8, NQ, WPC, WIN>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.num_parts, p.H_kv);
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    if (p.cluster_merge) {  // the splits of one (request, KV head) as one cluster
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = (unsigned)p.splits;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kern, tkv, tv, p);
}

// CTAs per SM the automatic partition counts for the build launch_gqa picks.
int gqa_ctas_per_sm(int D, bool fp8, int s_q) {
    return (!fp8 && D == 64 && s_q >= 3 && s_q <= 4) ? 2 : 1;
}

cudaError_t launch_gqa(int D, bool fp8, const CUtensorMap &tkv, const CUtensorMap &tv, const GqaParams &p,
                       cudaStream_t stream, bool pdl) {
    // one token without a window: the lean build; every other shape carries the
    // window logic. Three or four query tokens: four warps per chunk, one token
    // each, at D = 64 (8 consumer warps); a pair of warps, two each, at D = 128.
    if (p.s_q == 1 && p.window == 0) {
        if (!fp8 && D == 64) return launch_one<64, false, 1, 1, false>(tkv, tv, p, stream, pdl);
        if (!fp8 && D == 128) return launch_one<128, false, 1, 1, false>(tkv, tv, p, stream, pdl);
        if (fp8 && D == 128) return launch_one<128, true, 1, 1, false>(tkv, tv, p, stream, pdl);
    } else if (p.s_q == 1) {
        if (!fp8 && D == 64) return launch_one<64, false, 1, 1, true>(tkv, tv, p, stream, pdl);
        if (!fp8 && D == 128) return launch_one<128, false, 1, 1, true>(tkv, tv, p, stream, pdl);
        if (fp8 && D == 128) return launch_one<128, true, 1, 1, true>(tkv, tv, p, stream, pdl);
    } else if (p.s_q == 2) {
        if (!fp8 && D == 64) return launch_one<64, false, 2, 1, true>(tkv, tv, p, stream, pdl);
        if (!fp8 && D == 128) return launch_one<128, false, 2, 1, true>(tkv, tv, p, stream, pdl);
        if (fp8 && D == 128) return launch_one<128, true, 2, 1, true>(tkv, tv, p, stream, pdl);
    } else if (p.s_q <= 4) {
        if (!fp8 && D == 64) return launch_one<64, false, 1, 4, true>(tkv, tv, p, stream, pdl);
        if (!fp8 && D == 128) return launch_one<128, false, 2, 2, true>(tkv, tv, p, stream, pdl);
        if (fp8 && D == 128) return launch_one<128, true, 2, 2, true>(tkv, tv, p, stream, pdl);
    }
    return cudaErrorInvalidValue;
}


}  // namespace da
