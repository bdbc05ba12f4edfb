/*
 * decode_attn.h -- C ABI of the paged-KV decode attention library (GB300, sm_103a).
 *
 * The operation (XQA page "TensorRT-LLM 源码完全拆解(二十九)", section
 * "先把 decode 注意力的约束写清楚"): one new query token per request. For request
 * b, KV head h and the G query heads h*G+g that share it,
 *
 *     out[b, h*G+g, :] = softmax(sigma * q[b, h*G+g, :] . K_{b,h}^T) V_{b,h}
 *     lse[b, h*G+g]    = ln sum_t exp(sigma * q . k_t)           (natural log)
 *
 * where K_{b,h}, V_{b,h} are the first L_b = cache_seqlens[b] tokens of the
 * request, gathered through block_table from a pool of fixed-size pages
 * (XQA page, section "Hopper:一次 TMA 只搬一个页", "VLLM layout").
 *
 * The work is split along the sequence into split-KV partials, each with its
 * own lse, and a combine step merges them (XQA page, section "归约怎么记";
 * FlashMLA page "FlashMLA 注意力内核源码走读", sections "调度" and
 * "合并与性能账本"). The call sequence follows FlashMLA's two-call shape:
 *
 *     decode_attn_sched_meta(...)   once per change of cache_seqlens (reusable)
 *     decode_attn_fwd(...)          every decode step / layer
 *
 * Memory: the caller allocates every buffer. The library never allocates,
 * never synchronises inside decode_attn_fwd, and keeps no per-call state
 * outside the sched_meta buffer. All pointers below are DEVICE pointers unless
 * noted; all must be 16-byte aligned.
 *
 * Errors: every entry point returns DA_OK (0) or a negative DA_ERR_* code,
 * detected on the host before anything is launched. Errors that only the
 * device can see (a block-table entry outside the pool, a length beyond
 * max_pages_per_seq * page_size, a pipeline wait that ran out of time) set
 * bits in an error word inside sched_meta; the kernels skip the offending
 * work and never trap. Read the word with decode_attn_get_error.
 *
 * Determinism: identical inputs give bitwise identical out and lse (fixed
 * reduction order, no floating-point atomics).
 */
#ifndef DECODE_ATTN_H
#define DECODE_ATTN_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* KV cache formats. */
typedef enum {
    /* k_pool, v_pool: bf16 [num_pages][page_size][H_kv][D], D = D_qk = D_v. */
    DA_KV_BF16 = 0,
    /* k_pool, v_pool: float8 e4m3 bytes [num_pages][page_size][H_kv][D];
     * element value = e4m3 * k_scale[h] (resp. v_scale[h]), one fp32 scale per
     * (KV head, tensor) -- the per-tensor KV scale of the XQA page, section
     * "Hopper 路径上 V 不做显式反量化". */
    DA_KV_FP8_PER_TENSOR = 1,
    /* k_pool: 656-byte tokens [num_pages][page_size][1][656] (FlashMLA page,
     * section "数据加载"): 512 e4m3, 4 fp32 scales (one per 128 values), 64 bf16
     * RoPE values. K = the 576 dequantised values, V = the first 512. v_pool
     * must be NULL or equal to k_pool; H_kv = 1, D_qk = 576, D_v = 512.
     * Codes 0x7F / 0xFF decode to NaN (and so poison the rows that read
     * them), as in the bf16 and per-tensor formats; the quantiser,
     * decode_attn_append_kv, never writes them: it saturates at +-448. */
    DA_KV_FP8_MLA656 = 2
} da_kv_dtype;

/* Problem description (host struct, passed by pointer, not retained). */
typedef struct {
    int32_t B;                 /* requests */
    int32_t H_kv;              /* KV heads */
    int32_t G;                 /* query heads per KV head; H_q = H_kv * G */
    int32_t D_qk;              /* q / K head size */
    int32_t D_v;               /* V / out head size */
    int32_t page_size;         /* tokens per page P: 8, 16, 32 or a multiple of 64 */
    int32_t max_pages_per_seq; /* row length of block_table */
    int32_t num_pages;         /* pages in the pool */
    int32_t kv_dtype;          /* da_kv_dtype */
    int32_t splits;            /* 0: balanced over the SMs; S > 0: S splits per request */
    int32_t num_sms;           /* 0: query the current device; the automatic partition then counts
                                  the SMs that can hold the 656-byte kernel's clusters at once, or
                                  two slots per SM for the bf16 D = 64 build with 3-4 query tokens
                                  (it runs two CTAs per SM); > 0: the slot count to partition for */
    float softmax_scale;       /* sigma; 0: 1/sqrt(D_qk) */
    int32_t s_q;               /* query tokens per request (0 means 1); see decode_attn_fwd */
    int32_t window;            /* sliding window W in tokens (0: none); see decode_attn_fwd */
    int32_t topk;              /* sparse decode: positions listed per request (0: dense); see decode_attn_fwd */
} da_desc;

/* Return codes. */
#define DA_OK                  0
#define DA_ERR_NULL           -1   /* a required pointer is NULL */
#define DA_ERR_DIMS           -2   /* a size is out of range */
#define DA_ERR_UNSUPPORTED    -3   /* no kernel for this (dtype, D_qk, D_v, G, page_size, s_q) */
#define DA_ERR_ALIGN          -4   /* a pointer is not 16-byte aligned */
#define DA_ERR_SPLITS         -5   /* splits < 0 or too large */
#define DA_ERR_META_SIZE      -6   /* sched_meta buffer smaller than decode_attn_sched_meta_bytes */
#define DA_ERR_CUDA           -7   /* a CUDA runtime/driver call failed */
#define DA_ERR_SCALE          -8   /* FP8 format without k_scale / v_scale */

/* Device error bits (sched_meta error word). */
#define DA_DEV_BAD_PAGE        1   /* block_table entry outside [0, num_pages): page skipped */
#define DA_DEV_SEQ_TOO_LONG    2   /* cache_seqlens[b] > max_pages_per_seq * page_size: clamped */
#define DA_DEV_NEG_LEN         4   /* cache_seqlens[b] < 0: treated as 0 */
#define DA_DEV_TIMEOUT         8   /* a pipeline wait ran out of time: work unit abandoned */
#define DA_DEV_META_MISMATCH  16   /* sched_meta was built for another desc */

/*
 * Library plumbing from here to decode_attn_num_parts: no page defines these
 * calls; they size and describe the caller-owned sched_meta buffer.
 *
 * Size in bytes of the sched_meta buffer for this desc (host only, no CUDA
 * call except an SM-count query when desc->num_sms is 0). The buffer holds the
 * scheduling metadata, the split-KV partials (fp32 o and lse per split and
 * output row: query token x query head) and the device error word.
 */
int decode_attn_sched_meta_bytes(const da_desc *desc, size_t *bytes);

/*
 * Byte offsets inside sched_meta, for inspection and tests. offs[0..7] =
 * header, parts, chunk_offset, split_offset, num_splits, lse_part, o_part,
 * total size. Header (32 int32): magic, B, H_kv, G, splits, num_parts, cpc,
 * chunk (64), total_chunks, total_splits, per, error word, error detail,
 * kv_dtype, num_sms, s_q, window, topk, then zeros. parts: num_parts records of 8 int32
 * {b0, s0, c0, c1, co0, L0, so0, ns0}: first request, its split index there,
 * global chunk interval [c0, c1), then chunk_offset[b0], min(L_b0,
 * max_pages_per_seq*page_size), split_offset[b0], num_splits[b0] (all 0 when
 * b0 = -1, a part with no work). chunk_offset, split_offset: int32 [B+1]
 * prefix sums; num_splits: int32 [B].
 */
int decode_attn_meta_offsets(const da_desc *desc, size_t offs[8]);

/* Number of parts (grid x of the split-KV kernel) for this desc. */
int decode_attn_num_parts(const da_desc *desc, int32_t *num_parts);

/*
 * Scheduling metadata (FlashMLA page, section "调度": a small kernel hands the
 * (request, KV range) work units to the SMs ahead of time; the main kernel
 * only reads them). Work is counted in chunks of 64 tokens.
 *   splits = S > 0: request b is cut into S ranges of ceil(n_b / S) chunks
 *     (FlashAttention tiling page, section 5.3, block.h split range);
 *   splits = 0: all chunks of all requests are cut into
 *     num_parts = floor(num_sms / (H_kv * cpc)) equal intervals, one per part.
 * With a sliding window (desc->window = W > 0) a request's chunks start at the
 * one holding token max(0, L_b - s_q + 1 - W), the first its first query token
 * sees: the pages before it are never read (XQA page, section
 * "分页 KV:页号怎么变成 TMA 坐标"), and their block_table entries may hold
 * anything. Sparse decode (desc->topk = k > 0) gives every request k slots,
 * ceil(k / 64) chunks, whatever its length.
 * cache_seqlens: device int32 [B]. sched_meta: device, caller-owned, at least
 * decode_attn_sched_meta_bytes. Launches one small kernel on `stream`; the
 * result may be reused by any number of decode_attn_fwd calls while
 * cache_seqlens and desc stay the same. Clears the device error word.
 */
int decode_attn_sched_meta(const da_desc *desc, const int32_t *cache_seqlens,
                           void *sched_meta, size_t sched_meta_bytes, cudaStream_t stream);

/*
 * Decode attention forward. Launches the split-KV kernel and the LSE combine
 * kernel (chained with programmatic dependent launch) on `stream`. With a
 * fixed split count of 2-8 (desc->splits) and the bf16 or e4m3 formats, the
 * splits of a (request, KV head) run as one thread-block cluster and merge
 * their partials through distributed shared memory: the split-KV kernel then
 * writes out and lse itself and no combine kernel is launched.
 *
 * Several query tokens per request (desc->s_q > 1) verify a chain of draft
 * tokens (XQA page, section "投机解码:XQA 的第二个工作负载", the linear case;
 * FlashMLA's call passes s_q * h_q / h_kv rows per KV head): the request's
 * last s_q tokens are already in the pool (L_b counts them) and draft token
 * j < s_q sees the first L_b - s_q + 1 + j tokens -- the history and the
 * drafts up to itself. A row that sees no token gets out = 0, lse = -inf.
 * Supported: s_q <= 4 for all three formats (on the 656-byte format the
 * sliding window and, when s_q > 1, sparse decode are not offered:
 * DA_ERR_UNSUPPORTED). The rows of q, out and lse below are
 * then [B][s_q][H_kv*G]; the scheduling metadata must be built with the same s_q.
 *
 * Sliding window (desc->window = W > 0; XQA page, section
 * "分页 KV:页号怎么变成 TMA 坐标"): a query token at position p sees only the
 * tokens (p - W, p]. Attention sinks (da_launch_opts.sinks; XQA page, section
 * "一个容易漏掉的细节:attention sink"): one fp32 logit per query head, in the
 * units of sigma * q.k, that joins each row's softmax denominator and carries
 * no value: lse = ln(e^sink + sum_t e^{s_t}), out = sum_t e^{s_t - lse} v_t;
 * a row that sees no token gets out = 0 and lse = sink. Both are for the
 * bf16 and e4m3 formats (DA_ERR_UNSUPPORTED with the 656-byte format).
 *
 * Sparse top-k decode (desc->topk = k > 0, da_launch_opts.indices; the
 * FlashMLA page's decode call with `indices`, ledger rows "FP8 稀疏解码"): for
 * the 656-byte format only. indices is device int32 [B][k]; request b attends
 * over the token positions indices[b][0..k) instead of [0, L_b): each is a
 * position in the request, mapped through block_table like a dense token;
 * entries outside [0, L_b) (-1 padding, stale positions) are skipped, and a
 * position listed twice counts twice. A request with no valid entry gets
 * out = 0, lse = -inf. Pages that no listed position touches are never read.
 *
 *   q:            bf16 [B][H_kv*G][D_qk], query head h*G+g belongs to KV head h
 *   k_pool/v_pool: see da_kv_dtype
 *   k_scale/v_scale: fp32 [H_kv] for DA_KV_FP8_PER_TENSOR, else ignored
 *   block_table:  int32 [B][max_pages_per_seq]; entries past ceil(L_b/P) are never read
 *   cache_seqlens: int32 [B] (must match what sched_meta was built from)
 *   sched_meta:   from decode_attn_sched_meta; its partial buffers are overwritten,
 *                 so two calls sharing one sched_meta must not overlap in time
 *   out:          bf16 [B][H_kv*G][D_v]; lse: fp32 [B][H_kv*G]
 * A request with L_b = 0 gets out = 0 and lse = -inf.
 */
int decode_attn_fwd(const da_desc *desc, const void *q, const void *k_pool, const void *v_pool,
                    const float *k_scale, const float *v_scale, const int32_t *block_table,
                    const int32_t *cache_seqlens, void *sched_meta, size_t sched_meta_bytes,
                    void *out, float *lse, cudaStream_t stream);

/* Launch options for decode_attn_fwd_ex. */
typedef struct {
    int32_t use_pdl;          /* 1 (default behaviour of decode_attn_fwd): PDL-chain the kernels */
    cudaEvent_t main_begin;   /* if not NULL: recorded on `stream` just before the split-KV kernel */
    cudaEvent_t main_end;     /* if not NULL: recorded just after it (before the combine kernel) */
    const float *sinks;       /* if not NULL: device fp32 [H_kv*G] attention-sink logits (see decode_attn_fwd) */
    const int32_t *indices;   /* sparse decode (desc->topk > 0): device int32 [B][topk] token positions */
} da_launch_opts;

/* decode_attn_fwd with launch options and optional inputs (opts may be NULL). */
int decode_attn_fwd_ex(const da_desc *desc, const void *q, const void *k_pool, const void *v_pool,
                       const float *k_scale, const float *v_scale, const int32_t *block_table,
                       const int32_t *cache_seqlens, void *sched_meta, size_t sched_meta_bytes,
                       void *out, float *lse, const da_launch_opts *opts, cudaStream_t stream);

/*
 * KV append: writes each request's new token into the pool, the step that
 * precedes decode attention (XQA page, section "一次 decode step 的完整时序":
 * the new K/V lands in the paged pool upstream, and the attention kernel then
 * reads it through the page table). Request b's token, at position
 * t = positions[b] (its index in the request: the cache_seqlens[b] of the
 * step before, so the next decode uses t + 1), goes to slot t % page_size of
 * page block_table[b][t / page_size], for every KV head.
 *   desc: B, H_kv, D_qk, D_v, page_size, max_pages_per_seq, num_pages and
 *     kv_dtype are used (the others are ignored). bf16 and e4m3 pools need
 *     D_qk == D_v, a multiple of 8; the 656-byte token H_kv = 1, D_qk = 576,
 *     D_v = 512. The pools are those of decode_attn_fwd.
 *   k_new, v_new: device bf16, request b's row at (k_new + b * new_row_stride):
 *     H_kv x D values (head-major), or for the 656-byte token the 576 values of
 *     the latent vector (512 NoPE, then 64 RoPE) with v_new = NULL (V is the
 *     first 512 of them). new_row_stride counts bf16 elements (0: packed rows;
 *     else at least the row length and a multiple of 8), so rows may sit inside
 *     a larger fused projection output.
 *   positions: device int32 [B]; a negative position skips the request.
 *   block_table: device int32 [B][max_pages_per_seq].
 *   k_pool, v_pool: device, written in place; only the addressed slots change.
 *     v_pool must be NULL or k_pool for the 656-byte token.
 *   k_scale, v_scale: device fp32 [H_kv] for DA_KV_FP8_PER_TENSOR (read only).
 *   device_error: device int32 or NULL; DA_DEV_SEQ_TOO_LONG (t >=
 *     max_pages_per_seq * page_size) and DA_DEV_BAD_PAGE (page id outside
 *     [0, num_pages)) are OR-ed into it, and such a request is skipped.
 * Quantisation (e4m3, OCP FP8: largest finite 448): code = nearest e4m3 to the
 * fp32 quotient x / scale (IEEE division, round to nearest even), ties to the
 * even code, saturating at +-448, NaN -> 0x7F. Per-tensor pools divide by
 * k_scale[h] / v_scale[h] (XQA page, section "Hopper 路径上 V 不做显式反量化");
 * the 656-byte token (FlashMLA page, section "数据加载") takes, per block of 128
 * NoPE values, scale = max|x| / 448 in fp32 (1 for an all-zero block), stores
 * the 512 codes, the 4 fp32 scales and the 64 RoPE values unchanged.
 * Pointers to bf16 rows and pools must be 16-byte aligned, the others 4-byte.
 * Launches one kernel on `stream` (programmatic dependent launch: a following
 * decode_attn_fwd may start early and waits for it before reading the pool).
 * Two requests that address the same slot race. No allocation, no sync.
 */
int decode_attn_append_kv(const da_desc *desc, const void *k_new, const void *v_new, int64_t new_row_stride,
                          const int32_t *positions, const int32_t *block_table, void *k_pool, void *v_pool,
                          const float *k_scale, const float *v_scale, int32_t *device_error, cudaStream_t stream);

/*
 * Reads the device error word of sched_meta into *device_error (host int32).
 * Synchronises `stream`. Library plumbing: no page defines this call.
 */
int decode_attn_get_error(const void *sched_meta, int32_t *device_error, cudaStream_t stream);

/* Size of the library's fixed device scratch buffer (16 MiB). */
#define DA_STATIC_SCRATCH_BYTES (16u << 20)

/*
 * decode_attn_sched_meta + decode_attn_fwd in one call that allocates
 * nothing and needs no caller-provided scratch. (No counterpart on the source
 * pages: it exists for deployment.) It is meant for callers that cannot
 * allocate device memory or hand the library a buffer -- a server that plans
 * all device memory up front and may not call cudaMalloc later, a plug-in that
 * cannot reach its host's allocator, a real-time path that must not risk an
 * allocation.
 *
 * The scheduling metadata and the split-KV partials live in a static device
 * array of DA_STATIC_SCRATCH_BYTES that the library owns; every GPU that loads
 * the library keeps it until the process exits. Problems whose
 * decode_attn_sched_meta_bytes exceeds that size are rejected with
 * DA_ERR_META_SIZE. With the 656-byte format the automatic split count
 * (desc->splits = 0) of a GB300 needs (76 + B) x 256 KB of partials at s_q = 1,
 * over 16 MiB for any B, and is rejected: pass a fixed split count or a
 * smaller desc->num_sms. Sparse decode (desc->topk > 0) needs
 * indices, which this call cannot take: DA_ERR_UNSUPPORTED.
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current): make that first call
 * before any stream capture. The address is kept per device and CUDA context;
 * after a device reset the next call looks it up again. Every call reuses the
 * same array and leaves its contents behind; the scheduling kernel rewrites
 * all it reads, so nothing needs clearing, but calls whose work overlaps on
 * the GPU race on the array. Every argument is checked on the host before
 * anything is launched, so a rejected call leaves the array untouched.
 * Arguments, layouts and errors are those of decode_attn_fwd; device errors
 * land in the array's error word and are not readable from outside.
 */
int decode_attn_fwd_static_scratch(const da_desc *desc, const void *q, const void *k_pool, const void *v_pool,
                                   const float *k_scale, const float *v_scale, const int32_t *block_table,
                                   const int32_t *cache_seqlens, void *out, float *lse, cudaStream_t stream);

/* Static description of a return code (never NULL). Library plumbing: no
 * page defines this call. */
const char *decode_attn_strerror(int code);

#ifdef DA_PAGE_TRACE
/* Test build only (the library compiled with -DDA_PAGE_TRACE; the product
 * build does not export it). Makes every later decode_attn_fwd record the
 * pool rows its kernels read into `trace` (device memory, int32, caller-owned,
 * written in place): for the GQA formats, per (part, KV head) unit, per chunk
 * in reading order, per TMA box of min(page_size, 64) tokens, the first pool
 * row of the box (page * page_size + offset within the page), or -2 for a box
 * past the sequence; for the 656-byte format, per part, per chunk, per token,
 * the token's pool row or -2. `cap` chunks are kept per unit (later ones are
 * not recorded); the unit stride is cap * rows_per_chunk. A null `trace`
 * stops recording. Returns DA_ERR_DIMS for cap < 1 with a non-null trace.
 * There is no counterpart on the pages: it checks the page gather (block
 * table -> page -> slot, XQA page section "Hopper:一次 TMA 只搬一个页") bit for
 * bit against a reference built from the partition and the block table. */
int decode_attn_debug_page_trace(int32_t *trace, int32_t cap);

/* Test build only. Limits every bounded wait (mbarrier phase, peer CTA) of
 * later launches to `ns` nanoseconds; 0 restores the product limit of 2 s. A
 * wait that runs out sets DA_DEV_TIMEOUT in the device error word, the
 * kernel's CTAs stop their work units and return, and the CUDA context stays
 * usable; it exists so that tests can make waits run out without a fault.
 * No counterpart on the pages. Always returns DA_OK. */
int decode_attn_debug_wait_limit(uint64_t ns);

/* Test build only. With `on` != 0, the consumer warps of later GQA-format
 * launches first wait (bounded, see above) on an mbarrier that nothing
 * completes: the wait runs out, DA_DEV_TIMEOUT is set and the CTAs return.
 * 0 turns it off. No counterpart on the pages. Always returns DA_OK. */
int decode_attn_debug_stall(int32_t on);
#endif

#ifdef __cplusplus
}
#endif

#endif /* DECODE_ATTN_H */
