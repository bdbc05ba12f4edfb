// Host/device shared definitions: sched_meta layout and kernel parameter blocks.
#pragma once

#include <cstddef>
#include <cstdint>

namespace da {

constexpr int kChunk = 64;                 // tokens per scheduling chunk
constexpr int kTmaElemBytes = 8;           // element size the pool tensor maps are described with
constexpr int32_t kMetaMagic = 0x44414d31;  // "DAM1"
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per pipeline wait
constexpr int kMaxSqD64 = 4;               // query tokens per request: bf16 D = 64 kernel
constexpr int kMaxSqD128 = 4;              // bf16 / e4m3 D = 128 kernels
constexpr int kMaxSqMla = 4;               // 656-byte latent format (one CTA pair per query token)

// sched_meta header words
enum MetaHeader : int {
    kHMagic = 0,
    kHB = 1,
    kHHkv = 2,
    kHG = 3,
    kHSplits = 4,
    kHNumParts = 5,
    kHCpc = 6,
    kHChunk = 7,
    kHTotalChunks = 8,
    kHTotalSplits = 9,
    kHPer = 10,
    kHError = 11,
    kHErrorDetail = 12,
    kHKvDtype = 13,
    kHNumSms = 14,
    kHSq = 15,
    kHWindow = 16,
    kHTopk = 17,
    kHeaderWords = 32,
};

// One part record (32 bytes): the part's first request b0, that request's
// split index s0 there, the global chunk interval [c0, c1), and -- so that the
// split-KV kernel needs no further dependent load for the first segment --
// chunk_offset[b0], min(L_b0, max_len), split_offset[b0], num_splits[b0].
struct PartRec {
    int32_t b0, s0, c0, c1, co0, L0, so0, ns0;
};
constexpr int kPartRecInts = 8;

struct MetaLayout {
    size_t header, parts, chunk_offset, split_offset, num_splits, lse_part, o_part, total;
    int32_t num_parts, max_splits, cpc;
};

// Device-side view of sched_meta.
struct MetaView {
    int32_t *header;
    const int4 *parts;            // PartRec as two int4 per part
    const int32_t *chunk_offset;
    const int32_t *split_offset;
    const int32_t *num_splits;
    float *lse_part;   // [max_splits][s_q * H_q]
    float *o_part;     // [max_splits][s_q * H_q][D_v]
    int32_t max_splits;
};

struct SchedParams {
    const int32_t *seqlens;
    int32_t *meta;           // header base
    int32_t *parts;          // PartRec records
    int32_t *chunk_offset;
    int32_t *split_offset;
    int32_t *num_splits;
    int32_t B, H_kv, G, splits, num_parts, cpc, max_len, kv_dtype, num_sms, s_q;
    int32_t window;          // sliding window in tokens, 0: none
    int32_t topk;            // sparse decode: listed positions per request (0: dense)
};

// First token that any of a request's s_q query tokens sees, with a sliding
// window of `window` tokens (0: none): the chunks before the one holding it
// are never read (XQA page, section "分页 KV:页号怎么变成 TMA 坐标").
__host__ __device__ inline int window_start(int L, int s_q, int window) {
    const int st = L - s_q + 1 - window;
    return (window > 0 && st > 0) ? st : 0;
}

// Chunks of a request of (clamped) length L in the schedule: the listed
// positions for sparse decode, else the chunks from the one holding the
// window's first token to the end.
__host__ __device__ inline int chunks_of(int L, int s_q, int window, int topk) {
    return topk > 0 ? (topk + kChunk - 1) / kChunk : (L + kChunk - 1) / kChunk - window_start(L, s_q, window) / kChunk;
}

struct GqaParams {
    const void *q;                 // bf16 [B][s_q][H_q][D]
    const int32_t *block_table;    // [B][max_pages]
    const int32_t *seqlens;        // [B]
    const float *k_scale;          // [H_kv] (fp8) or null
    const float *v_scale;
    MetaView meta;
    void *out;                     // bf16 [B][s_q][H_q][D]
    float *lse;                    // [B][s_q][H_q]
    int32_t B, H_kv, G, H_q, max_pages, num_pages, page_size, box_tokens, boxes_per_chunk;
    int32_t s_q;                   // query tokens per request (draft j sees L - s_q + 1 + j tokens)
    int32_t window;                // sliding window in tokens (0: none)
    const float *sinks;            // [H_q] attention-sink logits (natural-log units) or null
    int32_t cluster_merge;         // 1: fixed split count 2..8, the splits merge inside a cluster (no combine)
    int32_t half_major;            // 1: the tensor maps deliver boxes as [pool][half][token][128 B]
    int32_t log2_box_tokens;       // box_tokens is 8, 16, 32 or 64
    int32_t kv_swap;               // 1: the V pool lies below the K pool (its rows come first in a box)
    int32_t kv_combined;           // 1: one 5-D map covers both pools; 0: one 4-D map per pool
    int32_t splits, num_parts;
    float scale_log2;              // softmax_scale * log2(e)
    uint64_t wait_limit_ns;
    int32_t *page_trace;           // page-trace test build only (null otherwise): rows read, per box
    int32_t page_trace_cap;        // chunks recorded per CTA
    int32_t debug_stall;           // test build only: consumers first wait on a barrier nothing completes
};

struct MlaParams {
    const void *q;                 // bf16 [B][s_q][H_q][576]
    const uint8_t *pool;           // 656-byte tokens
    const int32_t *block_table;
    const int32_t *seqlens;
    MetaView meta;
    void *out;                     // bf16 [B][s_q][H_q][512]
    float *lse;                    // [B][s_q][H_q]
    int32_t B, H_q, max_pages, num_pages, page_size;
    int32_t s_q;                   // query tokens per request (draft j sees L - s_q + 1 + j tokens)
    int32_t log2_page;             // log2(page_size) when it is a power of two, else -1
    int32_t splits, num_parts;
    float scale_log2;
    uint64_t wait_limit_ns;
    int32_t *page_trace;           // page-trace test build only (null otherwise): rows read, per token
    int32_t page_trace_cap;        // chunks recorded per part
    const int32_t *indices;        // sparse decode: [B][topk] token positions, or null
    int32_t topk;                  // 0: dense (tokens [0, L_b))
    int32_t debug_stall;           // test build only: the softmax warps first wait on a barrier nothing completes
};

struct CombineParams {
    MetaView meta;
    void *out;       // bf16 [B][rows][D_v]
    float *lse;      // [B][rows]
    int32_t B, rows, D_v, H_kv, G, splits, num_parts, s_q;   // rows = s_q * H_q per request
    int32_t window, topk;
    const float *sinks;  // [H_q] or null: joins each row's denominator after the merge
};

struct AppendParams {
    const uint16_t *k_new;         // bf16 rows, request b at k_new + b * row_stride
    const uint16_t *v_new;         // same layout (unused for the 656-byte token)
    const int32_t *positions;      // [B]; < 0: request skipped
    const int32_t *block_table;    // [B][max_pages]
    uint8_t *k_pool, *v_pool;
    const float *k_scale, *v_scale;  // [H_kv], e4m3 pools only
    int32_t *error;                // device word, error bits OR-ed in; may be null
    int64_t row_stride;            // bf16 elements between consecutive requests of k_new / v_new
    int32_t B, H_kv, D, page_size, max_pages, num_pages;
};

}  // namespace da
