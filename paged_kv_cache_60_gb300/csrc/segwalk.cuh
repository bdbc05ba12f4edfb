// Walking the (request, split, chunk range) segments of one part of the
// scheduling metadata; shared by the split-KV kernels.
#pragma once

#include "layout.h"

namespace da {

// One (request, split, local chunk range) piece of a part, with the request's
// clamped length, split base and split count.
struct Seg {
    int b, s, lc0, lc1, L, so, ns;
};

// Walks the segments of one part. The first segment comes entirely from the
// part record, with no dependent load: its request's chunk count follows from
// the record's length as the scheduling kernel computed it (chunk_offset[b + 1]
// - chunk_offset[b] = chunks_of(L)); later segments read the per-request arrays.
struct SegWalker {
    const int32_t *chunk_offset, *split_offset, *num_splits, *seqlens;
    int B, max_len, b, s, c, c1, s_q, window, topk;
    int co0, L0, so0, ns0;
    bool first, pending_empty;
    __device__ bool next(Seg &g) {
        if (pending_empty) {
            pending_empty = false;
            g.b = b;
            g.s = s;
            g.lc0 = g.lc1 = c - co0;
            g.L = L0;
            g.so = so0;
            g.ns = ns0;
            c = c1;
            return true;
        }
        if (b < 0 || c >= c1) return false;
        int cb, ce;
        if (first) {
            cb = co0;
            ce = co0 + chunks_of(L0, s_q, window, topk);
            if (ce <= c) return false;  // inconsistent record
        } else {
            while (b < B && chunk_offset[b + 1] <= c) {
                ++b;
                s = 0;
            }
            if (b >= B) return false;
            cb = chunk_offset[b];
            ce = chunk_offset[b + 1];
        }
        const int end = min(c1, ce);
        g.b = b;
        g.s = s;
        g.lc0 = c - cb;
        g.lc1 = end - cb;
        if (first) {
            g.L = L0;
            g.so = so0;
            g.ns = ns0;
        } else {
            g.L = min(max(seqlens[b], 0), max_len);
            g.so = split_offset[b];
            g.ns = num_splits[b];
        }
        first = false;
        c = end;
        ++b;
        s = 0;
        return true;
    }
};

__device__ __forceinline__ SegWalker make_walker(const MetaView &mv, const int4 r0, const int4 r1, int B,
                                                 const int32_t *seqlens, int max_len, int s_q, int window,
                                                 int topk) {
    SegWalker w;
    w.chunk_offset = mv.chunk_offset;
    w.split_offset = mv.split_offset;
    w.num_splits = mv.num_splits;
    w.seqlens = seqlens;
    w.B = B;
    w.max_len = max_len;
    w.s_q = s_q;
    w.window = window;
    w.topk = topk;
    const bool valid = r0.x >= 0 && r0.x < B && r0.z <= r0.w;
    w.b = valid ? r0.x : -1;
    w.s = r0.y;
    w.c = r0.z;
    w.c1 = r0.w;
    w.co0 = r1.x;
    w.L0 = r1.y;
    w.so0 = r1.z;
    w.ns0 = r1.w;
    w.first = true;
    w.pending_empty = valid && (r0.z == r0.w);
    return w;
}

}  // namespace da
