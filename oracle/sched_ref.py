"""Oracle for the split-KV scheduling metadata (integer, bit-exact).

TEST INFRASTRUCTURE ONLY: imported by tests/, the smoke check and the
benchmark's CPU baseline, never by the library.

Work is counted in chunks of C = 64 tokens; request b has
n_b = ceil(L_b / C) - f_b chunks, its chunks f_b .. ceil(L_b / C) - 1. f_b = 0
unless a sliding window of W tokens is set: then the first query token (of s_q
per request) sees tokens from start_b = max(0, L_b - s_q + 1 - W) on, and the
chunks before the one holding start_b are never read, f_b = floor(start_b / C)
(XQA page, section "分页 KV:页号怎么变成 TMA 坐标": with a sliding window the
leading pages are skipped). Sparse top-k decode reads topk listed positions per
request, so n_b = ceil(topk / C) whatever L_b (FlashMLA page: the metadata call
takes topk).

* Fixed mode (splits = S > 0) follows the split range of FlashAttention's
  block.h (FlashAttention tiling page, section 5.3 "Split 在 block.h 中的实现"):
  per = ceil(n_b / S); split s covers chunks [s*per, min((s+1)*per, n_b))
  (clamped to n_b, so a split may be empty). One part per (b, s).

* Auto mode (splits = 0) is the FlashMLA sched-meta idea (FlashMLA page,
  section "调度"): cut the concatenation of all requests' chunks into
  num_parts equal intervals so every SM gets about the same work;
  num_parts = max(1, floor(num_sms / (H_kv * cpc))) where cpc is the number of
  CTAs that share one (part, KV head); per = max(1, ceil(total / num_parts));
  part p covers global chunks [p*per, min((p+1)*per, total)). A request gets
  one split per part it touches; split_offset is the prefix sum of the
  per-request split counts.

Part records are (b0, s0, c0, c1): the first request the part touches, that
request's split index at this part, and the global chunk interval. An auto
mode part that lies past the last chunk is (-1, 0, total, total).
"""
from dataclasses import dataclass
from typing import List, Tuple

CHUNK = 64


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def window_start(L: int, window: int = 0, s_q: int = 1) -> int:
    """First token any query token of the request sees."""
    return max(0, L - s_q + 1 - window) if window > 0 else 0


def first_chunk(L: int, window: int = 0, s_q: int = 1) -> int:
    return window_start(max(0, L), window, s_q) // CHUNK


def auto_num_parts(num_sms: int, H_kv: int, cpc: int) -> int:
    return max(1, num_sms // (H_kv * cpc))


@dataclass
class SchedRef:
    num_parts: int
    per: int                       # auto mode chunk quota per part (0 in fixed mode)
    total_chunks: int
    total_splits: int
    chunk_offset: List[int]        # [B+1]
    split_offset: List[int]        # [B+1]
    num_splits: List[int]          # [B]
    parts: List[Tuple[int, int, int, int]]


def sched_ref(seqlens: List[int], H_kv: int, splits: int, num_sms: int, cpc: int = 1, window: int = 0,
              s_q: int = 1, topk: int = 0) -> SchedRef:
    B = len(seqlens)
    if topk > 0:   # sparse decode: every request has topk listed positions to read
        n = [ceil_div(topk, CHUNK)] * B
    else:
        n = [ceil_div(max(0, L), CHUNK) - first_chunk(L, window, s_q) for L in seqlens]
    chunk_offset = [0]
    for x in n:
        chunk_offset.append(chunk_offset[-1] + x)
    total = chunk_offset[-1]
    parts = []
    if splits > 0:
        S = splits
        num_splits = [S] * B
        for b in range(B):
            per_b = ceil_div(n[b], S)
            for s in range(S):
                lo = min(s * per_b, n[b])
                hi = min((s + 1) * per_b, n[b])
                parts.append((b, s, chunk_offset[b] + lo, chunk_offset[b] + hi))
        num_parts, per = B * S, 0
    else:
        num_parts = auto_num_parts(num_sms, H_kv, cpc)
        per = max(1, ceil_div(total, num_parts))
        first_part = [-1] * B
        num_splits = [0] * B
        for b in range(B):
            if n[b] > 0:
                first = chunk_offset[b] // per
                last = (chunk_offset[b + 1] - 1) // per
                first_part[b] = first
                num_splits[b] = last - first + 1
        for p in range(num_parts):
            c0 = min(p * per, total)
            c1 = min(c0 + per, total)
            if c0 >= total:
                parts.append((-1, 0, total, total))
                continue
            b0 = next(b for b in range(B) if chunk_offset[b] <= c0 < chunk_offset[b + 1])
            parts.append((b0, p - first_part[b0], c0, c1))
    split_offset = [0]
    for x in num_splits:
        split_offset.append(split_offset[-1] + x)
    return SchedRef(num_parts=num_parts, per=per, total_chunks=total,
                    total_splits=split_offset[-1], chunk_offset=chunk_offset,
                    split_offset=split_offset, num_splits=num_splits, parts=parts)


def part_segments(ref: SchedRef, p: int):
    """The (b, split, first_local_chunk, end_local_chunk) pieces of part p, in order."""
    b0, s0, c0, c1 = ref.parts[p]
    if b0 < 0:
        return []
    if c0 == c1:            # fixed-mode empty split
        lc = c0 - ref.chunk_offset[b0]
        return [(b0, s0, lc, lc)]
    out = []
    b, s, c = b0, s0, c0
    B = len(ref.num_splits)
    while c < c1:
        while ref.chunk_offset[b + 1] <= c:
            b += 1
            s = 0
        end = min(c1, ref.chunk_offset[b + 1])
        out.append((b, s, c - ref.chunk_offset[b], end - ref.chunk_offset[b]))
        c = end
        b += 1
        s = 0
        if b >= B:
            break
    return out


def split_token_ranges(ref: SchedRef, seqlens: List[int], window: int = 0, s_q: int = 1):
    """For every request, the token range [t0, t1) of each of its splits, in
    split order (local chunk lc is the request's chunk f_b + lc; the first
    split starts at the window start)."""
    B = len(seqlens)
    ranges = [[None] * ref.num_splits[b] for b in range(B)]
    for p in range(ref.num_parts):
        for (b, s, lc0, lc1) in part_segments(ref, p):
            L = seqlens[b]
            f = first_chunk(L, window, s_q)
            t0 = max(window_start(L, window, s_q), min((f + lc0) * CHUNK, L))
            t1 = max(t0, min((f + lc1) * CHUNK, L))
            ranges[b][s] = (t0, t1)
    return ranges
