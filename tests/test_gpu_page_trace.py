"""Page gather, bit for bit. A test build of the library (compiled with
-DDA_PAGE_TRACE, in its own directory) records every pool row the split-KV
kernels read; the ordered lists must equal the reference built from the
oracle's partition and the block table: for each work unit (part, KV head),
chunk by chunk, the rows its boxes (GQA: one TMA box of min(P, 64) tokens;
MLA: one token) must read, and -2 where a box lies past the sequence (or,
with a sliding window, wholly before it; with sparse decode, where a slot
lists no valid position)."""
import ctypes

import pytest
import torch

import paged_kv_cache_60_gb300 as da
from oracle.sched_ref import CHUNK, first_chunk, part_segments, sched_ref, window_start
from workloads import KV_BF16, KV_FP8, KV_MLA656, WorkloadSpec, make_workload

from gpu_util import DeviceWorkload, auto_slots, device_sms, make_desc, debug_build_library

pytestmark = pytest.mark.gpu

FILL = -7


@pytest.fixture(scope="module")
def tlib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    return debug_build_library()


def _reference(w, ref, rows_per_chunk, row_of):
    """Per part: the list of chunks, each a list of rows_per_chunk pool rows."""
    bt = w.block_table.tolist()
    parts = []
    for p in range(ref.num_parts):
        chunks = []
        for (b, _split, lc0, lc1) in part_segments(ref, p):
            L = w.lengths[b]
            for lc in range(lc0, lc1):
                chunks.append([row_of(bt[b], L, lc, j, b) for j in range(rows_per_chunk)])
        parts.append(chunks)
    return parts


def _run(tlib, w, desc, units, cap, per_chunk):
    dw = DeviceWorkload(w)
    s = w.spec
    trace = torch.full((units, cap, per_chunk), FILL, dtype=torch.int32, device="cuda")
    meta = torch.empty(da.sched_meta_bytes(desc), dtype=torch.uint8, device="cuda")
    out = torch.empty(s.B, s.s_q * s.H_q, s.D_v, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(s.B, s.s_q * s.H_q, dtype=torch.float32, device="cuda")
    assert tlib.decode_attn_debug_page_trace(ctypes.c_void_p(trace.data_ptr()), cap) == 0
    try:
        da.sched_meta(desc, dw.cache_seqlens, meta, lib=tlib)
        da.fwd(desc, dw.q, dw.k_pool, dw.v_pool, dw.k_scale, dw.v_scale, dw.block_table, dw.cache_seqlens,
               meta, out, lse, sinks=dw.sinks, indices=dw.indices, lib=tlib)
        torch.cuda.synchronize()
    finally:
        tlib.decode_attn_debug_page_trace(None, 0)
    assert da.get_error(meta) == 0
    return trace.cpu()


def _check(trace, expected_per_unit):
    for u, chunks in enumerate(expected_per_unit):
        n = len(chunks)
        if n:
            assert trace[u, :n].tolist() == chunks, f"unit {u}"
        assert (trace[u, n:] == FILL).all(), f"unit {u} read more than its chunks"


def _gqa(**kw):
    base = dict(name="t", B=3, H_kv=2, G=8, D_qk=128, D_v=128, page_size=16, lengths=[517, 1, 300],
                splits=0, extra_pages=5, seed=41)
    base.update(kw)
    if "lengths" in kw:
        base["B"] = len(kw["lengths"])
    return WorkloadSpec(**base)


GQA_CASES = [
    (dict(), 0),
    (dict(D_qk=64, D_v=64, page_size=256, lengths=[1536, 700, 0, 64], splits=8), 0),
    (dict(kv_dtype=KV_FP8, page_size=32, lengths=[5000, 333], H_kv=4), 0),
    (dict(page_size=64, lengths=[700, 70, 7, 1300, 0, 64]), 6),
    (dict(page_size=8, lengths=[129, 64, 65], splits=3), 0),
    (dict(page_size=128, lengths=[1000, 130]), 0),
    # sliding windows: the pages before each window are never read
    (dict(page_size=16, lengths=[517, 1, 300, 64, 65], window=100), 0),
    (dict(page_size=8, lengths=[1000, 129], window=37, splits=2), 0),
    (dict(page_size=256, lengths=[1536, 300], window=700, sinks=True), 0),
    (dict(D_qk=64, D_v=64, page_size=32, lengths=[900, 3, 70], window=64, s_q=3), 0),
]


@pytest.mark.parametrize("case", range(len(GQA_CASES)))
def test_gqa_page_trace_bit_exact(tlib, case):
    kw, nsm = GQA_CASES[case]
    w = make_workload(_gqa(**kw))
    s = w.spec
    desc = make_desc(w, num_sms=nsm)
    ref = sched_ref(w.lengths, s.H_kv, s.splits, nsm or auto_slots(s), window=s.window, s_q=s.s_q)
    P = s.page_size
    bt_tok = min(P, CHUNK)
    nb = CHUNK // bt_tok

    def row_of(bt_row, L, lc, j, b):
        # local chunk lc is the request's chunk fc + lc; boxes wholly before the
        # window (or past the sequence) are not read
        fc = first_chunk(L, s.window, s.s_q)
        start = window_start(L, s.window, s.s_q)
        tok = (fc + lc) * CHUNK + j * bt_tok
        if tok >= L or tok + bt_tok <= start:
            return -2
        return bt_row[tok // P] * P + (tok % P if P > CHUNK else 0)

    per_part = _reference(w, ref, nb, row_of)
    cap = max(1, max(len(c) for c in per_part))
    trace = _run(tlib, w, desc, ref.num_parts * s.H_kv, cap, nb)
    # unit index = part * H_kv + head; every head of a part reads the same rows
    _check(trace, [per_part[u // s.H_kv] for u in range(ref.num_parts * s.H_kv)])


MLA_CASES = [
    dict(),
    dict(page_size=16, splits=3),
    dict(page_size=32, lengths=[2500, 90, 0, 64]),
    # sparse top-k: the rows of the listed positions, slot by slot
    dict(page_size=16, lengths=[2500, 90, 0, 64], topk=200),
    dict(page_size=64, lengths=[5000, 3000, 10], topk=130, splits=2),
]


@pytest.mark.parametrize("case", range(len(MLA_CASES)))
def test_mla_page_trace_bit_exact(tlib, case):
    base = dict(name="m", B=3, H_kv=1, G=128, D_qk=576, D_v=512, page_size=64, kv_dtype=KV_MLA656,
                lengths=[300, 1, 777], splits=0, extra_pages=3, seed=43)
    base.update(MLA_CASES[case])
    base["B"] = len(base["lengths"])
    w = make_workload(WorkloadSpec(**base))
    s = w.spec
    desc = make_desc(w)
    nsm = device_sms() if s.splits else 2 * da.num_parts(desc)
    ref = sched_ref(w.lengths, 1, s.splits, nsm, cpc=2, topk=s.topk)
    P = s.page_size

    def row_of(bt_row, L, lc, j, b):
        t = lc * CHUNK + j
        if s.topk > 0:   # sparse: the position listed in slot t, if valid
            t = int(w.indices[b, t]) if t < s.topk else -1
            return bt_row[t // P] * P + t % P if 0 <= t < L else -2
        return bt_row[t // P] * P + t % P if t < L else -2

    per_part = _reference(w, ref, CHUNK, row_of)
    cap = max(1, max(len(c) for c in per_part))
    trace = _run(tlib, w, desc, ref.num_parts, cap, CHUNK)
    _check(trace, per_part)
