"""GPU parity for the sliding window and attention sinks (bf16 and e4m3 KV,
one or several query tokens) against oracle.attend_multi, with the pages
before each window taken out of the block table; the windowed schedule is
bit-exact against the scheduling oracle."""
import pytest
import torch

import oracle
import paged_kv_cache_60_gb300 as da
from oracle.sched_ref import sched_ref, window_start
from workloads import WorkloadSpec, make_workload, spec_by_name, KV_BF16, KV_FP8

from gpu_util import LSE_TOL, OUT_TOL, DeviceWorkload, device_sms, ensure_built, make_desc, max_err, read_meta, run

pytestmark = pytest.mark.gpu

LENGTHS = [0, 1, 5, 63, 64, 65, 100, 129, 700, 2000]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    ensure_built()
    oracle.build_oracle()


def _drop_pages_before_window(w):
    """Block-table entries of pages that lie wholly before a request's window
    become -1: a kernel that read one would flag a bad page."""
    s = w.spec
    P = s.page_size
    for b, L in enumerate(w.lengths):
        st = window_start(L, s.window, s.s_q)
        for j in range(st // P):
            w.block_table[b, j] = -1


CASES = [
    # kv, D, s_q, window, sinks, page size, splits
    (KV_BF16, 128, 1, 100, True, 16, 0),
    (KV_BF16, 128, 1, 64, False, 64, 2),
    (KV_BF16, 64, 1, 37, True, 8, 0),
    (KV_BF16, 64, 3, 70, True, 32, 0),
    (KV_BF16, 128, 2, 1, True, 16, 3),
    (KV_BF16, 128, 1, 0, True, 256, 0),
    (KV_FP8, 128, 1, 500, True, 32, 0),
    (KV_FP8, 128, 2, 129, False, 16, 1),
    (KV_BF16, 128, 1, 10 ** 6, True, 16, 0),
]


@pytest.mark.parametrize("kv,D,s_q,W,sinks,P,splits", CASES)
def test_window_sinks_parity(kv, D, s_q, W, sinks, P, splits):
    spec = WorkloadSpec(name="t", B=len(LENGTHS), H_kv=2, G=8, D_qk=D, D_v=D, page_size=P, kv_dtype=kv,
                        lengths=LENGTHS, splits=splits, extra_pages=5, seed=70 + P + W % 97, s_q=s_q,
                        window=W, sinks=sinks)
    w = make_workload(spec)
    _drop_pages_before_window(w)
    out, lse, meta, desc = run(w)
    torch.cuda.synchronize()
    assert da.get_error(meta) == 0
    ref_out, ref_lse = oracle.attend_multi(w)
    e_out, e_lse = max_err(out.view(ref_out.shape), lse.view(ref_lse.shape), ref_out, ref_lse)
    assert e_out <= OUT_TOL and e_lse <= LSE_TOL, (e_out, e_lse)


@pytest.mark.parametrize("splits,s_q,W", [(0, 1, 100), (3, 1, 64), (0, 2, 1), (1, 3, 1000)])
def test_windowed_schedule_bitexact(splits, s_q, W):
    D = 64 if s_q > 2 else 128
    spec = WorkloadSpec(name="t", B=len(LENGTHS), H_kv=2, G=8, D_qk=D, D_v=D, page_size=16, lengths=LENGTHS,
                        splits=splits, extra_pages=2, seed=3, s_q=s_q, window=W)
    w = make_workload(spec)
    dw = DeviceWorkload(w)
    desc = make_desc(w)
    meta = torch.empty(da.sched_meta_bytes(desc), dtype=torch.uint8, device="cuda")
    da.sched_meta(desc, dw.cache_seqlens, meta)
    torch.cuda.synchronize()
    got = read_meta(meta, desc)
    ref = sched_ref(w.lengths, spec.H_kv, splits, num_sms=device_sms(), window=W, s_q=s_q)
    assert got["chunk_offset"] == ref.chunk_offset
    assert got["split_offset"] == ref.split_offset
    assert got["num_splits"] == ref.num_splits
    assert got["parts"] == ref.parts
    assert got["header"][15] == s_q


def test_sinks_dominating_and_absent():
    """A sink of +60 takes all the weight (out = 0, lse = sink); -inf sinks
    equal no sinks, bit for bit."""
    spec = WorkloadSpec(name="t", B=4, H_kv=2, G=8, D_qk=128, D_v=128, page_size=16, lengths=[1, 64, 300, 1000],
                        extra_pages=2, seed=8, sinks=True)
    w = make_workload(spec)
    dw = DeviceWorkload(w)
    o_plain, l_plain, _, _ = run(w, dw=dw)
    dw.sinks = None
    o_none, l_none, _, _ = run(w, dw=dw)
    dw.sinks = torch.full_like(w.sinks, float("-inf")).cuda()
    o_ninf, l_ninf, _, _ = run(w, dw=dw)
    dw.sinks = torch.full_like(w.sinks, 60.0).cuda()
    o_big, l_big, _, _ = run(w, dw=dw)
    torch.cuda.synchronize()
    assert torch.equal(o_none, o_ninf) and torch.equal(l_none, l_ninf)
    assert not torch.equal(o_plain, o_none)
    assert o_big.float().abs().max().item() < 1e-20
    assert (l_big - 60.0).abs().max().item() < 1e-5


def test_window_sinks_bench_workload():
    """The window + sinks workload at full size: every (request, KV head) unit
    against the oracle."""
    spec = spec_by_name("window_sinks_gqa_bf16")
    w = make_workload(spec)
    _drop_pages_before_window(w)
    out, lse, meta, _ = run(w)
    torch.cuda.synchronize()
    assert da.get_error(meta) == 0
    ref_out, ref_lse = oracle.attend_multi(w)
    assert not torch.isnan(ref_lse).any()
    e_out, e_lse = max_err(out.view(ref_out.shape), lse.view(ref_lse.shape), ref_out, ref_lse)
    assert e_out <= OUT_TOL and e_lse <= LSE_TOL, (e_out, e_lse)
