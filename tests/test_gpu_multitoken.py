"""GPU parity for several query tokens per request (a chain of s_q drafts;
draft j sees the first L - s_q + 1 + j tokens) against oracle.attend_multi:
lse within 1e-4, out within 2e-2, through the C ABI."""
import dataclasses

import pytest
import torch

import oracle
import paged_kv_cache_60_gb300 as da
from workloads import WorkloadSpec, make_workload, spec_by_name, KV_BF16, KV_FP8

from oracle.sched_ref import sched_ref

from gpu_util import LSE_TOL, OUT_TOL, DeviceWorkload, auto_slots, device_sms, ensure_built, make_desc, max_err, read_meta, run

pytestmark = pytest.mark.gpu

# lengths below s_q (drafts that see nothing), chunk edges, several chunks
LENGTHS = [0, 1, 2, 3, 63, 64, 65, 66, 127, 130, 517, 1000]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    ensure_built()
    oracle.build_oracle()


def _check(w, splits=None, **kw):
    out, lse, _, _ = run(w, splits=splits, **kw)
    torch.cuda.synchronize()
    ref_out, ref_lse = oracle.attend_multi(w)
    e_out, e_lse = max_err(out.view(ref_out.shape), lse.view(ref_lse.shape), ref_out, ref_lse)
    assert e_out <= OUT_TOL and e_lse <= LSE_TOL, (e_out, e_lse)
    return out, lse


CASES = [
    # kv, D, s_q, page size, splits
    (KV_BF16, 64, 2, 16, 0),
    (KV_BF16, 64, 3, 8, 0),
    (KV_BF16, 64, 4, 64, 3),
    (KV_BF16, 64, 4, 256, 0),
    (KV_BF16, 128, 2, 16, 0),
    (KV_BF16, 128, 2, 32, 4),
    (KV_FP8, 128, 2, 16, 0),
    (KV_FP8, 128, 2, 64, 1),
    # three or four query tokens at D = 128: a pair of warps per chunk
    (KV_BF16, 128, 3, 16, 0),
    (KV_BF16, 128, 4, 64, 2),
    (KV_FP8, 128, 4, 32, 0),
    (KV_FP8, 128, 3, 8, 3),
]


@pytest.mark.parametrize("kv,D,s_q,P,splits", CASES)
def test_multitoken_parity(kv, D, s_q, P, splits):
    spec = WorkloadSpec(name="t", B=len(LENGTHS), H_kv=2, G=8, D_qk=D, D_v=D, page_size=P, kv_dtype=kv,
                        lengths=LENGTHS, splits=splits, extra_pages=5, seed=40 + s_q + P, s_q=s_q)
    _check(make_workload(spec))


def test_s_q_one_and_zero_are_single_token():
    """s_q = 1 (and 0, meaning 1) is the single-token path, bit for bit."""
    spec = WorkloadSpec(name="t", B=4, H_kv=2, G=8, D_qk=128, D_v=128, page_size=16,
                        lengths=[5, 300, 64, 129], extra_pages=3, seed=9)
    w = make_workload(spec)
    dw = DeviceWorkload(w)
    o1, l1, _, _ = run(w, dw=dw, desc=make_desc(w))
    d0 = make_desc(w)
    d0.s_q = 0
    o0, l0, _, _ = run(w, dw=dw, desc=d0)
    torch.cuda.synchronize()
    assert torch.equal(o1, o0) and torch.equal(l1, l0)


def test_last_draft_matches_single_token_kernel():
    """The last draft sees the whole sequence: the same rows as a one-token
    decode with that query (compared within tolerance: another kernel build)."""
    spec = WorkloadSpec(name="t", B=5, H_kv=2, G=8, D_qk=128, D_v=128, page_size=32,
                        lengths=[70, 1, 640, 2000, 33], extra_pages=3, seed=12, s_q=2)
    w = make_workload(spec)
    out, lse, _, _ = run(w)
    single = dataclasses.replace(w, spec=spec.with_(s_q=1), q=w.q[:, -1].contiguous())
    o1, l1, _, _ = run(single)
    torch.cuda.synchronize()
    assert (out[:, -1].float() - o1.float()).abs().max().item() <= OUT_TOL
    assert (lse[:, -1] - l1).abs().max().item() <= LSE_TOL


@pytest.mark.parametrize("name", ["spec2_gqa_bf16", "spec4_gqa_d64", "spec2_fp8_gqa", "spec4_gqa_bf16"])
def test_multitoken_bench_workloads(name):
    """The benchmark's multi-token workloads at full size, in its launch
    configuration; every (request, KV head) unit against the oracle."""
    spec = spec_by_name(name)
    w = make_workload(spec)
    out, lse, _, _ = run(w)
    torch.cuda.synchronize()
    ref_out, ref_lse = oracle.attend_multi(w)
    assert not torch.isnan(ref_lse).any()
    e_out, e_lse = max_err(out.view(ref_out.shape), lse.view(ref_lse.shape), ref_out, ref_lse)
    assert e_out <= OUT_TOL and e_lse <= LSE_TOL, (e_out, e_lse)


def test_unsupported_s_q_rejected_on_host():
    ensure_built()
    d = da.Desc.make(B=2, H_kv=2, G=8, D_qk=128, D_v=128, page_size=16, max_pages_per_seq=4, num_pages=10,
                     s_q=5)
    with pytest.raises(da.DecodeAttnError):
        da.sched_meta_bytes(d)


def test_two_ctas_per_sm_partition():
    """The bf16 D = 64 build for three or four query tokens runs two CTAs per
    SM: its automatic partition counts two slots per SM, bit-exact against the
    oracle's partition for that count, and the results still match the oracle."""
    for s_q in (3, 4):
        spec = WorkloadSpec(name="t", B=len(LENGTHS), H_kv=2, G=8, D_qk=64, D_v=64, page_size=16, kv_dtype=KV_BF16,
                            lengths=LENGTHS, splits=0, extra_pages=5, seed=90 + s_q, s_q=s_q)
        w = make_workload(spec)
        desc = make_desc(w)
        assert da.num_parts(desc) == (2 * device_sms()) // spec.H_kv
        out, lse, meta, desc = run(w)
        torch.cuda.synchronize()
        assert da.get_error(meta) == 0
        got = read_meta(meta, desc)
        ref = sched_ref(w.lengths, spec.H_kv, 0, num_sms=auto_slots(spec), s_q=s_q)
        assert got["parts"] == ref.parts
        assert got["split_offset"] == ref.split_offset
        ref_out, ref_lse = oracle.attend_multi(w)
        e_out, e_lse = max_err(out.view(ref_out.shape), lse.view(ref_lse.shape), ref_out, ref_lse)
        assert e_out <= OUT_TOL and e_lse <= LSE_TOL, (e_out, e_lse)
    # the other multi-token builds keep one slot per SM
    spec = WorkloadSpec(name="t", B=2, H_kv=2, G=8, D_qk=128, D_v=128, page_size=16, kv_dtype=KV_BF16,
                        lengths=[100, 200], splits=0, seed=95, s_q=4)
    assert da.num_parts(make_desc(make_workload(spec))) == device_sms() // 2
