"""GPU parity for the 656-byte FP8 latent-token path (128 query heads on one
KV head, D_qk = 576, D_v = 512): the tensor-core kernel through the C ABI
against the float64 oracle. Metadata bit-exact (two CTAs per part), lse within
1e-4, out within 2e-2."""
import dataclasses

import pytest
import torch

import oracle
import paged_kv_cache_60_gb300 as da
from oracle.sched_ref import sched_ref
from workloads import WorkloadSpec, make_workload, spec_by_name, KV_MLA656

from gpu_util import LSE_TOL, OUT_TOL, device_sms, ensure_built, expected_part_extra, max_err, read_meta, run

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    ensure_built()
    oracle.build_oracle()


def _auto_sms(desc):
    """SM count the auto partition was built for: the library counts only the
    SMs that can hold its clusters (2 s_q CTAs, one per SM) at the same time."""
    cpc = 2 * max(1, desc.s_q)
    if desc.splits > 0:
        return device_sms()
    n = da.num_parts(desc)
    assert 1 <= cpc * n <= device_sms()
    return cpc * n


def _mla(**kw):
    base = dict(name="m", B=3, H_kv=1, G=128, D_qk=576, D_v=512, page_size=64, kv_dtype=KV_MLA656,
                lengths=[300, 1, 777], splits=0, extra_pages=3, seed=31)
    base.update(kw)
    if "lengths" in kw:
        base["B"] = len(kw["lengths"])
    return WorkloadSpec(**base)


SMALL = [
    dict(),
    dict(splits=1),
    dict(splits=3),
    dict(page_size=16),
    dict(page_size=16, splits=5),
    dict(lengths=[64, 65, 63, 128, 129]),
    dict(lengths=[0, 200, 0], splits=2),
    dict(lengths=[4000], splits=0),
    dict(lengths=[2500, 90], page_size=32, splits=4),
]


@pytest.mark.parametrize("case", range(len(SMALL)))
def test_mla_small_parity(case):
    w = make_workload(_mla(**SMALL[case]))
    out, lse, meta, desc = run(w)
    torch.cuda.synchronize()
    err = da.get_error(meta)
    assert err == 0, err
    got = read_meta(meta, desc)
    ref = sched_ref(w.lengths, 1, w.spec.splits, _auto_sms(desc), cpc=2)
    assert got["parts"] == ref.parts
    ref_out, ref_lse = oracle.attend(w)
    e_out, e_lse = max_err(out, lse, ref_out, ref_lse)
    assert e_out <= OUT_TOL, (SMALL[case], e_out)
    assert e_lse <= LSE_TOL, (SMALL[case], e_lse)


def test_mla_few_sms_parts_span_requests():
    w = make_workload(_mla(lengths=[700, 70, 7, 1300, 0, 64]))
    for nsm in (2, 6, 10):
        out, lse, meta, desc = run(w, num_sms=nsm)
        torch.cuda.synchronize()
        assert da.get_error(meta) == 0
        got = read_meta(meta, desc)
        ref = sched_ref(w.lengths, 1, 0, nsm, cpc=2)
        assert got["parts"] == ref.parts
        assert got["part_extra"] == expected_part_extra(ref, w.lengths, w.max_pages_per_seq * w.spec.page_size)
        ref_out, ref_lse = oracle.attend(w)
        e_out, e_lse = max_err(out, lse, ref_out, ref_lse)
        assert e_out <= OUT_TOL and e_lse <= LSE_TOL, (nsm, e_out, e_lse)


def test_mla_repeat_bitwise():
    w = make_workload(_mla(lengths=[1500, 333, 64]))
    o1, l1, _, _ = run(w)
    o2, l2, _, _ = run(w)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


# ------------------------------------------------------------------ several query tokens (drafts)

MULTI = [
    dict(s_q=2),
    dict(s_q=2, splits=3),
    dict(s_q=2, lengths=[1, 2, 64, 65, 129, 0]),
    dict(s_q=2, lengths=[2500, 90], page_size=32, splits=4),
    dict(s_q=3, lengths=[700, 3, 1300]),
]


@pytest.mark.parametrize("case", range(len(MULTI)))
def test_mla_multitoken_parity(case):
    """s_q query tokens per request on the latent format: one CTA pair per
    draft, draft j seeing the first L - s_q + 1 + j tokens; against the
    oracle's masked decode step, with the schedule bit-exact (2 s_q CTAs per
    part)."""
    kw = MULTI[case]
    w = make_workload(_mla(**kw))
    out, lse, meta, desc = run(w)
    torch.cuda.synchronize()
    assert da.get_error(meta) == 0
    sq = kw["s_q"]
    got = read_meta(meta, desc)
    ref = sched_ref(w.lengths, 1, w.spec.splits, _auto_sms(desc), cpc=2 * sq, s_q=sq)
    assert got["parts"] == ref.parts
    ref_out, ref_lse = oracle.attend_multi(w)
    e_out, e_lse = max_err(out.view(ref_out.shape), lse.view(ref_lse.shape), ref_out, ref_lse)
    assert e_out <= OUT_TOL, (kw, e_out)
    assert e_lse <= LSE_TOL, (kw, e_lse)


def test_mla_last_draft_matches_single_token():
    """The last of two drafts sees every token: it equals the one-token call on
    the same pool (same kernel arithmetic, same partition shape per CTA pair)."""
    w = make_workload(_mla(s_q=2, lengths=[1500, 333, 64], splits=2))
    out, lse, _, _ = run(w)
    single = dataclasses.replace(w, spec=w.spec.with_(s_q=1), q=w.q[:, -1].contiguous())
    o1, l1, _, _ = run(single)
    torch.cuda.synchronize()
    assert torch.equal(out[:, -1], o1) and torch.equal(lse[:, -1], l1)


def test_mla_multitoken_workload_parity():
    """The latent workload with two query tokens per request (spec2_mla_fp8),
    full launch; every request against the oracle."""
    w = make_workload(spec_by_name("spec2_mla_fp8"))
    out, lse, meta, desc = run(w)
    torch.cuda.synchronize()
    assert da.get_error(meta) == 0
    ref_out, ref_lse = oracle.attend_multi(w)
    assert not torch.isnan(ref_lse).any()
    e_out, e_lse = max_err(out.view(ref_out.shape), lse.view(ref_lse.shape), ref_out, ref_lse)
    assert e_out <= OUT_TOL, e_out
    assert e_lse <= LSE_TOL, e_lse
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()


def test_mla_bad_page_sets_error_word():
    w = make_workload(_mla(lengths=[200, 100]))
    w.block_table[0, 1] = w.num_pages + 7
    out, lse, meta, _ = run(w)
    torch.cuda.synchronize()
    assert da.get_error(meta) & da.DA_DEV_BAD_PAGE


def test_mla_workload_parity():
    """The 32-request latent-token workload (lengths log-uniform in [4096, 131072]),
    full launch; every request against the oracle."""
    w = make_workload(spec_by_name("mla_fp8"))
    out, lse, meta, desc = run(w)
    torch.cuda.synchronize()
    assert da.get_error(meta) == 0
    got = read_meta(meta, desc)
    ref = sched_ref(w.lengths, 1, 0, _auto_sms(desc), cpc=2)
    assert got["parts"] == ref.parts and got["split_offset"] == ref.split_offset
    ref_out, ref_lse = oracle.attend(w)
    assert not torch.isnan(ref_lse).any()
    e_out, e_lse = max_err(out, lse, ref_out, ref_lse)
    assert e_out <= OUT_TOL, e_out
    assert e_lse <= LSE_TOL, e_lse
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
