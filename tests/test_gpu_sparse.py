"""GPU parity for sparse top-k decode on the 656-byte latent-token format:
each request attends over its listed token positions (invalid entries
skipped, repeats counted) against oracle.attend_sparse; the schedule is
bit-exact against the scheduling oracle; with the full in-order list the
sparse kernel reproduces the dense kernel bit for bit."""
import dataclasses

import pytest
import torch

import oracle
import paged_kv_cache_60_gb300 as da
from oracle.sched_ref import sched_ref
from workloads import WorkloadSpec, make_workload, spec_by_name, KV_MLA656

from gpu_util import LSE_TOL, OUT_TOL, DeviceWorkload, device_sms, ensure_built, make_desc, max_err, read_meta, run

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    ensure_built()
    oracle.build_oracle()


def _spec(**kw):
    base = dict(name="s", B=6, H_kv=1, G=128, D_qk=576, D_v=512, page_size=16, kv_dtype=KV_MLA656,
                lengths=[1, 30, 77, 0, 200, 1000], splits=0, extra_pages=3, seed=51, topk=100)
    base.update(kw)
    if "lengths" in kw:
        base["B"] = len(kw["lengths"])
    return WorkloadSpec(**base)


def _check(w):
    out, lse, meta, _ = run(w)
    torch.cuda.synchronize()
    assert da.get_error(meta) == 0
    ref_out, ref_lse = oracle.attend_sparse(w)
    e_out, e_lse = max_err(out, lse, ref_out, ref_lse)
    assert e_out <= OUT_TOL and e_lse <= LSE_TOL, (e_out, e_lse)


CASES = [
    dict(),
    dict(splits=2),
    dict(page_size=64, topk=64),
    dict(page_size=64, topk=200, splits=1),
    dict(lengths=[5000, 3000], topk=2048),
    dict(lengths=[300, 300, 300], topk=300, page_size=32),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_sparse_parity(case):
    _check(make_workload(_spec(**CASES[case])))


def test_sparse_invalid_and_repeated_entries():
    w = make_workload(_spec())
    idx = w.indices.clone()
    idx[4, :10] = -1                 # padding inside the list
    idx[5, 5] = 5000                 # a position past the request
    idx[5, 6] = -3
    idx[5, 7] = idx[5, 8]            # a position listed twice
    idx[0, :] = -1                   # a request with no valid entry: out 0, lse -inf
    _check(dataclasses.replace(w, indices=idx))


def test_full_in_order_list_equals_dense_bitwise():
    spec = _spec(lengths=[300, 300, 300, 300], topk=300, page_size=32)
    w = make_workload(spec)
    idx = torch.full((spec.B, spec.topk), -1, dtype=torch.int32)
    for b, L in enumerate(w.lengths):
        idx[b, :L] = torch.arange(L, dtype=torch.int32)
    ws = dataclasses.replace(w, indices=idx)
    o_s, l_s, _, _ = run(ws)
    dense = dataclasses.replace(w, spec=spec.with_(topk=0), indices=None)
    o_d, l_d, _, _ = run(dense)
    torch.cuda.synchronize()
    # the same schedule (topk = L for every request), the same tokens in the same order
    assert torch.equal(o_s, o_d) and torch.equal(l_s, l_d)


@pytest.mark.parametrize("splits", [0, 3])
def test_sparse_schedule_bitexact(splits):
    spec = _spec(splits=splits, topk=300)
    w = make_workload(spec)
    dw = DeviceWorkload(w)
    desc = make_desc(w)
    meta = torch.empty(da.sched_meta_bytes(desc), dtype=torch.uint8, device="cuda")
    da.sched_meta(desc, dw.cache_seqlens, meta)
    torch.cuda.synchronize()
    got = read_meta(meta, desc)
    nsm = device_sms() if splits > 0 else 2 * da.num_parts(desc)
    ref = sched_ref(w.lengths, 1, splits, num_sms=nsm, cpc=2, topk=300)
    assert got["chunk_offset"] == ref.chunk_offset
    assert got["parts"] == ref.parts
    assert got["num_splits"] == ref.num_splits


@pytest.mark.parametrize("name", ["sparse_mla_topk2048", "sparse_mla_topk32768"])
def test_sparse_bench_workload(name):
    """The top-k workloads at full size: every request against the oracle."""
    spec = spec_by_name(name)
    w = make_workload(spec)
    out, lse, meta, _ = run(w)
    torch.cuda.synchronize()
    assert da.get_error(meta) == 0
    ref_out, ref_lse = oracle.attend_sparse(w)
    assert not torch.isnan(ref_lse).any()
    e_out, e_lse = max_err(out, lse, ref_out, ref_lse)
    assert e_out <= OUT_TOL and e_lse <= LSE_TOL, (e_out, e_lse)


def test_sparse_needs_indices_and_the_latent_format():
    ensure_built()
    w = make_workload(_spec())
    dw = DeviceWorkload(w)
    desc = make_desc(w)
    meta = torch.empty(da.sched_meta_bytes(desc), dtype=torch.uint8, device="cuda")
    out = torch.empty(6, 128, 512, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(6, 128, dtype=torch.float32, device="cuda")
    with pytest.raises(da.DecodeAttnError):
        da.fwd(desc, dw.q, dw.k_pool, None, None, None, dw.block_table, dw.cache_seqlens, meta, out, lse)
    gqa = da.Desc.make(B=2, H_kv=2, G=8, D_qk=128, D_v=128, page_size=16, max_pages_per_seq=4, num_pages=10,
                       topk=64)
    with pytest.raises(da.DecodeAttnError):
        da.sched_meta_bytes(gqa)
