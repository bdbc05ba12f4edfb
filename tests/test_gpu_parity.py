"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle on
the same seeded inputs. Integer metadata bit-exact; lse within 1e-4; out
within 2e-2 (bf16 output, fp32 accumulation)."""
import math
import random

import pytest
import torch

import oracle
import paged_kv_cache_60_gb300 as da
from oracle.sched_ref import sched_ref
from workloads import CONFIGS, WorkloadSpec, make_workload, spec_by_name, KV_BF16, KV_FP8
from workloads.gen import repermute_pages

from gpu_util import (LSE_TOL, OUT_TOL, DeviceWorkload, device_sms, ensure_built, expected_part_extra,
                      make_desc, max_err, read_meta, run)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    ensure_built()
    oracle.build_oracle()


def _spec(**kw):
    base = dict(name="t", B=3, H_kv=2, G=8, D_qk=128, D_v=128, page_size=16,
                lengths=[517, 1, 300], splits=0, extra_pages=5, seed=11)
    base.update(kw)
    return WorkloadSpec(**base)


# ------------------------------------------------------------------ metadata

SEQLEN_CASES = [
    [256], [1536] * 8, [0, 1, 63, 64, 65, 127, 128, 129], [5000, 17, 0, 3000, 64 * 37],
    [1] * 40, [0, 0, 0], [8192, 1024, 4096, 2048] * 8,
]


@pytest.mark.parametrize("seqlens", SEQLEN_CASES)
@pytest.mark.parametrize("splits", [0, 1, 3, 8])
@pytest.mark.parametrize("H_kv", [1, 4, 8])
def test_sched_meta_bit_exact(seqlens, splits, H_kv):
    B = len(seqlens)
    P = 64
    maxp = max(1, max(-(-L // P) for L in seqlens))
    desc = da.Desc.make(B=B, H_kv=H_kv, G=8, D_qk=128, D_v=128, page_size=P, max_pages_per_seq=maxp,
                        num_pages=B * maxp, kv_dtype=KV_BF16, splits=splits)
    meta = torch.empty(da.sched_meta_bytes(desc), dtype=torch.uint8, device="cuda")
    meta.fill_(0xAB)
    sl = torch.tensor(seqlens, dtype=torch.int32, device="cuda")
    da.sched_meta(desc, sl, meta)
    got = read_meta(meta, desc)
    ref = sched_ref(seqlens, H_kv, splits, device_sms(), cpc=1)
    h = got["header"]
    assert h[0] == 0x44414d31 and h[1] == B and h[5] == ref.num_parts
    assert h[8] == ref.total_chunks and h[9] == ref.total_splits and h[10] == ref.per and h[11] == 0
    assert got["parts"] == ref.parts
    assert got["part_extra"] == expected_part_extra(ref, seqlens, maxp * P)
    assert got["chunk_offset"] == ref.chunk_offset
    assert got["split_offset"] == ref.split_offset
    assert got["num_splits"] == ref.num_splits


def test_sched_meta_large_batch_bit_exact():
    rnd = random.Random(5)
    seqlens = [rnd.randint(0, 9000) for _ in range(3000)]
    P = 32
    maxp = max(-(-L // P) for L in seqlens)
    for splits in (0, 2):
        desc = da.Desc.make(B=3000, H_kv=1, G=8, D_qk=128, D_v=128, page_size=P, max_pages_per_seq=maxp,
                            num_pages=1 << 20, kv_dtype=KV_BF16, splits=splits)
        meta = torch.zeros(da.sched_meta_bytes(desc), dtype=torch.uint8, device="cuda")
        da.sched_meta(desc, torch.tensor(seqlens, dtype=torch.int32, device="cuda"), meta)
        got = read_meta(meta, desc)
        ref = sched_ref(seqlens, 1, splits, device_sms())
        assert got["parts"] == ref.parts and got["split_offset"] == ref.split_offset
        assert got["chunk_offset"] == ref.chunk_offset and got["num_splits"] == ref.num_splits
        assert got["part_extra"] == expected_part_extra(ref, seqlens, maxp * P)


# ------------------------------------------------------------------ attention, small cases

SMALL = [
    dict(),
    dict(splits=1), dict(splits=4), dict(splits=7),
    dict(D_qk=64, D_v=64), dict(D_qk=64, D_v=64, splits=3, page_size=8),
    dict(page_size=8), dict(page_size=32), dict(page_size=64), dict(page_size=128), dict(page_size=256),
    dict(kv_dtype=KV_FP8), dict(kv_dtype=KV_FP8, splits=5, page_size=32), dict(kv_dtype=KV_FP8, page_size=256),
    dict(lengths=[64, 65, 63, 1, 2, 129], B=6, H_kv=1),
    dict(lengths=[3000, 17], B=2, H_kv=3, page_size=64),
    dict(lengths=[1000], B=1, H_kv=1, splits=16, page_size=16),
]


@pytest.mark.parametrize("case", range(len(SMALL)))
def test_small_parity(case):
    kw = SMALL[case]
    spec = _spec(**kw)
    if "lengths" in kw:
        spec = spec.with_(B=len(kw["lengths"]))
    w = make_workload(spec)
    out, lse, meta, desc = run(w)
    torch.cuda.synchronize()
    assert da.get_error(meta) == 0
    ref_out, ref_lse = oracle.attend(w)
    e_out, e_lse = max_err(out, lse, ref_out, ref_lse)
    assert e_out <= OUT_TOL, (kw, e_out)
    assert e_lse <= LSE_TOL, (kw, e_lse)


def test_auto_mode_with_few_sms_spans_requests():
    # a small SM count makes parts cross request boundaries
    w = make_workload(_spec(lengths=[700, 70, 7, 1300, 0, 64], B=6, H_kv=2, page_size=32))
    for nsm in (2, 6, 10):
        out, lse, meta, desc = run(w, num_sms=nsm)
        ref_out, ref_lse = oracle.attend(w)
        e_out, e_lse = max_err(out, lse, ref_out, ref_lse)
        assert e_out <= OUT_TOL and e_lse <= LSE_TOL, (nsm, e_out, e_lse)


@pytest.mark.parametrize("splits", [0, 2])
def test_empty_requests(splits):
    w = make_workload(_spec(lengths=[0, 200, 0], B=3, splits=splits))
    out, lse, meta, _ = run(w)
    o = out.float().cpu()
    l = lse.cpu()
    assert torch.all(o[0] == 0) and torch.all(o[2] == 0)
    assert torch.all(torch.isneginf(l[0])) and torch.all(torch.isneginf(l[2]))
    ref_out, ref_lse = oracle.attend(w)
    e_out, e_lse = max_err(out, lse, ref_out, ref_lse)
    assert e_out <= OUT_TOL and e_lse <= LSE_TOL


# ------------------------------------------------------------------ invariants on the GPU

@pytest.mark.parametrize("kv", [KV_BF16, KV_FP8])
def test_page_permutation_bitwise(kv):
    w = make_workload(_spec(kv_dtype=kv, lengths=[900, 33, 400], page_size=16, extra_pages=20))
    w2 = repermute_pages(w, seed=3)
    o1, l1, _, _ = run(w)
    o2, l2, _, _ = run(w2)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_repeat_runs_bitwise():
    w = make_workload(_spec(lengths=[2000, 999, 5], page_size=32))
    dw = DeviceWorkload(w)
    o1, l1, meta, desc = run(w, dw=dw)
    for _ in range(3):
        o2, l2, _, _ = run(w, dw=dw, meta=meta, desc=desc)
        assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_graph_replay_100():
    w = make_workload(_spec(lengths=[1536] * 4, B=4, H_kv=4, D_qk=64, D_v=64, page_size=256, splits=8))
    dw = DeviceWorkload(w)
    desc = make_desc(w)
    meta = torch.empty(da.sched_meta_bytes(desc), dtype=torch.uint8, device="cuda")
    out = torch.empty(4, 32, 64, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(4, 32, dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        da.sched_meta(desc, dw.cache_seqlens, meta)
        run(w, dw=dw, meta=meta, desc=desc, out=out, lse=lse)   # warm-up outside the capture
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            da.sched_meta(desc, dw.cache_seqlens, meta)
            run(w, dw=dw, meta=meta, desc=desc, out=out, lse=lse)
    ref_out, ref_lse = oracle.attend(w)
    first = None
    for _ in range(100):
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        if first is None:
            first = (out.clone(), lse.clone())
            e_out, e_lse = max_err(out, lse, ref_out, ref_lse)
            assert e_out <= OUT_TOL and e_lse <= LSE_TOL
        else:
            assert torch.equal(out, first[0]) and torch.equal(lse, first[1])


# ------------------------------------------------------------------ device-detected errors

def test_bad_page_id_sets_error_word():
    w = make_workload(_spec(lengths=[300, 100], B=2))
    w.block_table[1, 2] = w.num_pages + 7
    out, lse, meta, _ = run(w)
    err = da.get_error(meta)
    assert err & da.DA_DEV_BAD_PAGE
    # the other request is unaffected
    ref_out, ref_lse = oracle.attend(w, heads=[(0, 0), (0, 1)])
    e_out, e_lse = max_err(out, lse, ref_out, ref_lse)
    assert e_out <= OUT_TOL and e_lse <= LSE_TOL


def test_meta_from_other_desc_is_refused_on_device():
    w = make_workload(_spec())
    out, lse, meta, desc = run(w)
    desc2 = make_desc(w, splits=2)
    meta2 = torch.zeros(max(da.sched_meta_bytes(desc2), da.sched_meta_bytes(desc)), dtype=torch.uint8,
                        device="cuda")
    da.sched_meta(desc, DeviceWorkload(w).cache_seqlens, meta2)     # built for desc (auto)
    run(w, desc=desc2, meta=meta2)                                   # used with desc2 (fixed)
    assert da.get_error(meta2) & da.DA_DEV_META_MISMATCH


def test_too_long_sequence_is_clamped_and_flagged():
    w = make_workload(_spec(lengths=[300, 100], B=2))
    dw = DeviceWorkload(w)
    dw.cache_seqlens[1] = w.max_pages_per_seq * w.spec.page_size + 50
    out, lse, meta, _ = run(w, dw=dw)
    assert da.get_error(meta) & da.DA_DEV_SEQ_TOO_LONG


# ------------------------------------------------------------------ the five workloads

@pytest.mark.parametrize("name", ["tiny_gqa_bf16", "gqa_bf16_b8", "mixed_gqa_bf16", "fp8_gqa"])
def test_workload_parity(name):
    """The full-size workloads in the benchmark's launch configuration: every
    output row against the oracle (the oracle computes every (request, KV
    head) unit)."""
    w = make_workload(spec_by_name(name))
    out, lse, meta, desc = run(w)
    torch.cuda.synchronize()
    assert da.get_error(meta) == 0
    got = read_meta(meta, desc)
    ref = sched_ref(w.lengths, w.spec.H_kv, w.spec.splits, device_sms())
    assert got["parts"] == ref.parts and got["split_offset"] == ref.split_offset
    ref_out, ref_lse = oracle.attend(w)
    assert not torch.isnan(ref_lse).any()
    e_out, e_lse = max_err(out, lse, ref_out, ref_lse)
    assert e_out <= OUT_TOL, (name, e_out)
    assert e_lse <= LSE_TOL, (name, e_lse)
    # every output of the full run is finite (poisoned slots never read)
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()


# ------------------------------------------------------------------ pool placement

@pytest.mark.parametrize("kv", [KV_BF16, KV_FP8])
def test_v_pool_below_k_pool(kv):
    # one buffer, V in the lower half and K in the upper half
    w = make_workload(_spec(kv_dtype=kv, lengths=[700, 90, 300]))
    dw = DeviceWorkload(w)
    both = torch.empty((2,) + tuple(w.k_pool.shape), dtype=w.k_pool.dtype, device="cuda")
    both[0].copy_(dw.v_pool)
    both[1].copy_(dw.k_pool)
    dw.v_pool, dw.k_pool = both[0], both[1]
    out, lse, _, _ = run(w, dw=dw)
    ref_out, ref_lse = oracle.attend(w)
    e_out, e_lse = max_err(out, lse, ref_out, ref_lse)
    assert e_out <= OUT_TOL and e_lse <= LSE_TOL


@pytest.mark.parametrize("kv", [KV_BF16, KV_FP8])
def test_same_buffer_for_k_and_v(kv):
    # K = V: the pools cannot share one tensor map, each gets its own
    w = make_workload(_spec(kv_dtype=kv, lengths=[700, 90, 300]))
    w.v_pool = w.k_pool
    if w.k_scale is not None:
        w.v_scale = w.k_scale
    dw = DeviceWorkload(w)
    dw.v_pool = dw.k_pool
    out, lse, _, _ = run(w, dw=dw)
    ref_out, ref_lse = oracle.attend(w)
    e_out, e_lse = max_err(out, lse, ref_out, ref_lse)
    assert e_out <= OUT_TOL and e_lse <= LSE_TOL
