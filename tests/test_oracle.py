"""Pins for the float64 oracle: closed forms, invariants, library decodes and
the pages' printed values. None of these re-types the oracle's own formula."""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from workloads import WorkloadSpec, make_workload, KV_BF16, KV_FP8, KV_MLA656
from workloads.gen import Workload, repermute_pages, MLA_ROW_BYTES

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _small(**kw):
    base = dict(name="t", B=2, H_kv=2, G=4, D_qk=16, D_v=16, page_size=8, lengths=[37, 20],
                splits=0, extra_pages=3, seed=7)
    base.update(kw)
    return WorkloadSpec(**base)


def _bf16(x):
    return torch.tensor(x, dtype=torch.float64).to(torch.bfloat16)


def _set_logical(w, b, t, h, k=None, v=None):
    """Write logical token t of (b, h); uses the generator's own placement."""
    P = w.spec.page_size
    page = int(w.block_table[b, t // P])
    if k is not None:
        w.k_pool[page, t % P, h] = k
    if v is not None:
        w.v_pool[page, t % P, h] = v


# ---------------------------------------------------------------- element decodes

def test_e4m3_points_from_pages_and_definition(oracle_lib):
    with open(os.path.join(GOLDEN, "e4m3_points.txt")) as f:
        rows = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    assert len(rows) >= 10
    for code, val in rows:
        assert oracle.e4m3_value(int(code, 16)) == float(val), code
    assert math.isnan(oracle.e4m3_value(0x7F)) and math.isnan(oracle.e4m3_value(0xFF))


def test_e4m3_all_codes_match_torch_decode(oracle_lib):
    codes = torch.arange(256, dtype=torch.uint8)
    lib_vals = codes.view(torch.float8_e4m3fn).to(torch.float64)
    for c in range(256):
        a = oracle.e4m3_value(c)
        b = float(lib_vals[c])
        if math.isnan(b):
            assert math.isnan(a), c
        else:
            assert a == b, (c, a, b)


def test_bf16_decode_matches_torch(oracle_lib):
    g = torch.Generator().manual_seed(3)
    bits = torch.randint(0, 1 << 16, (4000,), generator=g, dtype=torch.int32)
    vals = bits.to(torch.int16).view(torch.bfloat16).to(torch.float64)
    for i in range(bits.numel()):
        a = oracle.bf16_value(int(bits[i]))
        b = float(vals[i])
        assert (math.isnan(a) and math.isnan(b)) or a == b


# ---------------------------------------------------------------- closed forms

def test_single_token_returns_v0_and_its_score(oracle_lib):
    spec = _small(lengths=[1, 1], B=2)
    w = make_workload(spec)
    q = torch.zeros(2, spec.H_q, spec.D_qk, dtype=torch.bfloat16)
    q[:, :, 0] = 1.0
    q[:, :, 1] = -2.0
    w.q = q
    for b in range(2):
        for h in range(spec.H_kv):
            k = torch.zeros(spec.D_qk)
            k[0], k[1] = 3.0, 0.5
            _set_logical(w, b, 0, h, k=k.to(torch.bfloat16),
                         v=_bf16([float(i + 10 * b + 100 * h) for i in range(spec.D_v)]))
    out, lse = oracle.attend(w)
    score = (1.0 * 3.0 + (-2.0) * 0.5) * w.softmax_scale
    for b in range(2):
        for h in range(spec.H_kv):
            exp_v = torch.tensor([float(i + 10 * b + 100 * h) for i in range(spec.D_v)],
                                 dtype=torch.float64)
            for g in range(spec.G):
                assert torch.equal(out[b, h * spec.G + g], exp_v)
                assert lse[b, h * spec.G + g] == pytest.approx(score, abs=1e-15)


def test_zero_query_gives_mean_of_v_and_log_length(oracle_lib):
    spec = _small(lengths=[37, 20])
    w = make_workload(spec)
    w.q = torch.zeros_like(w.q)
    # V known by construction (small integers: exact in bf16)
    for b, L in enumerate(spec.lengths):
        for t in range(L):
            for h in range(spec.H_kv):
                _set_logical(w, b, t, h, v=_bf16([float((t * 3 + d + h) % 11 - 5) for d in range(spec.D_v)]))
    out, lse = oracle.attend(w)
    for b, L in enumerate(spec.lengths):
        for h in range(spec.H_kv):
            mean = torch.tensor([sum(float((t * 3 + d + h) % 11 - 5) for t in range(L)) / L
                                 for d in range(spec.D_v)], dtype=torch.float64)
            for g in range(spec.G):
                assert torch.allclose(out[b, h * spec.G + g], mean, rtol=0, atol=1e-13)
                assert lse[b, h * spec.G + g] == pytest.approx(math.log(L), abs=1e-13)


def test_two_tokens_closed_form(oracle_lib):
    # s0 = 0, s1 = ln 3 (scale chosen so the product is exact): weights 1/4, 3/4
    spec = _small(B=1, lengths=[2], H_kv=1, G=2, softmax_scale=math.log(3.0) / 4.0)
    w = make_workload(spec)
    q = torch.zeros_like(w.q)
    q[0, :, 0] = 2.0
    w.q = q
    k1 = torch.zeros(spec.D_qk)
    k1[0] = 2.0
    _set_logical(w, 0, 0, 0, k=torch.zeros(spec.D_qk).to(torch.bfloat16), v=_bf16([4.0] * spec.D_v))
    _set_logical(w, 0, 1, 0, k=k1.to(torch.bfloat16), v=_bf16([-8.0] * spec.D_v))
    out, lse = oracle.attend(w)
    expect = 0.25 * 4.0 + 0.75 * (-8.0)
    assert torch.allclose(out[0], torch.full_like(out[0], expect), atol=1e-14, rtol=0)
    assert lse[0, 0] == pytest.approx(math.log(4.0), abs=1e-14)


def test_dominant_token_selects_its_value(oracle_lib):
    spec = _small(lengths=[37, 20])
    w = make_workload(spec)
    q = torch.zeros_like(w.q)
    q[:, :, 3] = 8.0
    w.q = q
    picks = {(0, 0): 29, (0, 1): 5, (1, 0): 19, (1, 1): 0}
    for (b, h), j in picks.items():
        for t in range(spec.lengths[b]):
            k = torch.zeros(spec.D_qk)
            k[3] = 64.0 if t == j else 0.0
            _set_logical(w, b, t, h, k=k.to(torch.bfloat16),
                         v=_bf16([float(t + 0.5 * d) for d in range(spec.D_v)]))
    out, lse = oracle.attend(w)
    for (b, h), j in picks.items():
        want = torch.tensor([float(j + 0.5 * d) for d in range(spec.D_v)], dtype=torch.float64)
        for g in range(spec.G):
            assert torch.allclose(out[b, h * spec.G + g], want, atol=1e-9, rtol=0)
            assert lse[b, h * spec.G + g] == pytest.approx(512.0 * w.softmax_scale, abs=1e-9)


def test_unit_value_gives_unit_output(oracle_lib):
    spec = _small()
    w = make_workload(spec)
    for b, L in enumerate(spec.lengths):
        for t in range(L):
            for h in range(spec.H_kv):
                _set_logical(w, b, t, h, v=_bf16([1.0] * spec.D_v))
    out, _ = oracle.attend(w)
    assert torch.allclose(out, torch.ones_like(out), atol=1e-13, rtol=0)


# ---------------------------------------------------------------- invariants

def test_page_permutation_invariance_bitwise(oracle_lib):
    w = make_workload(_small(lengths=[61, 17], page_size=4, extra_pages=9))
    w2 = repermute_pages(w, seed=99)
    assert not torch.equal(w.block_table, w2.block_table)
    o1, l1 = oracle.attend(w)
    o2, l2 = oracle.attend(w2)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_token_duplication_keeps_output_and_adds_ln2(oracle_lib):
    spec = _small(B=1, lengths=[19], H_kv=1, G=3, D_qk=8, D_v=8, page_size=4)
    w = make_workload(spec)
    spec2 = spec.with_(lengths=[38])
    w2 = make_workload(spec2)
    w2.q = w.q.clone()
    for t in range(19):
        page = int(w.block_table[0, t // 4])
        k, v = w.k_pool[page, t % 4, 0], w.v_pool[page, t % 4, 0]
        _set_logical(w2, 0, t, 0, k=k, v=v)
        _set_logical(w2, 0, t + 19, 0, k=k, v=v)
    o1, l1 = oracle.attend(w)
    o2, l2 = oracle.attend(w2)
    assert torch.allclose(o1, o2, atol=1e-13, rtol=0)
    assert torch.allclose(l2, l1 + math.log(2.0), atol=1e-13, rtol=0)


def test_value_scaling_scales_output(oracle_lib):
    w = make_workload(_small())
    o1, l1 = oracle.attend(w)
    w.v_pool = w.v_pool * 2          # exact in bf16
    o2, l2 = oracle.attend(w)
    assert torch.equal(o2, 2 * o1) and torch.equal(l1, l2)


def test_gqa_heads_equal_separate_mha_problems(oracle_lib):
    spec = _small(B=1, lengths=[45], H_kv=1, G=4)
    w = make_workload(spec)
    out, lse = oracle.attend(w)
    for g in range(spec.G):
        w1 = Workload(spec=spec.with_(G=1), lengths=w.lengths, num_pages=w.num_pages,
                      max_pages_per_seq=w.max_pages_per_seq, q=w.q[:, g:g + 1].clone(),
                      k_pool=w.k_pool, v_pool=w.v_pool, k_scale=None, v_scale=None,
                      block_table=w.block_table, cache_seqlens=w.cache_seqlens)
        o1, l1 = oracle.attend(w1)
        assert torch.equal(o1[0, 0], out[0, g]) and torch.equal(l1[0, 0], lse[0, g])


@pytest.mark.parametrize("splits", [1, 2, 3, 8, 0])
def test_split_then_combine_equals_unsplit(oracle_lib, splits):
    spec = _small(B=4, lengths=[300, 1, 64, 129], page_size=16, splits=splits)
    w = make_workload(spec)
    ref = oracle.sched_ref(w.lengths, spec.H_kv, splits, num_sms=7)
    o1, l1 = oracle.attend(w)
    o2, l2 = oracle.attend_split_combine(w, ref)
    assert torch.allclose(o1, o2, atol=1e-12, rtol=0)
    assert torch.allclose(l1, l2, atol=1e-12, rtol=0)


def test_empty_request_and_empty_splits(oracle_lib):
    spec = _small(B=3, lengths=[0, 70, 0], page_size=16, splits=4)
    w = make_workload(spec)
    ref = oracle.sched_ref(w.lengths, spec.H_kv, 4, num_sms=7)
    out, lse = oracle.attend_split_combine(w, ref)
    assert torch.all(out[0] == 0) and torch.all(torch.isneginf(lse[0]))
    assert torch.all(out[2] == 0) and torch.all(torch.isneginf(lse[2]))
    o1, l1 = oracle.attend(w)
    assert torch.allclose(out[1], o1[1], atol=1e-12, rtol=0)


def test_combine_reproduces_rescale_example(oracle_lib):
    vals = {}
    with open(os.path.join(GOLDEN, "rescale_example.txt")) as f:
        for ln in f:
            if ln.strip() and not ln.startswith("#"):
                k, v = ln.split()
                vals[k] = float(v)
    # two partials each of one token: scores old_max and new_max, values 1 and 0
    o = torch.tensor([[1.0], [0.0]], dtype=torch.float64)
    l = torch.tensor([vals["old_max"], vals["new_max"]], dtype=torch.float64)
    out, lse = oracle.combine(o, l)
    r = vals["rescale"]
    assert r == pytest.approx(math.exp(vals["old_max"] - vals["new_max"]), rel=1e-15)
    # weight of the old partial relative to the new one is the printed rescale factor
    assert out[0] == pytest.approx(r / (1.0 + r), rel=1e-14)
    assert lse == pytest.approx(vals["new_max"] + math.log(1.0 + r), rel=1e-14)


# ---------------------------------------------------------------- FP8 formats

def _as_f64_workload(w, kd, vd):
    spec = w.spec.with_(kv_dtype=3)
    return Workload(spec=spec, lengths=w.lengths, num_pages=w.num_pages,
                    max_pages_per_seq=w.max_pages_per_seq, q=w.q, k_pool=kd.contiguous(),
                    v_pool=vd.contiguous(), k_scale=None, v_scale=None,
                    block_table=w.block_table, cache_seqlens=w.cache_seqlens)


def test_fp8_per_tensor_equals_predequantised(oracle_lib):
    spec = _small(kv_dtype=KV_FP8, D_qk=32, D_v=32)
    w = make_workload(spec)
    ks = w.k_scale.to(torch.float64).view(1, 1, -1, 1)
    vs = w.v_scale.to(torch.float64).view(1, 1, -1, 1)
    kd = w.k_pool.view(torch.float8_e4m3fn).to(torch.float64) * ks
    vd = w.v_pool.view(torch.float8_e4m3fn).to(torch.float64) * vs
    o1, l1 = oracle.attend(w)
    o2, l2 = oracle.attend(_as_f64_workload(w, kd, vd))
    assert torch.allclose(o1, o2, atol=1e-13, rtol=0) and torch.allclose(l1, l2, atol=1e-13, rtol=0)


def test_mla_token_layout_matches_page(oracle_lib):
    rows = {}
    with open(os.path.join(GOLDEN, "mla_token_layout.txt")) as f:
        for ln in f:
            if ln.strip() and not ln.startswith("#"):
                p = ln.split()
                rows[p[0]] = p[1:]
    assert int(rows["token"][2]) == MLA_ROW_BYTES == 656
    assert sum(int(rows[k][2]) for k in ("nope_e4m3", "scale_f32", "rope_bf16")) == 656
    assert int(rows["scale_block"][0]) * int(rows["scale_f32"][0]) == int(rows["nope_e4m3"][0])


def test_mla656_equals_predequantised(oracle_lib):
    spec = WorkloadSpec(name="m", B=2, H_kv=1, G=3, D_qk=576, D_v=512, page_size=8,
                        kv_dtype=KV_MLA656, lengths=[21, 9], extra_pages=2, seed=5)
    w = make_workload(spec)
    raw = w.k_pool.reshape(-1, 656)
    rope = raw[:, 528:].contiguous().view(torch.bfloat16).to(torch.float64)
    # the page's chain: float32 value times float32 scale, then bfloat16
    nope32 = raw[:, :512].contiguous().view(torch.float8_e4m3fn).to(torch.float32)
    deq = (nope32 * raw[:, 512:528].contiguous().view(torch.float32).repeat_interleave(128, dim=1))
    k = torch.cat([deq.to(torch.bfloat16).to(torch.float64), rope], dim=1)
    kd = k.reshape(w.num_pages, 8, 1, 576)
    vd = k[:, :512].reshape(w.num_pages, 8, 1, 512)
    o1, l1 = oracle.attend(w)
    o2, l2 = oracle.attend(_as_f64_workload(w, kd, vd))
    assert torch.isfinite(o1).all()
    assert torch.allclose(o1, o2, atol=1e-13, rtol=0) and torch.allclose(l1, l2, atol=1e-13, rtol=0)


def test_poisoned_slots_are_never_read(oracle_lib):
    # every slot outside the valid tokens is NaN; a finite result proves none was read
    for kv in (KV_BF16, KV_FP8):
        w = make_workload(_small(kv_dtype=kv, lengths=[37, 5], page_size=16, extra_pages=4))
        out, lse = oracle.attend(w)
        assert torch.isfinite(out).all() and torch.isfinite(lse).all()


def test_bad_page_id_is_reported(oracle_lib):
    w = make_workload(_small())
    w.block_table[0, 1] = w.num_pages + 5
    with pytest.raises(ValueError):
        oracle.attend(w)


def test_query_head_order_h_times_g_plus_g(oracle_lib):
    # query head h*G+g belongs to KV head h (XQA page, GQA layout section):
    # give each global query head a one-hot query that selects its own token
    spec = _small(B=1, lengths=[16], H_kv=3, G=2, D_qk=8, D_v=8, page_size=4)
    w = make_workload(spec)
    q = torch.zeros_like(w.q)
    for hq in range(spec.H_q):
        q[0, hq, hq] = 8.0
    w.q = q
    for h in range(spec.H_kv):
        for t in range(16):
            k = torch.zeros(8)
            if t < spec.H_q:
                k[t] = 64.0
            _set_logical(w, 0, t, h, k=k.to(torch.bfloat16),
                         v=_bf16([float(100 * h + t)] * 8))
    out, _ = oracle.attend(w)
    for h in range(spec.H_kv):
        for g in range(spec.G):
            hq = h * spec.G + g
            assert torch.allclose(out[0, hq], torch.full((8,), float(100 * h + hq), dtype=torch.float64),
                                  atol=1e-9, rtol=0)


def test_mla_dequant_rounds_like_torch_float32_then_bf16(oracle_lib):
    # single-token requests: out equals the token's dequantised V row exactly
    spec = WorkloadSpec(name="m1", B=3, H_kv=1, G=2, D_qk=576, D_v=512, page_size=8,
                        kv_dtype=KV_MLA656, lengths=[1, 1, 1], seed=9)
    w = make_workload(spec)
    out, _ = oracle.attend(w)
    for b in range(3):
        page = int(w.block_table[b, 0])
        raw = w.k_pool[page, 0, 0]
        v32 = raw[:512].contiguous().view(torch.float8_e4m3fn).to(torch.float32)
        sc = raw[512:528].contiguous().view(torch.float32).repeat_interleave(128)
        want = (v32 * sc).to(torch.bfloat16).to(torch.float64)
        assert torch.equal(out[b, 0], want) and torch.equal(out[b, 1], want)
