"""Pins for the multi-token (linear draft chain) oracle, oracle.attend_multi:
a masked-matrix formulation with torch's softmax / logsumexp, the reduction of
the last draft to single-token decode, and causality (a draft never sees the
tokens after it)."""
import dataclasses

import pytest
import torch

import oracle
from workloads import WorkloadSpec, make_workload, KV_BF16, KV_FP8, KV_MLA656


def _spec(**kw):
    base = dict(name="t", B=6, H_kv=2, G=4, D_qk=16, D_v=16, page_size=8, lengths=[1, 2, 3, 9, 17, 0],
                splits=0, extra_pages=3, seed=5, s_q=3)
    base.update(kw)
    return WorkloadSpec(**base)


def _kv_rows(w, b, h):
    """Dequantised K [L, D_qk] and V [L, D_v] of (b, h) in float64, gathered
    through the block table."""
    s = w.spec
    P = s.page_size
    L = w.lengths[b]
    ks, vs = [], []
    for t in range(L):
        page = int(w.block_table[b, t // P])
        k = w.k_pool[page, t % P, h]
        v = w.v_pool[page, t % P, h]
        if s.kv_dtype == KV_FP8:
            k = k.view(torch.float8_e4m3fn).double() * float(w.k_scale[h])
            v = v.view(torch.float8_e4m3fn).double() * float(w.v_scale[h])
        ks.append(k.double())
        vs.append(v.double())
    if not ks:
        return torch.zeros(0, s.D_qk, dtype=torch.float64), torch.zeros(0, s.D_v, dtype=torch.float64)
    return torch.stack(ks), torch.stack(vs)


@pytest.mark.parametrize("kv_dtype,s_q,window,sinks", [
    (KV_BF16, 3, 0, False), (KV_FP8, 3, 0, False), (KV_BF16, 1, 5, False), (KV_BF16, 3, 4, True),
    (KV_FP8, 2, 7, True), (KV_BF16, 1, 0, True),
])
def test_masked_matrix_formulation(oracle_lib, kv_dtype, s_q, window, sinks):
    """Scores as one matrix per (request, query head): rows = query tokens,
    columns = [sink] + tokens, invisible tokens set to -inf; torch's softmax
    and logsumexp give the weights and lse; the sink column carries no value."""
    spec = _spec(kv_dtype=kv_dtype, s_q=s_q, window=window, sinks=sinks)
    w = make_workload(spec, poison=False)
    out, lse = oracle.attend_multi(w)
    s = spec
    sigma = w.softmax_scale
    q = w.q.double().view(s.B, s.s_q, s.H_q, s.D_qk)
    for b in range(s.B):
        L = w.lengths[b]
        for h in range(s.H_kv):
            K, V = _kv_rows(w, b, h)
            # visible[j, t]: query token j sits at position L - s_q + j and sees
            # token t at or before it, and within the last `window` tokens
            t = torch.arange(L).view(1, L)
            pos = (L - s.s_q + torch.arange(s.s_q)).view(s.s_q, 1)
            visible = t <= pos
            if window:
                visible &= t > pos - window
            for g in range(s.G):
                hq = h * s.G + g
                S = sigma * (q[b, :, hq] @ K.T)                     # [s_q, L]
                S = S.masked_fill(~visible, float("-inf"))
                sink = float(w.sinks[hq]) if sinks else float("-inf")
                S = torch.cat([torch.full((s.s_q, 1), sink, dtype=torch.float64), S], dim=1)
                ref_lse = torch.logsumexp(S, dim=1)
                for jj in range(s.s_q):
                    if torch.isinf(ref_lse[jj]):
                        assert lse[b, jj, hq] == float("-inf")
                        assert torch.all(out[b, jj, hq] == 0)
                        continue
                    p = torch.softmax(S[jj], dim=0)[1:]
                    assert abs(float(lse[b, jj, hq] - ref_lse[jj])) < 1e-12
                    ref_o = p @ V if L else torch.zeros(s.D_v, dtype=torch.float64)
                    assert torch.allclose(out[b, jj, hq], ref_o, rtol=0, atol=1e-12)


def test_window_covering_everything_and_window_one(oracle_lib):
    spec = _spec(s_q=2)
    w = make_workload(spec, poison=False)
    out0, lse0 = oracle.attend_multi(w)
    wide = dataclasses.replace(w, spec=spec.with_(window=10 ** 6))
    out1, lse1 = oracle.attend_multi(wide)
    assert torch.equal(out0, out1) and torch.equal(lse0, lse1)
    # a window of one token: each query token sees only itself
    one = dataclasses.replace(w, spec=spec.with_(window=1))
    out, lse = oracle.attend_multi(one)
    P = spec.page_size
    for b, L in enumerate(w.lengths):
        for j in range(2):
            t = L - 2 + j
            if t < 0:
                assert torch.all(torch.isneginf(lse[b, j]))
                continue
            page = int(w.block_table[b, t // P])
            for h in range(spec.H_kv):
                v = w.v_pool[page, t % P, h].double()
                k = w.k_pool[page, t % P, h].double()
                for g in range(spec.G):
                    hq = h * spec.G + g
                    assert torch.equal(out[b, j, hq], v)
                    s_t = w.softmax_scale * float(w.q[b, j, hq].double() @ k)
                    assert abs(float(lse[b, j, hq]) - s_t) < 1e-12


def test_sinks_limits(oracle_lib):
    """A sink of -inf is no sink; a very large sink takes all the weight."""
    spec = _spec(s_q=1, sinks=True)
    w = make_workload(spec, poison=False)
    plain = dataclasses.replace(w, sinks=None)
    out0, lse0 = oracle.attend_multi(plain)
    out1, lse1 = oracle.attend_multi(dataclasses.replace(w, sinks=torch.full_like(w.sinks, float("-inf"))))
    assert torch.equal(out0, out1) and torch.equal(lse0, lse1)
    out2, lse2 = oracle.attend_multi(dataclasses.replace(w, sinks=torch.full_like(w.sinks, 80.0)))
    assert torch.all(out2.abs() < 1e-25)
    assert torch.allclose(lse2, torch.full_like(lse2, 80.0), rtol=0, atol=1e-12)


def test_last_draft_is_single_token_decode(oracle_lib):
    spec = _spec()
    w = make_workload(spec, poison=False)
    out, lse = oracle.attend_multi(w)
    single = dataclasses.replace(w, spec=spec.with_(s_q=1), q=w.q[:, -1].contiguous())
    ref_out, ref_lse = oracle.attend(single)
    assert torch.equal(out[:, -1], ref_out)
    assert torch.equal(lse[:, -1], ref_lse)


def test_drafts_do_not_see_later_tokens(oracle_lib):
    """Changing the last token of a request changes only its last draft."""
    spec = _spec(lengths=[20, 33, 9, 64, 65, 7])
    w = make_workload(spec, poison=False)
    out0, lse0 = oracle.attend_multi(w)
    P = spec.page_size
    for b, L in enumerate(w.lengths):
        page = int(w.block_table[b, (L - 1) // P])
        w.k_pool[page, (L - 1) % P] = w.k_pool[page, (L - 1) % P] * 3 + 1
        w.v_pool[page, (L - 1) % P] = -w.v_pool[page, (L - 1) % P]
    out1, lse1 = oracle.attend_multi(w)
    assert torch.equal(out0[:, :-1], out1[:, :-1]) and torch.equal(lse0[:, :-1], lse1[:, :-1])
    assert not torch.equal(out0[:, -1], out1[:, -1])
    assert not torch.equal(lse0[:, -1], lse1[:, -1])


@pytest.mark.parametrize("splits", [0, 1, 3])
def test_windowed_split_and_combine_equals_unsplit(oracle_lib, splits):
    from oracle.sched_ref import sched_ref
    spec = _spec(s_q=1, window=70, lengths=[1, 64, 65, 200, 333, 0], splits=splits)
    w = make_workload(spec, poison=False)
    ref = sched_ref(w.lengths, spec.H_kv, splits, num_sms=16, window=70)
    o, l = oracle.attend_split_combine(w, ref)
    out, lse = oracle.attend_multi(w)
    assert torch.allclose(o, out[:, 0], rtol=0, atol=1e-12)
    fin = ~torch.isneginf(lse[:, 0])
    assert torch.equal(torch.isneginf(l), ~fin)
    assert torch.allclose(l[fin], lse[:, 0][fin], rtol=0, atol=1e-12)


# ------------------------------------------------------------------ the 656-byte latent token, two drafts

def _mla_spec(**kw):
    base = dict(name="m", B=4, H_kv=1, G=4, D_qk=576, D_v=512, page_size=16, kv_dtype=KV_MLA656,
                lengths=[1, 2, 40, 0], splits=0, extra_pages=3, seed=9, s_q=2)
    base.update(kw)
    return WorkloadSpec(**base)


def _mla_rows(w, b):
    """K [L, 576] and V [L, 512] of request b in float64, decoded from the
    656-byte rows with torch's float8_e4m3fn type, independently of the
    oracle's decoder: 512 codes times their block's fp32 scale, rounded to
    bf16 (the FlashMLA page's chain, section 计算环节一), then the 64 bf16 RoPE
    values; V is the first 512."""
    P = w.spec.page_size
    ks = []
    for t in range(w.lengths[b]):
        row = w.k_pool[int(w.block_table[b, t // P]), t % P, 0]
        codes = row[:512].view(torch.float8_e4m3fn).float()
        scales = row[512:528].view(torch.float32).repeat_interleave(128)
        nope = (codes * scales).to(torch.bfloat16).double()
        rope = row[528:656].view(torch.bfloat16).double()
        ks.append(torch.cat([nope, rope]))
    if not ks:
        return torch.zeros(0, 576, dtype=torch.float64), torch.zeros(0, 512, dtype=torch.float64)
    K = torch.stack(ks)
    return K, K[:, :512]


def test_mla_two_drafts_masked_matrix(oracle_lib):
    """Two query tokens on the latent format: per (request, query head) the
    score matrix has one row per draft, later tokens set to -inf; torch's
    softmax and logsumexp over K, V decoded independently give out and lse."""
    spec = _mla_spec()
    w = make_workload(spec, poison=False)
    out, lse = oracle.attend_multi(w)
    q = w.q.double().view(spec.B, 2, spec.H_q, 576)
    for b, L in enumerate(w.lengths):
        K, V = _mla_rows(w, b)
        t = torch.arange(L).view(1, L)
        pos = (L - 2 + torch.arange(2)).view(2, 1)
        for hq in range(spec.H_q):
            S = (w.softmax_scale * (q[b, :, hq] @ K.T)).masked_fill(~(t <= pos), float("-inf"))
            for j in range(2):
                if L - 1 + j <= 0:
                    assert lse[b, j, hq] == float("-inf") and torch.all(out[b, j, hq] == 0)
                    continue
                assert abs(float(lse[b, j, hq] - torch.logsumexp(S[j], 0))) < 1e-11
                ref_o = torch.softmax(S[j], 0) @ V
                assert torch.allclose(out[b, j, hq], ref_o, rtol=0, atol=1e-11)


def test_mla_last_draft_is_single_token_decode(oracle_lib):
    spec = _mla_spec(lengths=[3, 70, 129, 1])
    w = make_workload(spec, poison=False)
    out, lse = oracle.attend_multi(w)
    single = dataclasses.replace(w, spec=spec.with_(s_q=1), q=w.q[:, -1].contiguous())
    ref_out, ref_lse = oracle.attend(single)
    assert torch.equal(out[:, -1], ref_out)
    assert torch.equal(lse[:, -1], ref_lse)
