"""Pins for the multi-token (linear draft chain) oracle, oracle.attend_multi:
a masked-matrix formulation with torch's softmax / logsumexp, the reduction of
the last draft to single-token decode, and causality (a draft never sees the
tokens after it)."""
import dataclasses

import pytest
import torch

import oracle
from workloads import WorkloadSpec, make_workload, KV_BF16, KV_FP8


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


@pytest.mark.parametrize("kv_dtype", [KV_BF16, KV_FP8])
def test_masked_matrix_formulation(oracle_lib, kv_dtype):
    spec = _spec(kv_dtype=kv_dtype)
    w = make_workload(spec, poison=False)
    out, lse = oracle.attend_multi(w)
    s = spec
    sigma = w.softmax_scale
    q = w.q.double()
    for b in range(s.B):
        L = w.lengths[b]
        for h in range(s.H_kv):
            K, V = _kv_rows(w, b, h)
            # mask[j, t]: draft j (at position L - s_q + j) sees token t <= its own position
            t = torch.arange(L).view(1, L)
            j = torch.arange(s.s_q).view(s.s_q, 1)
            visible = t <= (L - s.s_q + j)
            for g in range(s.G):
                hq = h * s.G + g
                S = sigma * (q[b, :, hq] @ K.T)                     # [s_q, L]
                S = S.masked_fill(~visible, float("-inf"))
                ref_lse = torch.logsumexp(S, dim=1) if L else torch.full((s.s_q,), float("-inf"), dtype=torch.float64)
                for jj in range(s.s_q):
                    if torch.isinf(ref_lse[jj]):
                        assert lse[b, jj, hq] == float("-inf")
                        assert torch.all(out[b, jj, hq] == 0)
                        continue
                    p = torch.softmax(S[jj], dim=0)
                    assert abs(float(lse[b, jj, hq] - ref_lse[jj])) < 1e-12
                    assert torch.allclose(out[b, jj, hq], p @ V, rtol=0, atol=1e-12)


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
