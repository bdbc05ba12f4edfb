"""Pins for the sparse (top-k) decode oracle, oracle.attend_sparse: the full
in-order list is dense decode bit for bit, the order of the list does not
matter, invalid entries are skipped, a listed-twice position counts twice."""
import dataclasses
import math

import pytest
import torch

import oracle
from workloads import WorkloadSpec, make_workload, KV_BF16, KV_MLA656


def _spec(kv, **kw):
    if kv == KV_MLA656:
        base = dict(name="t", B=4, H_kv=1, G=8, D_qk=576, D_v=512, page_size=16, lengths=[1, 30, 77, 0],
                    kv_dtype=KV_MLA656, extra_pages=2, seed=4, topk=40)
    else:
        base = dict(name="t", B=4, H_kv=2, G=4, D_qk=16, D_v=16, page_size=8, lengths=[1, 30, 77, 0],
                    extra_pages=2, seed=4, topk=40)
    base.update(kw)
    return WorkloadSpec(**base)


KINDS = [KV_BF16, KV_MLA656]


@pytest.mark.parametrize("kv", KINDS)
def test_full_in_order_list_is_dense_decode(oracle_lib, kv):
    spec = _spec(kv)
    w = make_workload(spec, poison=False)
    Lmax = max(w.lengths)
    idx = torch.full((spec.B, Lmax), -1, dtype=torch.int32)
    for b, L in enumerate(w.lengths):
        idx[b, :L] = torch.arange(L, dtype=torch.int32)
    out, lse = oracle.attend_sparse(w, idx)
    ref_out, ref_lse = oracle.attend(w)
    assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)


@pytest.mark.parametrize("kv", KINDS)
def test_order_invalid_entries_and_duplicates(oracle_lib, kv):
    spec = _spec(kv)
    w = make_workload(spec, poison=False)
    out, lse = oracle.attend_sparse(w)
    g = torch.Generator().manual_seed(9)
    perm = torch.stack([row[torch.randperm(row.numel(), generator=g)] for row in w.indices])
    o2, l2 = oracle.attend_sparse(w, perm)
    assert torch.allclose(o2, out, rtol=0, atol=1e-12) and torch.equal(torch.isneginf(l2), torch.isneginf(lse))
    fin = ~torch.isneginf(lse)
    assert torch.allclose(l2[fin], lse[fin], rtol=0, atol=1e-12)
    # entries outside [0, L_b) are skipped
    junk = torch.tensor([[-1, -7, 10 ** 6, L] for L in w.lengths], dtype=torch.int32)
    o3, l3 = oracle.attend_sparse(w, torch.cat([junk[:, :2], w.indices, junk[:, 2:]], dim=1))
    assert torch.equal(o3, out) and torch.equal(l3, lse)
    # every position twice: the same weights, lse + ln 2
    o4, l4 = oracle.attend_sparse(w, torch.cat([w.indices, w.indices], dim=1))
    assert torch.allclose(o4, out, rtol=0, atol=1e-12)
    assert torch.allclose(l4[fin], lse[fin] + math.log(2.0), rtol=0, atol=1e-12)
    assert torch.all(torch.isneginf(l4[~fin])) and torch.all(o4[~fin.unsqueeze(-1).expand_as(o4)] == 0)


def test_generator_indices_are_distinct_valid_positions():
    spec = _spec(KV_BF16, lengths=[100, 5, 40, 0], topk=40)
    w = make_workload(spec, poison=False)
    for b, L in enumerate(w.lengths):
        row = w.indices[b].tolist()
        valid = [t for t in row if t >= 0]
        assert len(valid) == min(L, 40) and len(set(valid)) == len(valid) and all(t < L for t in valid)
        assert row[len(valid):] == [-1] * (40 - len(valid))
