"""GPU parity for the cluster merge: with a fixed split count of 2-8 the
splits of a (request, KV head) run as one thread-block cluster and merge their
partials through distributed shared memory instead of a combine kernel. Split
counts that do and do not divide D, empty requests (every split empty),
splits with no tokens, sinks and several query tokens, against the oracle;
and one count past the cluster limit (the combine kernel) for comparison."""
import pytest
import torch

import oracle
import paged_kv_cache_60_gb300 as da
from workloads import WorkloadSpec, make_workload, KV_BF16, KV_FP8

from gpu_util import LSE_TOL, OUT_TOL, ensure_built, max_err, run

pytestmark = pytest.mark.gpu

LENGTHS = [0, 1, 5, 63, 64, 65, 130, 517, 1000, 3000]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    ensure_built()
    oracle.build_oracle()


CASES = [
    # kv, D, splits, s_q, sinks, page size
    (KV_BF16, 64, 2, 1, False, 16),
    (KV_BF16, 64, 5, 1, True, 64),
    (KV_BF16, 64, 8, 3, False, 256),
    (KV_BF16, 128, 2, 2, True, 32),
    (KV_BF16, 128, 7, 1, False, 8),
    (KV_BF16, 128, 8, 4, True, 16),
    (KV_FP8, 128, 3, 1, True, 32),
    (KV_FP8, 128, 8, 2, False, 64),
    (KV_BF16, 128, 9, 1, True, 16),   # past the cluster limit: combine kernel
]


@pytest.mark.parametrize("kv,D,S,s_q,sinks,P", CASES)
def test_cluster_merge_parity(kv, D, S, s_q, sinks, P):
    spec = WorkloadSpec(name="t", B=len(LENGTHS), H_kv=2, G=8, D_qk=D, D_v=D, page_size=P, kv_dtype=kv,
                        lengths=LENGTHS, splits=S, extra_pages=4, seed=90 + S + P, s_q=s_q, sinks=sinks)
    w = make_workload(spec)
    out, lse, meta, _ = run(w)
    torch.cuda.synchronize()
    assert da.get_error(meta) == 0
    ref_out, ref_lse = oracle.attend_multi(w)
    e_out, e_lse = max_err(out.view(ref_out.shape), lse.view(ref_lse.shape), ref_out, ref_lse)
    assert e_out <= OUT_TOL and e_lse <= LSE_TOL, (e_out, e_lse)


def test_cluster_merge_is_deterministic():
    spec = WorkloadSpec(name="t", B=4, H_kv=2, G=8, D_qk=128, D_v=128, page_size=16, lengths=[700, 3, 1500, 64],
                        splits=6, extra_pages=2, seed=5)
    w = make_workload(spec)
    o1, l1, _, _ = run(w)
    o2, l2, _, _ = run(w)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
