"""NaN in the KV pool -- the e4m3 codes 0x7F / 0xFF, a NaN block scale of the
656-byte token, a NaN bf16 RoPE value -- reaches exactly the outputs it
reaches in the float64 oracle: a NaN in K poisons the score of every query
head that reads the token, and so the out and lse rows of that (request, KV
head); a NaN in V only the out column it sits in. Every other value matches
the oracle within the usual tolerances. Checked through the C ABI with the
automatic split count (the combine kernel merges the partials) and with a
fixed one (3 splits: on the GQA formats the cluster merge), so the NaN has to
cross the merge of the split partials."""
import pytest
import torch

import oracle
from workloads import WorkloadSpec, make_workload, KV_FP8, KV_MLA656

from gpu_util import LSE_TOL, OUT_TOL, ensure_built, run

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    ensure_built()
    oracle.build_oracle()


def _spec(kind, splits):
    if kind == "mla":
        return WorkloadSpec(name="nan_mla", B=3, H_kv=1, G=128, D_qk=576, D_v=512, page_size=64,
                            kv_dtype=KV_MLA656, lengths=[300, 1, 777], splits=splits, seed=41)
    return WorkloadSpec(name="nan_fp8", B=3, H_kv=2, G=8, D_qk=128, D_v=128, page_size=32,
                        kv_dtype=KV_FP8, lengths=[300, 1, 777], splits=splits, seed=42)


# (format, pool, byte edits of one token row, what the edit is)
CASES = [
    ("mla", "k", [(5, 0x7F)], "e4m3 0x7F in the value dims"),
    ("mla", "k", [(300, 0xFF)], "e4m3 0xFF in the value dims"),
    ("mla", "k", [(512, 0x00), (513, 0x00), (514, 0xC0), (515, 0x7F)], "NaN scale of the first 128 values"),
    ("mla", "k", [(528, 0xC0), (529, 0x7F)], "NaN bf16 RoPE value (K only)"),
    ("fp8", "k", [(5, 0x7F)], "e4m3 0x7F in K"),
    ("fp8", "k", [(70, 0xFF)], "e4m3 0xFF in K"),
    ("fp8", "v", [(5, 0x7F)], "e4m3 0x7F in V: one out column"),
]


@pytest.mark.parametrize("splits", [0, 3])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_nan_in_the_pool_reaches_what_it_reaches_in_the_oracle(case, splits):
    kind, pool, edits, _ = CASES[case]
    w = make_workload(_spec(kind, splits))
    s = w.spec
    b, t = 2, 400                                # token 400 of request 2
    page = int(w.block_table[b, t // s.page_size])
    rows = w.k_pool if pool == "k" else w.v_pool
    for byte, val in edits:
        rows[page, t % s.page_size, 0, byte] = val
    ref_out, ref_lse = oracle.attend(w)
    assert torch.isnan(ref_out).any()            # the edit is a NaN for the oracle too
    out, lse, meta, desc = run(w)
    torch.cuda.synchronize()
    out = out.float().cpu()
    lse = lse.cpu()
    assert torch.equal(torch.isnan(lse), torch.isnan(ref_lse))
    assert torch.equal(torch.isnan(out), torch.isnan(ref_out))
    ok_o, ok_l = ~torch.isnan(ref_out), ~torch.isnan(ref_lse)
    e_out = (out[ok_o].double() - ref_out[ok_o]).abs().max().item()
    e_lse = (lse[ok_l].double() - ref_lse[ok_l]).abs().max().item() if ok_l.any() else 0.0
    assert e_out <= OUT_TOL and e_lse <= LSE_TOL, (e_out, e_lse)
