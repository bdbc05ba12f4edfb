"""Failure detection without a GPU fault: every pipeline wait in the split-KV
kernel is bounded. In the test build of the library (-DDA_PAGE_TRACE) the
consumer warps can be made to wait first on a barrier that nothing completes,
with the bound shortened to 1 ms: the wait runs out, the kernel sets the
timeout bit in the device error word and its CTAs return, and the CUDA context
stays usable: the next call without the stall matches the oracle."""
import pytest
import torch

import oracle
import paged_kv_cache_60_gb300 as da
from workloads import KV_BF16, KV_FP8, KV_MLA656, WorkloadSpec, make_workload

from gpu_util import LSE_TOL, OUT_TOL, DeviceWorkload, debug_build_library, make_desc, max_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tlib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    oracle.build_oracle()
    return debug_build_library()


def _call(tlib, w, dw, desc):
    s = w.spec
    meta = torch.empty(da.sched_meta_bytes(desc), dtype=torch.uint8, device="cuda")
    out = torch.zeros(s.B, s.H_q, s.D_v, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(s.B, s.H_q, dtype=torch.float32, device="cuda")
    da.sched_meta(desc, dw.cache_seqlens, meta, lib=tlib)
    da.fwd(desc, dw.q, dw.k_pool, dw.v_pool, dw.k_scale, dw.v_scale, dw.block_table, dw.cache_seqlens, meta, out,
           lse, lib=tlib)
    torch.cuda.synchronize()
    return out, lse, da.get_error(meta)


@pytest.mark.parametrize("kv", [KV_BF16, KV_FP8])
def test_wait_that_runs_out_sets_timeout_and_context_survives(tlib, kv):
    # automatic splits on purpose: with a fixed split count of 2-8 the splits
    # merge through each other's shared memory, and a CTA whose handshake wait
    # ran out could exit while a slower split still arrives on its barriers
    spec = WorkloadSpec(name="t", B=4, H_kv=4, G=8, D_qk=128, D_v=128, page_size=32, kv_dtype=kv,
                        lengths=[4000, 3000, 2000, 1000], splits=0, seed=51)
    w = make_workload(spec)
    dw = DeviceWorkload(w)
    desc = make_desc(w)
    assert tlib.decode_attn_debug_wait_limit(1000000) == 0
    assert tlib.decode_attn_debug_stall(1) == 0
    try:
        _, _, err = _call(tlib, w, dw, desc)
    finally:
        tlib.decode_attn_debug_stall(0)
        tlib.decode_attn_debug_wait_limit(0)
    assert err & da.DA_DEV_TIMEOUT, err
    # the context is still usable and the normal bound gives the oracle's result
    out, lse, err = _call(tlib, w, dw, desc)
    assert err == 0
    ref_out, ref_lse = oracle.attend(w)
    e_out, e_lse = max_err(out, lse, ref_out, ref_lse)
    assert e_out <= OUT_TOL and e_lse <= LSE_TOL, (e_out, e_lse)


def test_latent_kernel_wait_that_runs_out(tlib):
    """The same on the 656-byte latent format: its CTAs never read each
    other's memory, so a CTA that gives up leaves nothing in flight; the MMA
    warp drains what it issued before the tensor memory is freed."""
    spec = WorkloadSpec(name="t", B=3, H_kv=1, G=128, D_qk=576, D_v=512, page_size=64, kv_dtype=KV_MLA656,
                        lengths=[3000, 700, 1500], splits=0, seed=52)
    w = make_workload(spec)
    dw = DeviceWorkload(w)
    desc = make_desc(w)
    assert tlib.decode_attn_debug_wait_limit(1000000) == 0
    assert tlib.decode_attn_debug_stall(1) == 0
    try:
        _, _, err = _call(tlib, w, dw, desc)
    finally:
        tlib.decode_attn_debug_stall(0)
        tlib.decode_attn_debug_wait_limit(0)
    assert err & da.DA_DEV_TIMEOUT, err
    out, lse, err = _call(tlib, w, dw, desc)
    assert err == 0
    ref_out, ref_lse = oracle.attend(w)
    e_out, e_lse = max_err(out, lse, ref_out, ref_lse)
    assert e_out <= OUT_TOL and e_lse <= LSE_TOL, (e_out, e_lse)
