"""The allocation-free decode entry point, for callers that cannot allocate
device memory (pre-planned memory arenas, plug-ins without access to their
host's allocator, real-time paths): decode_attn_fwd_static_scratch keeps its
scratch in a fixed device array owned by the library.

Checked through the C ABI against decode_attn_sched_meta + decode_attn_fwd
with a caller-allocated scratch buffer, bit for bit, on two calls in a row
(the second call reuses the array the first one left behind), and once
against the float64 oracle. This file is collected last.
"""
import ctypes

import pytest
import torch

import oracle
import paged_kv_cache_60_gb300 as da
from workloads import WorkloadSpec, make_workload, spec_by_name, KV_BF16, KV_FP8, KV_MLA656

from gpu_util import LSE_TOL, OUT_TOL, DeviceWorkload, ensure_built, make_desc, max_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    lib = ensure_built()
    oracle.build_oracle()
    f = lib.decode_attn_fwd_static_scratch
    P = ctypes.c_void_p
    f.argtypes = [ctypes.POINTER(da.Desc), P, P, P, P, P, P, P, P, P, P]
    f.restype = ctypes.c_int
    return lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _static_call(lib, desc, dw, out, lse, q=None):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    q = dw.q if q is None else q
    return lib.decode_attn_fwd_static_scratch(ctypes.byref(desc), _ptr(q), _ptr(dw.k_pool), _ptr(dw.v_pool),
                                              _ptr(dw.k_scale), _ptr(dw.v_scale), _ptr(dw.block_table),
                                              _ptr(dw.cache_seqlens), _ptr(out), _ptr(lse), stream)


CASES = [
    (WorkloadSpec(name="a", B=3, H_kv=2, G=8, D_qk=128, D_v=128, page_size=16, lengths=[517, 1, 300],
                  splits=0, extra_pages=5, seed=21), 0),
    (WorkloadSpec(name="b", B=4, H_kv=4, G=8, D_qk=64, D_v=64, page_size=256, lengths=[1536, 700, 0, 64],
                  splits=8, seed=22), 0),
    (WorkloadSpec(name="c", B=2, H_kv=4, G=8, D_qk=128, D_v=128, page_size=32, lengths=[5000, 333],
                  kv_dtype=KV_FP8, splits=0, seed=23), 0),
    # the 656-byte latent token: its partials and score-swap slots share the
    # array; a fixed split count keeps them inside it
    (WorkloadSpec(name="d", B=3, H_kv=1, G=128, D_qk=576, D_v=512, page_size=64, lengths=[3000, 65, 700],
                  kv_dtype=KV_MLA656, splits=4, seed=24), 0),
    # ... and the automatic split count on fewer SMs
    (WorkloadSpec(name="e", B=2, H_kv=1, G=128, D_qk=576, D_v=512, page_size=64, lengths=[4100, 900],
                  kv_dtype=KV_MLA656, splits=0, seed=25), 24),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_static_scratch_matches_caller_scratch_twice(lib, case):
    spec, num_sms = CASES[case]
    w = make_workload(spec)
    dw = DeviceWorkload(w)
    desc = make_desc(w, num_sms=num_sms)
    s = w.spec
    assert da.sched_meta_bytes(desc) <= (16 << 20)
    # reference: the existing entry points with a caller-allocated buffer
    meta = torch.empty(da.sched_meta_bytes(desc), dtype=torch.uint8, device="cuda")
    ref_out = torch.empty(s.B, s.H_q, s.D_v, dtype=torch.bfloat16, device="cuda")
    ref_lse = torch.empty(s.B, s.H_q, dtype=torch.float32, device="cuda")
    da.sched_meta(desc, dw.cache_seqlens, meta)
    da.fwd(desc, dw.q, dw.k_pool, dw.v_pool, dw.k_scale, dw.v_scale, dw.block_table, dw.cache_seqlens, meta,
           ref_out, ref_lse)
    torch.cuda.synchronize()
    assert da.get_error(meta) == 0
    for call in range(2):
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        assert _static_call(lib, desc, dw, out, lse) == 0
        torch.cuda.synchronize()
        # the same kernels on the same schedule: identical bits
        assert torch.equal(out, ref_out), call
        assert torch.equal(lse, ref_lse), call
    # and the float64 oracle, at the tolerances of the other parity tests
    o_ref, l_ref = oracle.attend(w)
    e_out, e_lse = max_err(out, lse, o_ref, l_ref)
    assert e_out <= OUT_TOL and e_lse <= LSE_TOL, (e_out, e_lse)


def test_static_scratch_rejects_a_problem_too_large(lib):
    spec = spec_by_name("mixed_gqa_bf16").with_(B=2, lengths=[64, 64], length_dist="fixed")
    w = make_workload(spec)
    dw = DeviceWorkload(w)
    desc = make_desc(w, splits=4096)        # 2 x 4096 splits of 64 x 128 fp32 partials: far above 16 MiB
    assert da.sched_meta_bytes(desc) > (16 << 20)
    out = torch.empty(2, spec.H_q, spec.D_v, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(2, spec.H_q, dtype=torch.float32, device="cuda")
    assert _static_call(lib, desc, dw, out, lse) == -6


def test_static_scratch_rejects_before_launching(lib):
    """A call that fails a host check launches nothing: the array keeps the
    previous call's schedule, and the next valid call still matches."""
    w = make_workload(CASES[0][0])
    dw = DeviceWorkload(w)
    desc = make_desc(w)
    s = w.spec
    out = torch.full((s.B, s.H_q, s.D_v), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((s.B, s.H_q), float("nan"), dtype=torch.float32, device="cuda")
    assert _static_call(lib, desc, dw, out, lse) == 0
    torch.cuda.synchronize()
    first = (out.clone(), lse.clone())
    misaligned_q = torch.empty(dw.q.numel() + 8, dtype=torch.bfloat16, device="cuda")[1:1 + dw.q.numel()]
    out.fill_(float("nan"))
    assert _static_call(lib, desc, dw, out, lse, q=misaligned_q) == da.DA_ERR_ALIGN
    wm = make_workload(CASES[3][0])             # the 656-byte format, listed positions: no way to pass them
    dwm = DeviceWorkload(wm)
    sparse = make_desc(wm)
    sparse.topk = 64
    out_m = torch.full((wm.spec.B, wm.spec.H_q, wm.spec.D_v), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse_m = torch.full((wm.spec.B, wm.spec.H_q), float("nan"), dtype=torch.float32, device="cuda")
    assert _static_call(lib, sparse, dwm, out_m, lse_m) == da.DA_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert torch.isnan(out_m.float()).all()
    assert torch.isnan(out.float()).all()       # nothing ran
    assert _static_call(lib, desc, dw, out, lse) == 0
    torch.cuda.synchronize()
    assert torch.equal(out, first[0]) and torch.equal(lse, first[1])
