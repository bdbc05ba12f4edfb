"""GPU parity of the KV append (decode_attn_append_kv through the C ABI)
against the append oracle: every byte of both pools (and a guard region past
them) bit-exact, the error word exact; then append followed by decode, on one
stream without a sync between them, against the attention oracle."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_60_gb300 as da
from oracle.append_ref import append_ref
from workloads import WorkloadSpec, make_workload, make_append_batch, KV_BF16, KV_FP8, KV_MLA656

from gpu_util import LSE_TOL, OUT_TOL, DeviceWorkload, ensure_built, make_desc, max_err, run

pytestmark = pytest.mark.gpu

GUARD = 4096   # bytes after each pool that must stay untouched

# Edge values (bf16-exact): signed zeros, bf16 subnormals, e4m3 midpoints at
# scale 1 (1.0625, 1.1875, 232, 3 * 2^-10, 2^-10), 448 and beyond, infinities, NaN.
SPECIAL = [0.0, -0.0, 1e-40, -1e-40, 1.0625, -1.0625, 1.1875, 232.0, 3 * 2.0 ** -10, 2.0 ** -10,
           -(2.0 ** -10), 448.0, 464.0, 500.0, -1e4, math.inf, -math.inf, math.nan, 240.0, -0.0234375]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    ensure_built()
    oracle.build_oracle()


def _desc(kv_dtype, B, H_kv, D, P, max_pages, num_pages):
    if kv_dtype == KV_MLA656:
        return da.Desc.make(B=B, H_kv=1, G=128, D_qk=576, D_v=512, page_size=P, max_pages_per_seq=max_pages,
                            num_pages=num_pages, kv_dtype=kv_dtype)
    return da.Desc.make(B=B, H_kv=H_kv, G=8, D_qk=D, D_v=D, page_size=P, max_pages_per_seq=max_pages,
                        num_pages=num_pages, kv_dtype=kv_dtype)


def _random_pool(g, kv_dtype, num_pages, P, H_kv, D):
    """Pool of random bytes (any content: the append must leave it alone)
    followed by a guard region, as (buffer, pool view)."""
    if kv_dtype == KV_MLA656:
        shape, dt = (num_pages, P, 1, 656), torch.uint8
    elif kv_dtype == KV_FP8:
        shape, dt = (num_pages, P, H_kv, D), torch.uint8
    else:
        shape, dt = (num_pages, P, H_kv, D), torch.bfloat16
    nbytes = int(np.prod(shape)) * (2 if dt == torch.bfloat16 else 1)
    buf = torch.randint(0, 256, (nbytes + GUARD,), generator=g, dtype=torch.uint8)
    return buf, buf[:nbytes].view(dt).view(shape)


def _case(kv_dtype, B, H_kv, D, P, seed, max_pages=5, specials=True):
    g = torch.Generator().manual_seed(seed)
    num_pages = B * max_pages + 7
    perm = torch.randperm(num_pages, generator=g).to(torch.int32)
    bt = perm[:B * max_pages].reshape(B, max_pages).clone()   # distinct pages: no two requests share a slot
    pos = torch.randint(0, max_pages * P, (B,), generator=g, dtype=torch.int32)
    if B > 5:
        pos[1] = -5                                   # skipped
        pos[2] = max_pages * P                        # past the table: error 2
        bt[3, int(pos[3]) // P] = -1                  # bad page: error 1
        bt[4, int(pos[4]) // P] = num_pages           # bad page: error 1
        pos[5] = max_pages * P - 1                    # last slot of the last page
    if kv_dtype == KV_MLA656:
        k_new = torch.randn(B, 1, 576, generator=g).to(torch.bfloat16)
        v_new = None
        ks = vs = None
        if specials:
            k_new[0, 0, 0:20] = torch.tensor(SPECIAL[:17] + [1.0, 2.0, 3.0]).to(torch.bfloat16)   # inf in block 0
            k_new[0, 0, 128:256] = 0.0
            k_new[0, 0, 130:140] = -0.0                                                          # all-zero block
            k_new[0, 0, 256:266] = torch.tensor([math.nan] + [0.5] * 9).to(torch.bfloat16)       # NaN block
            if B > 6:
                k_new[6, 0, 0:128] = (torch.randn(128, generator=g) * 1e-39).to(torch.bfloat16)  # subnormal block
                k_new[6, 0, 128:256] = (torch.randn(128, generator=g) * 1e30).to(torch.bfloat16)
    else:
        k_new = torch.randn(B, H_kv, D, generator=g).to(torch.bfloat16)
        v_new = torch.randn(B, H_kv, D, generator=g).to(torch.bfloat16)
        if kv_dtype == KV_FP8:
            base = [1.0, 0.25, 0.0137, 3.7, 2.0 ** -12, 0.5, 1.5, 7.0]
            ks = torch.tensor((base * H_kv)[:H_kv], dtype=torch.float32)
            vs = torch.tensor((base[::-1] * H_kv)[:H_kv], dtype=torch.float32)
            k_new = (k_new.float() * ks.view(1, H_kv, 1) * 40).to(torch.bfloat16)   # some values saturate
        else:
            ks = vs = None
        if specials:
            n = min(len(SPECIAL), D)
            k_new[0, 0, :n] = torch.tensor(SPECIAL[:n]).to(torch.bfloat16)
            v_new[0, H_kv - 1, :n] = torch.tensor(SPECIAL[::-1][:n]).to(torch.bfloat16)
    kbuf, kp = _random_pool(g, kv_dtype, num_pages, P, H_kv, D)
    vbuf, vp = (None, None) if kv_dtype == KV_MLA656 else _random_pool(g, kv_dtype, num_pages, P, H_kv, D)
    return dict(kv_dtype=kv_dtype, B=B, H_kv=H_kv, D=D, P=P, max_pages=max_pages, num_pages=num_pages,
                bt=bt, pos=pos, k_new=k_new, v_new=v_new, ks=ks, vs=vs, kbuf=kbuf, kp=kp, vbuf=vbuf, vp=vp)


def _expected(c):
    ek, ev, err = append_ref(c["kv_dtype"], c["P"], c["kp"], c["vp"], c["k_new"], c["v_new"], c["pos"], c["bt"],
                             c["ks"], c["vs"])
    guard_k = c["kbuf"][-GUARD:].numpy()
    want_k = np.concatenate([ek, guard_k])
    want_v = None if ev is None else np.concatenate([ev, c["vbuf"][-GUARD:].numpy()])
    return want_k, want_v, err


def _run_gpu(c, row_stride_pad=0):
    B, H_kv, D = c["B"], c["H_kv"], c["D"]
    kbuf = c["kbuf"].cuda()
    vbuf = None if c["vbuf"] is None else c["vbuf"].cuda()
    npool = c["kbuf"].numel() - GUARD
    kp = kbuf[:npool]
    vp = None if vbuf is None else vbuf[:npool]
    row = 576 if c["kv_dtype"] == KV_MLA656 else H_kv * D
    if row_stride_pad:
        # the new rows sit inside a wider per-request buffer (a fused projection output)
        stride = row * (1 if c["v_new"] is None else 2) + row_stride_pad
        fused = torch.full((B, stride), float("nan"), dtype=torch.bfloat16)
        fused[:, row_stride_pad:row_stride_pad + row] = c["k_new"].reshape(B, row)
        if c["v_new"] is not None:
            fused[:, row_stride_pad + row:row_stride_pad + 2 * row] = c["v_new"].reshape(B, row)
        fused = fused.cuda()
        k_new = fused[:, row_stride_pad:]
        v_new = None if c["v_new"] is None else fused[:, row_stride_pad + row:]
    else:
        stride = 0
        k_new = c["k_new"].cuda()
        v_new = None if c["v_new"] is None else c["v_new"].cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    desc = _desc(c["kv_dtype"], B, H_kv, D, c["P"], c["max_pages"], c["num_pages"])
    da.append_kv(desc, k_new, v_new, c["pos"].cuda(), c["bt"].cuda(), kp, vp,
                 None if c["ks"] is None else c["ks"].cuda(), None if c["vs"] is None else c["vs"].cuda(),
                 device_error=err, new_row_stride=stride)
    torch.cuda.synchronize()
    return kbuf.cpu().numpy(), None if vbuf is None else vbuf.cpu().numpy(), int(err.item())


def _check(c, row_stride_pad=0):
    want_k, want_v, want_err = _expected(c)
    got_k, got_v, got_err = _run_gpu(c, row_stride_pad)
    assert got_err == want_err
    bad = np.nonzero(got_k != want_k)[0]
    assert bad.size == 0, f"K pool differs at {bad.size} bytes, first {bad[:8].tolist()}"
    if want_v is not None:
        bad = np.nonzero(got_v != want_v)[0]
        assert bad.size == 0, f"V pool differs at {bad.size} bytes, first {bad[:8].tolist()}"


CASES = [
    (KV_BF16, 4, 128, 16, 37),
    (KV_BF16, 2, 64, 8, 300),
    (KV_BF16, 1, 64, 256, 1),
    (KV_FP8, 4, 128, 32, 37),
    (KV_FP8, 3, 64, 64, 129),
    (KV_FP8, 8, 128, 8, 2),
    (KV_MLA656, 1, 576, 64, 37),
    (KV_MLA656, 1, 576, 16, 300),
    (KV_MLA656, 1, 576, 128, 1),
]


@pytest.mark.parametrize("kv_dtype,H_kv,D,P,B", CASES)
def test_append_bitexact(kv_dtype, H_kv, D, P, B):
    _check(_case(kv_dtype, B, H_kv, D, P, seed=100 + B + P))


@pytest.mark.parametrize("kv_dtype,H_kv,D", [(KV_BF16, 4, 128), (KV_FP8, 2, 128), (KV_MLA656, 1, 576)])
def test_append_strided_rows(kv_dtype, H_kv, D):
    c = _case(kv_dtype, 50, H_kv, D, 32, seed=7)
    _check(c, row_stride_pad=32 * 8)


@pytest.mark.parametrize("kv_dtype,H_kv,D", [(KV_BF16, 8, 128), (KV_FP8, 8, 128), (KV_MLA656, 1, 576)])
def test_append_large_batch(kv_dtype, H_kv, D):
    """More work items than the grid holds (grid-stride loop), every request valid."""
    _check(_case(kv_dtype, 4096, H_kv, D, 8, seed=3, max_pages=1, specials=False))


def test_append_extreme_scales():
    """Per-tensor scales at and beyond the range in which the quotient takes
    the corrected multiply (2^-80 .. 2^100), and inputs whose quotient would
    overflow the residual: the codes still equal the oracle's, byte for byte."""
    c = _case(KV_FP8, 64, 6, 128, 16, seed=13, specials=False)
    c["ks"] = torch.tensor([2.0 ** -90, 2.0 ** 105, 2.0 ** -79, 1e-30, 2.0 ** 100, 2.0 ** -80], dtype=torch.float32)
    c["vs"] = torch.tensor([2.0 ** -81, 3.0 ** 60, 1e-24, 2.0 ** 99, 0.75, 2.0 ** -100], dtype=torch.float32)
    g = torch.Generator().manual_seed(14)
    mag = torch.tensor([1e-30, 1e-20, 1e-6, 1.0, 1e4, 1e20, 1e30, 3e38])
    for t in ("k_new", "v_new"):
        x = torch.randn(c[t].shape, generator=g) * mag[torch.randint(0, len(mag), c[t].shape, generator=g)]
        c[t] = x.to(torch.bfloat16)
    _check(c)


def test_append_all_skipped_writes_nothing():
    c = _case(KV_FP8, 16, 2, 128, 16, seed=9)
    c["pos"][:] = -1
    _check(c)


@pytest.mark.parametrize("kv_dtype", [KV_BF16, KV_FP8, KV_MLA656])
def test_append_then_decode(kv_dtype):
    """A decode step: append each request's new token at its last position,
    then decode over the grown sequences on the same stream (the decode
    kernels are chained to the append and wait for it)."""
    if kv_dtype == KV_MLA656:
        spec = WorkloadSpec(name="t", B=5, H_kv=1, G=128, D_qk=576, D_v=512, page_size=64,
                            lengths=[1, 65, 300, 0, 128], kv_dtype=kv_dtype, extra_pages=3, seed=21)
    else:
        spec = WorkloadSpec(name="t", B=5, H_kv=2, G=8, D_qk=128, D_v=128, page_size=16,
                            lengths=[1, 17, 300, 0, 64], kv_dtype=kv_dtype, extra_pages=3, seed=21)
    w = make_workload(spec)
    k_new, v_new, pos = make_append_batch(w, seed=5)
    dw = DeviceWorkload(w)
    desc = make_desc(w)
    da.append_kv(desc, k_new.cuda(), None if v_new is None else v_new.cuda(), pos.cuda(), dw.block_table,
                 dw.k_pool, dw.v_pool, dw.k_scale, dw.v_scale)
    out, lse, _, _ = run(w, dw=dw, desc=desc)
    torch.cuda.synchronize()
    ek, ev, err = append_ref(kv_dtype, spec.page_size, w.k_pool, w.v_pool, k_new, v_new, pos, w.block_table,
                             w.k_scale, w.v_scale)
    assert err == 0
    assert np.array_equal(dw.k_pool.cpu().contiguous().view(-1).view(torch.uint8).numpy(), ek)
    w.k_pool = torch.from_numpy(ek).view(w.k_pool.dtype).view(w.k_pool.shape)
    if ev is not None:
        assert np.array_equal(dw.v_pool.cpu().contiguous().view(-1).view(torch.uint8).numpy(), ev)
        w.v_pool = torch.from_numpy(ev).view(w.v_pool.dtype).view(w.v_pool.shape)
    ref_out, ref_lse = oracle.attend(w)
    e_out, e_lse = max_err(out, lse, ref_out, ref_lse)
    assert e_out <= OUT_TOL and e_lse <= LSE_TOL, (e_out, e_lse)
