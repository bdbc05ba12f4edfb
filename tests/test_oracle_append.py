"""Pins for the append oracle (oracle/append_ref.py): the e4m3 encoder against
the e4m3 decode pinned in test_oracle.py, against torch's float8_e4m3fn cast
(a library routine), closed forms of the rounding rule, and the 656-byte token
against its layout and the workload generator's block quantisation."""
import numpy as np
import pytest
import torch

import oracle
from oracle.append_ref import e4m3_encode, mla_row, append_ref

_FINITE = [c for c in range(256) if (c & 0x7F) != 0x7F]


def _values(codes):
    return np.array([oracle.e4m3_value(c) for c in codes])


def test_round_trip_every_finite_code(oracle_lib):
    v = _values(_FINITE).astype(np.float32)
    got = e4m3_encode(v)
    want = np.array(_FINITE, dtype=np.uint8)
    # +0 and -0 are distinct codes and both round trip through the sign bit.
    assert np.array_equal(got, want)


def test_midpoints_round_to_even_code(oracle_lib):
    pos = list(range(0, 0x7E))            # consecutive finite magnitudes c, c+1
    lo, hi = _values(pos), _values([c + 1 for c in pos])
    mid = ((lo + hi) / 2).astype(np.float32)
    assert np.array_equal(mid.astype(np.float64), (lo + hi) / 2)   # exact in fp32
    got = e4m3_encode(mid)
    want = np.array([c if c % 2 == 0 else c + 1 for c in pos], dtype=np.uint8)
    assert np.array_equal(got, want)
    assert np.array_equal(e4m3_encode(-mid), want | 0x80)
    # Just off the midpoint the nearer neighbour wins whatever its parity.
    below = np.nextafter(mid, np.float32(0))
    above = np.nextafter(mid, np.float32(np.inf))
    assert np.array_equal(e4m3_encode(below), np.array(pos, dtype=np.uint8))
    assert np.array_equal(e4m3_encode(above), np.array(pos, dtype=np.uint8) + 1)


def test_saturation_nan_and_signed_zero():
    v = np.array([448.0, 449.0, 480.0, 1e30, np.inf, -np.inf, -448.0, -1e9, np.nan, -np.nan,
                  0.0, -0.0, 2.0 ** -11, -(2.0 ** -11), 2.0 ** -10], dtype=np.float32)
    got = e4m3_encode(v).tolist()
    # 2^-10 is half the smallest subnormal 2^-9: a tie between 0x00 (even) and 0x01.
    assert got == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE, 0xFE, 0x7F, 0x7F,
                   0x00, 0x80, 0x00, 0x80, 0x00]


def test_agrees_with_torch_cast_in_range():
    g = torch.Generator().manual_seed(3)
    x = torch.cat([torch.randn(200000, generator=g) * s for s in (1e-3, 0.1, 1.0, 30.0, 150.0)])
    x = x.clamp(-448.0, 448.0)
    want = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(e4m3_encode(x.numpy()), want)


def test_mla_row_layout_and_generator_rule():
    g = torch.Generator().manual_seed(11)
    for trial in range(6):
        x = (torch.randn(576, generator=g) * (0.01 + trial)).to(torch.bfloat16)
        if trial == 5:
            x[128:256] = 0.0                       # an all-zero block takes scale 1
        bits = x.view(torch.int16).numpy().view(np.uint16)
        row = mla_row(bits)
        xf = x.float()
        blocks = xf[:512].reshape(4, 128)
        amax = blocks.abs().amax(dim=-1)
        scale = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
        codes = (blocks / scale.unsqueeze(-1)).clamp(-448, 448).to(torch.float8_e4m3fn)
        assert np.array_equal(row[:512], codes.view(torch.uint8).reshape(-1).numpy())
        assert np.array_equal(row[512:528].view(np.float32), scale.numpy())
        assert np.array_equal(row[528:656], x[512:].contiguous().view(torch.uint8).numpy())
        for blk in range(4):
            c = row[128 * blk:128 * blk + 128]
            if amax[blk] > 0:
                # the block's largest magnitude lands on +-448 exactly
                i = int(blocks[blk].abs().argmax())
                assert c[i] in (0x7E, 0xFE)
            else:
                assert np.all(c == 0)
            # decoded codes x scale reproduce the inputs within e4m3's half ulp
            dec = _values(c.tolist()) * float(row[512 + 4 * blk:516 + 4 * blk].view(np.float32)[0])
            ref = blocks[blk].double().numpy()
            tol = np.maximum(np.abs(ref) * 2.0 ** -4, 2.0 ** -10 * float(scale[blk]))
            assert np.all(np.abs(dec - ref) <= tol + 1e-30)


def _pools(kv_dtype, num_pages, P, H_kv, D):
    if kv_dtype == 0:
        return (torch.zeros(num_pages, P, H_kv, D, dtype=torch.bfloat16),
                torch.zeros(num_pages, P, H_kv, D, dtype=torch.bfloat16))
    if kv_dtype == 1:
        return (torch.zeros(num_pages, P, H_kv, D, dtype=torch.uint8),
                torch.zeros(num_pages, P, H_kv, D, dtype=torch.uint8))
    return torch.zeros(num_pages, P, 1, 656, dtype=torch.uint8), None


def test_append_places_tokens_by_block_table():
    """Brute force on a tiny case: each request's token lands in slot pos % P
    of page block_table[b][pos // P], every other byte is untouched, and the
    skip / error rules hold."""
    P, H_kv, D, num_pages = 4, 2, 8, 10
    bt = torch.tensor([[3, 7, 1], [0, 9, -1], [5, 2, 12], [4, 6, 8]], dtype=torch.int32)
    pos = torch.tensor([5, 9, 10, -1], dtype=torch.int32)     # page 7 slot 1; page -1 -> err 1; 12 -> err 1; skip
    g = torch.Generator().manual_seed(2)
    k_new = torch.randn(4, H_kv, D, generator=g).to(torch.bfloat16)
    v_new = torch.randn(4, H_kv, D, generator=g).to(torch.bfloat16)
    kp, vp = _pools(0, num_pages, P, H_kv, D)
    ek, ev, err = append_ref(0, P, kp, vp, k_new, v_new, pos, bt)
    assert err == 1
    ek = torch.from_numpy(ek).view(torch.bfloat16).view(num_pages, P, H_kv, D)
    ev = torch.from_numpy(ev).view(torch.bfloat16).view(num_pages, P, H_kv, D)
    want_k = torch.zeros_like(kp)
    want_k[7, 1] = k_new[0]
    assert torch.equal(ek, want_k)
    want_v = torch.zeros_like(vp)
    want_v[7, 1] = v_new[0]
    assert torch.equal(ev, want_v)
    # past the table: error bit 2
    _, _, err = append_ref(0, P, kp, vp, k_new[:1], v_new[:1], torch.tensor([12], dtype=torch.int32), bt[:1])
    assert err == 2


def test_append_fp8_uses_per_head_scale():
    P, H_kv, D, num_pages = 4, 3, 16, 3
    bt = torch.tensor([[2, 0]], dtype=torch.int32)
    pos = torch.tensor([6], dtype=torch.int32)
    g = torch.Generator().manual_seed(5)
    k_new = (torch.randn(1, H_kv, D, generator=g) * 3).to(torch.bfloat16)
    v_new = (torch.randn(1, H_kv, D, generator=g) * 3).to(torch.bfloat16)
    ks = torch.tensor([0.01, 0.5, 2.0])
    vs = torch.tensor([1.0, 0.03, 0.25])
    kp, vp = _pools(1, num_pages, P, H_kv, D)
    ek, ev, err = append_ref(1, P, kp, vp, k_new, v_new, pos, bt, ks, vs)
    assert err == 0
    ek = ek.reshape(num_pages, P, H_kv, D)
    ev = ev.reshape(num_pages, P, H_kv, D)
    for h in range(H_kv):
        wk = (k_new[0, h].float() / ks[h]).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
        wv = (v_new[0, h].float() / vs[h]).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
        assert np.array_equal(ek[0, 2, h], wk.numpy())
        assert np.array_equal(ev[0, 2, h], wv.numpy())
    ek[0, 2] = 0
    ev[0, 2] = 0
    assert not ek.any() and not ev.any()


@pytest.mark.parametrize("kv_dtype", [0, 1, 2])
def test_append_then_decode_sees_the_token(oracle_lib, kv_dtype):
    """The appended token is what the attention oracle reads at position L:
    with one token per request, softmax is 1 and out equals V (bf16 path) or
    its dequantised value."""
    from workloads import WorkloadSpec, make_workload
    if kv_dtype == 2:
        spec = WorkloadSpec(name="t", B=2, H_kv=1, G=4, D_qk=576, D_v=512, page_size=64,
                            lengths=[1, 1], kv_dtype=2, extra_pages=1, seed=3)
    else:
        spec = WorkloadSpec(name="t", B=2, H_kv=2, G=2, D_qk=16, D_v=16, page_size=8,
                            lengths=[1, 1], kv_dtype=kv_dtype, extra_pages=1, seed=3)
    w = make_workload(spec, poison=False)
    g = torch.Generator().manual_seed(8)
    k_new = torch.randn(spec.B, spec.H_kv, spec.D_qk, generator=g).to(torch.bfloat16)
    v_new = None if kv_dtype == 2 else torch.randn(spec.B, spec.H_kv, spec.D_v, generator=g).to(torch.bfloat16)
    pos = torch.zeros(spec.B, dtype=torch.int32)
    ek, ev, err = append_ref(kv_dtype, spec.page_size, w.k_pool, w.v_pool, k_new, v_new, pos,
                             w.block_table, w.k_scale, w.v_scale)
    assert err == 0
    w.k_pool = torch.from_numpy(ek).view(w.k_pool.dtype).view(w.k_pool.shape)
    if ev is not None:
        w.v_pool = torch.from_numpy(ev).view(w.v_pool.dtype).view(w.v_pool.shape)
    out, lse = oracle.attend(w)
    for b in range(spec.B):
        for h in range(spec.H_kv):
            for gq in range(spec.G):
                o = out[b, h * spec.G + gq].double()
                if kv_dtype == 0:
                    want = v_new[b, h].double()
                    assert torch.equal(o, want)
                elif kv_dtype == 1:
                    codes = ev.reshape(w.v_pool.shape)[int(w.block_table[b, 0]), 0, h]
                    want = torch.tensor(_values(codes.tolist())) * float(w.v_scale[h])
                    assert torch.allclose(o, want, rtol=0, atol=1e-12)
                    assert torch.allclose(o, v_new[b, h].double(), rtol=2.0 ** -4, atol=float(w.v_scale[h]) * 2.0 ** -9)
                else:
                    row = ek.reshape(w.k_pool.shape)[int(w.block_table[b, 0]), 0, h]
                    # the latent token dequantises as bf16(fp32(e4m3) * fp32 scale)
                    sc = torch.from_numpy(row[512:528].copy().view(np.float32)).repeat_interleave(128)
                    vals = torch.tensor(_values(row[:512].tolist()), dtype=torch.float32)
                    want = (vals * sc).to(torch.bfloat16).double()
                    assert torch.allclose(o, want, rtol=0, atol=1e-12)
                    assert torch.allclose(o, k_new[b, h, :512].double(), rtol=2.0 ** -4,
                                          atol=float(k_new[b, h, :512].float().abs().max()) / 448 * 2.0 ** -9)
