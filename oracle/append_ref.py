"""CPU oracle for appending one new token per request to the paged KV pool,
quantising on the way. TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

The pages place this step upstream of decode attention: the new token's K and
V are written into the page slot that the block table gives for its position
(XQA page, section "Hopper:一次 TMA 只搬一个页", the pool layout; FlashMLA page,
section "数据加载", the 656-byte token). Formats:

* bf16 pools: the new values, bit for bit.
* e4m3 pools with a per-KV-head scale (XQA page, FP8 KV cache): code =
  e4m3(x / scale[h]), the quotient an fp32 division rounded to nearest.
* 656-byte latent tokens: per 128-value block of the 512 NoPE values, scale =
  max|x| / 448 in fp32 (1 when the block is all zero), codes = e4m3(x / scale);
  the four scales as fp32; then the 64 RoPE values as bf16 (the layout of the
  FlashMLA page's token, the block rule of the workload generator).

e4m3(v) is the nearest finite e4m3 value (OCP FP8 definition: sign, 4
exponent bits with bias 7, 3 mantissa bits, largest finite 448), ties to the
even code, magnitudes beyond 448 saturating to 448 and NaN giving 0x7F.
"""
import numpy as np

from . import e4m3_value

E4M3_MAX = 448.0
_POS_CODES = np.arange(0x7F, dtype=np.uint8)                        # 0x00 .. 0x7E, increasing values
_POS_VALUES = np.array([e4m3_value(int(c)) for c in _POS_CODES])    # float64, exact


def e4m3_encode(v) -> np.ndarray:
    """fp32 values -> e4m3 codes (nearest, ties to even, saturating)."""
    v = np.asarray(v, dtype=np.float32)
    a = np.abs(v).astype(np.float64)
    hi = np.clip(np.searchsorted(_POS_VALUES, a, side="left"), 0, len(_POS_VALUES) - 1)
    lo = np.clip(hi - 1, 0, len(_POS_VALUES) - 1)
    d_lo = a - _POS_VALUES[lo]
    d_hi = _POS_VALUES[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (_POS_CODES[hi] % 2 == 0))
    code = np.where(pick_hi, _POS_CODES[hi], _POS_CODES[lo]).astype(np.uint8)
    code = np.where(a >= _POS_VALUES[-1], np.uint8(0x7E), code)     # saturate (448 and beyond)
    code = np.where(np.signbit(v), code | np.uint8(0x80), code)
    code = np.where(np.isnan(v), np.uint8(0x7F), code)
    return code.astype(np.uint8)


def _bf16_bits(t) -> np.ndarray:
    """torch bf16 tensor -> uint16 bit patterns."""
    import torch
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def mla_row(x_bits: np.ndarray) -> np.ndarray:
    """576 bf16 bit patterns (512 NoPE + 64 RoPE) -> the 656-byte token."""
    x = _bf16_to_f32(x_bits[:512]).reshape(4, 128)
    row = np.zeros(656, dtype=np.uint8)
    scales = np.zeros(4, dtype=np.float32)
    for blk in range(4):
        amax = np.float32(np.max(np.abs(x[blk])))
        scale = np.float32(amax / np.float32(E4M3_MAX)) if amax > 0 else np.float32(1.0)
        scales[blk] = scale
        with np.errstate(invalid="ignore", divide="ignore", over="ignore"):   # inf / inf -> NaN -> 0x7F
            q = x[blk] / scale
        row[128 * blk:128 * blk + 128] = e4m3_encode(q)
    row[512:528] = scales.view(np.uint8)
    row[528:656] = x_bits[512:576].astype(np.uint16).view(np.uint8)
    return row


def append_ref(kv_dtype, page_size, k_pool, v_pool, k_new, v_new, positions, block_table, k_scale=None,
               v_scale=None):
    """Expected pools after the append, as numpy byte arrays (uint8 views of
    the pool tensors), and the device error bits (1: page id outside the pool,
    2: position at or past max_pages * page_size). Requests with a negative
    position are skipped. Inputs are CPU torch tensors."""
    kp = k_pool.contiguous().view(-1).view(__import__("torch").uint8).numpy().copy()
    vp = None if v_pool is None else v_pool.contiguous().view(-1).view(__import__("torch").uint8).numpy().copy()
    num_pages, P, H_kv = k_pool.shape[0], k_pool.shape[1], k_pool.shape[2]
    bt = block_table.numpy()
    pos = positions.numpy()
    max_len = bt.shape[1] * P
    err = 0
    kb, vb = _bf16_bits(k_new), (None if v_new is None else _bf16_bits(v_new))
    ks = None if k_scale is None else k_scale.numpy().astype(np.float32)
    vs = None if v_scale is None else v_scale.numpy().astype(np.float32)
    B = pos.shape[0]
    for b in range(B):
        t = int(pos[b])
        if t < 0:
            continue
        if t >= max_len:
            err |= 2
            continue
        page = int(bt[b, t // P])
        if page < 0 or page >= num_pages:
            err |= 1
            continue
        slot = t % P
        for h in range(H_kv):
            if kv_dtype == 2:
                off = ((page * P + slot) * H_kv + h) * 656
                kp[off:off + 656] = mla_row(kb[b, h])
                continue
            D = kb.shape[2]
            if kv_dtype == 0:
                off = ((page * P + slot) * H_kv + h) * D * 2
                kp[off:off + 2 * D] = kb[b, h].view(np.uint8)
                vp[off:off + 2 * D] = vb[b, h].view(np.uint8)
            else:
                off = ((page * P + slot) * H_kv + h) * D
                with np.errstate(invalid="ignore", divide="ignore", over="ignore"):
                    qk = _bf16_to_f32(kb[b, h]) / ks[h]
                    qv = _bf16_to_f32(vb[b, h]) / vs[h]
                kp[off:off + D] = e4m3_encode(qk)
                vp[off:off + D] = e4m3_encode(qv)
    return kp, vp, err
