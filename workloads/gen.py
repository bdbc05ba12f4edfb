"""Seeded synthetic paged-KV inputs.

Layout produced (the "VLLM layout" of the XQA page, section
"Hopper:一次 TMA 只搬一个页"): separate K and V pools shaped
``[num_pages, page_size, H_kv, D]``; ``block_table[b, j]`` is the physical page
that holds logical page ``j`` of request ``b``; ``q`` is ``[B, H_q, D_qk]`` with
query head ``h*G + g`` belonging to KV head ``h``.

Recipe (all draws from one seeded torch CPU generator, then rounded):
  * lengths: fixed, uniform integer on [lo, hi] inclusive, or
    floor(exp(U(ln lo, ln hi))) clamped to [lo, hi];
  * pool: sum_b ceil(L_b / P) used pages plus ``extra_pages`` unused ones; the
    physical ids are a seeded random permutation handed out in
    (request, logical page) order; unused block-table entries are -1;
  * values: q, K, V ~ N(0, 1) in fp32, rounded to bf16 (RNE);
  * FP8 per-tensor KV: fp32 N(0,1) per (KV head, tensor) scaled by
    scale = amax / 448 (1 when amax is 0) and rounded to e4m3 (RNE, clipped
    to +-448 so that nothing becomes NaN);
  * 656-byte MLA token: 576 fp32 N(0,1) values; the first 512 are quantised
    per block of 128 with their own fp32 scale (same rule), the last 64 kept
    as bf16; bytes are [512 x e4m3][4 x fp32 scale][64 x bf16];
  * poison: every pool slot that no valid token occupies (unused pages and
    the tail of each request's last page) is NaN (bf16 0x7FC0, e4m3 0x7F,
    fp32 scale NaN) so that a stray read shows up in the result.

Nothing here computes attention: this module only draws and places data.
"""
from dataclasses import dataclass
from typing import List, Optional

import math
import numpy as np
import torch

from .configs import KV_BF16, KV_FP8, KV_MLA656, WorkloadSpec

KV_F64 = 3          # oracle-only: exact float64 pools for pinning tests

E4M3_MAX = 448.0    # largest finite e4m3 value (XQA page: kE4M3_MAX)
MLA_NOPE = 512
MLA_ROPE = 64
MLA_BLOCK = 128
MLA_ROW_BYTES = MLA_NOPE + 4 * (MLA_NOPE // MLA_BLOCK) + 2 * MLA_ROPE   # 656

_BF16_NAN = 0x7FC0
_E4M3_NAN = 0x7F


@dataclass
class Workload:
    spec: WorkloadSpec
    lengths: List[int]
    num_pages: int
    max_pages_per_seq: int
    q: torch.Tensor                 # bf16 [B, H_q, D_qk]
    k_pool: torch.Tensor            # bf16/uint8/float64 pool
    v_pool: Optional[torch.Tensor]  # None for MLA656 (K and V share the token)
    k_scale: Optional[torch.Tensor]  # fp32 [H_kv] (FP8 per-tensor)
    v_scale: Optional[torch.Tensor]
    block_table: torch.Tensor       # int32 [B, max_pages_per_seq]
    cache_seqlens: torch.Tensor     # int32 [B]
    sinks: Optional[torch.Tensor] = None  # fp32 [H_q] attention-sink logits, or None
    indices: Optional[torch.Tensor] = None  # int32 [B, topk] token positions (sparse decode), or None

    @property
    def softmax_scale(self) -> float:
        s = self.spec
        return s.softmax_scale if s.softmax_scale > 0 else 1.0 / math.sqrt(s.D_qk)

    def kv_bytes(self) -> int:
        """Bytes of K and V that a decode pass must read once per KV head."""
        s = self.spec
        if s.topk > 0:     # sparse decode reads the listed tokens (each valid entry once)
            tok = int(sum(min(L, s.topk) for L in self.lengths))
        elif s.window > 0:   # tokens before the first query token's window are not read
            tok = int(sum(L - max(0, L - s.s_q + 1 - s.window) for L in self.lengths if L > 0))
        else:
            tok = int(sum(self.lengths))
        if s.kv_dtype == KV_MLA656:
            return tok * s.H_kv * MLA_ROW_BYTES
        es = {KV_BF16: 2, KV_FP8: 1, KV_F64: 8}[s.kv_dtype]
        return tok * s.H_kv * (s.D_qk + s.D_v) * es


def draw_lengths(spec: WorkloadSpec) -> List[int]:
    if spec.lengths is not None:
        assert len(spec.lengths) == spec.B
        return [int(x) for x in spec.lengths]
    rng = np.random.Generator(np.random.PCG64(spec.seed + 7919))
    if spec.length_dist == "uniform":
        return [int(x) for x in rng.integers(spec.length_lo, spec.length_hi + 1, size=spec.B)]
    if spec.length_dist == "loguniform":
        u = rng.uniform(math.log(spec.length_lo), math.log(spec.length_hi), size=spec.B)
        return [int(min(max(math.floor(math.exp(x)), spec.length_lo), spec.length_hi)) for x in u]
    raise ValueError(spec.length_dist)


def _pages_for(L: int, P: int) -> int:
    return (L + P - 1) // P


def build_block_table(spec: WorkloadSpec, lengths: List[int]):
    P = spec.page_size
    n_pages = [_pages_for(L, P) for L in lengths]
    used = sum(n_pages)
    num_pages = max(1, used + spec.extra_pages)
    maxp = max(1, max(n_pages) if n_pages else 1)
    rng = np.random.Generator(np.random.PCG64(spec.seed + 104729))
    perm = rng.permutation(num_pages)
    bt = np.full((spec.B, maxp), -1, dtype=np.int32)
    k = 0
    for b, n in enumerate(n_pages):
        for j in range(n):
            bt[b, j] = perm[k]
            k += 1
    return torch.from_numpy(bt), num_pages, maxp


def valid_slot_mask(spec: WorkloadSpec, lengths, block_table, num_pages) -> torch.Tensor:
    """bool [num_pages, P]: True where a valid token of some request lives."""
    P = spec.page_size
    mask = torch.zeros(num_pages, P, dtype=torch.bool)
    bt = block_table.numpy()
    for b, L in enumerate(lengths):
        full, rem = divmod(L, P)
        for j in range(full):
            mask[bt[b, j]] = True
        if rem:
            mask[bt[b, full], :rem] = True
    return mask


def _randn(gen: torch.Generator, shape) -> torch.Tensor:
    return torch.randn(*shape, generator=gen, dtype=torch.float32)


def _page_chunks(num_pages: int, per_page_elems: int, budget: int = 1 << 26):
    step = max(1, budget // max(1, per_page_elems))
    for p0 in range(0, num_pages, step):
        yield p0, min(num_pages, p0 + step)


def _quantize_e4m3(x: torch.Tensor, scale) -> torch.Tensor:
    """fp32 tensor / scale -> e4m3 bytes (RNE, clipped to +-448)."""
    y = (x / scale).clamp_(-E4M3_MAX, E4M3_MAX)
    return y.to(torch.float8_e4m3fn).view(torch.uint8)


def make_workload(spec: WorkloadSpec, lengths: Optional[List[int]] = None,
                  poison: bool = True) -> Workload:
    if lengths is None:
        lengths = draw_lengths(spec)
    lengths = [int(x) for x in lengths]
    B, H_kv, G, Dq, Dv, P = spec.B, spec.H_kv, spec.G, spec.D_qk, spec.D_v, spec.page_size
    H_q = H_kv * G
    bt, num_pages, maxp = build_block_table(spec, lengths)
    gen = torch.Generator().manual_seed(spec.seed)

    # one query token per request: q [B, H_q, D_qk]; s_q > 1: q [B, s_q, H_q, D_qk]
    q_shape = (B, H_q, Dq) if spec.s_q == 1 else (B, spec.s_q, H_q, Dq)
    q = _randn(gen, q_shape).to(torch.bfloat16)
    valid = valid_slot_mask(spec, lengths, bt, num_pages) if poison else None
    k_scale = v_scale = None
    v_pool = None

    if spec.kv_dtype in (KV_BF16, KV_F64):
        assert Dq == Dv, "GQA pools carry K and V of the same head size"
        dt = torch.bfloat16 if spec.kv_dtype == KV_BF16 else torch.float64
        pools = []
        for _ in range(2):
            pool = torch.empty(num_pages, P, H_kv, Dq, dtype=dt)
            for p0, p1 in _page_chunks(num_pages, P * H_kv * Dq):
                pool[p0:p1] = _randn(gen, (p1 - p0, P, H_kv, Dq)).to(dt)
            if poison:
                pool[~valid] = float("nan")
            pools.append(pool)
        k_pool, v_pool = pools
    elif spec.kv_dtype == KV_FP8:
        assert Dq == Dv
        pools, scales = [], []
        for _ in range(2):
            parts = []
            amax = torch.zeros(H_kv, dtype=torch.float32)
            for p0, p1 in _page_chunks(num_pages, P * H_kv * Dq):
                x = _randn(gen, (p1 - p0, P, H_kv, Dq))
                amax = torch.maximum(amax, x.abs().amax(dim=(0, 1, 3)))
                parts.append(x)
            scale = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax))
            pool = torch.empty(num_pages, P, H_kv, Dq, dtype=torch.uint8)
            p0 = 0
            for x in parts:
                pool[p0:p0 + x.shape[0]] = _quantize_e4m3(x, scale.view(1, 1, H_kv, 1))
                p0 += x.shape[0]
            del parts
            if poison:
                pool[~valid] = _E4M3_NAN
            pools.append(pool)
            scales.append(scale)
        k_pool, v_pool = pools
        k_scale, v_scale = scales
    elif spec.kv_dtype == KV_MLA656:
        assert Dq == MLA_NOPE + MLA_ROPE and Dv == MLA_NOPE and H_kv == 1
        k_pool = torch.empty(num_pages, P, H_kv, MLA_ROW_BYTES, dtype=torch.uint8)
        nb = MLA_NOPE // MLA_BLOCK
        for p0, p1 in _page_chunks(num_pages, P * H_kv * Dq):
            n = (p1 - p0) * P * H_kv
            x = _randn(gen, (n, Dq))
            blocks = x[:, :MLA_NOPE].reshape(n, nb, MLA_BLOCK)
            amax = blocks.abs().amax(dim=-1)
            scale = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax))
            codes = _quantize_e4m3(blocks, scale.unsqueeze(-1)).reshape(n, MLA_NOPE)
            sbytes = scale.contiguous().view(torch.uint8).reshape(n, 4 * nb)
            rope = x[:, MLA_NOPE:].to(torch.bfloat16).contiguous().view(torch.uint8).reshape(n, 2 * MLA_ROPE)
            row = torch.cat([codes, sbytes, rope], dim=1)
            k_pool[p0:p1] = row.reshape(p1 - p0, P, H_kv, MLA_ROW_BYTES)
        if poison:
            bad = k_pool[~valid]              # [n_bad, H_kv, 656]
            bad[..., :MLA_NOPE] = _E4M3_NAN
            bad[..., MLA_NOPE:MLA_NOPE + 4 * nb] = torch.tensor(
                [float("nan")] * nb, dtype=torch.float32).view(torch.uint8)
            bad[..., MLA_NOPE + 4 * nb:] = torch.tensor(
                [_BF16_NAN] * MLA_ROPE, dtype=torch.int32).to(torch.int16).view(torch.uint8)
            k_pool[~valid] = bad
    else:
        raise ValueError(spec.kv_dtype)

    sinks = None
    if spec.sinks:
        # per query head, around ln 64: a sink worth tens of tokens of weight
        gs = torch.Generator().manual_seed(spec.seed + 17)
        sinks = (torch.randn(H_q, generator=gs) * 2.0 + math.log(64.0)).float()
    indices = None
    if spec.topk > 0:
        # top-k positions per request: topk distinct positions in random order,
        # or, for a request shorter than topk, all of its positions then -1
        gi = torch.Generator().manual_seed(spec.seed + 29)
        indices = torch.full((B, spec.topk), -1, dtype=torch.int32)
        for b, L in enumerate(lengths):
            if L > 0:
                pick = torch.randperm(L, generator=gi)[:spec.topk].to(torch.int32)
                indices[b, :pick.numel()] = pick
    return Workload(spec=spec, lengths=lengths, num_pages=num_pages, max_pages_per_seq=maxp,
                    q=q, k_pool=k_pool, v_pool=v_pool, k_scale=k_scale, v_scale=v_scale,
                    block_table=bt, cache_seqlens=torch.tensor(lengths, dtype=torch.int32), sinks=sinks,
                    indices=indices)


def place_logical(w: Workload, b: int, t: int, k_row=None, v_row=None):
    """Overwrite the pool slot holding logical token t of request b (tests only)."""
    P = w.spec.page_size
    page = int(w.block_table[b, t // P])
    slot = t % P
    if k_row is not None:
        w.k_pool[page, slot] = k_row
    if v_row is not None:
        w.v_pool[page, slot] = v_row


def repermute_pages(w: Workload, seed: int) -> Workload:
    """Same logical contents, new physical placement (and a new block table)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    perm = torch.from_numpy(rng.permutation(w.num_pages).astype(np.int64))
    # physical page p moves to perm[p]
    def move(pool):
        if pool is None:
            return None
        out = torch.empty_like(pool)
        out[perm] = pool
        return out
    bt = w.block_table.clone().to(torch.int64)
    ok = bt >= 0
    bt[ok] = perm[bt[ok]]
    return Workload(spec=w.spec, lengths=list(w.lengths), num_pages=w.num_pages,
                    max_pages_per_seq=w.max_pages_per_seq, q=w.q.clone(),
                    k_pool=move(w.k_pool), v_pool=move(w.v_pool),
                    k_scale=w.k_scale, v_scale=w.v_scale,
                    block_table=bt.to(torch.int32), cache_seqlens=w.cache_seqlens.clone(), sinks=w.sinks,
                    indices=w.indices)


def make_append_batch(w: Workload, seed: int):
    """Inputs of a KV append on workload ``w``: one new token per request,
    written at the slot of its last token (positions[b] = lengths[b] - 1, -1
    for an empty request, which the append skips). Returns (k_new, v_new,
    positions): bf16 N(0,1) rows [B, H_kv, D_qk] and [B, H_kv, D_v] like the
    pools' values, or for the 656-byte format the 576-value latent vector in
    k_new and v_new None; positions int32 [B]."""
    s = w.spec
    gen = torch.Generator().manual_seed(seed)
    k_new = _randn(gen, (s.B, s.H_kv, s.D_qk)).to(torch.bfloat16)
    v_new = None if s.kv_dtype == KV_MLA656 else _randn(gen, (s.B, s.H_kv, s.D_v)).to(torch.bfloat16)
    positions = torch.tensor([L - 1 for L in w.lengths], dtype=torch.int32)
    return k_new, v_new, positions
