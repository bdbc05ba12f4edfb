"""CPU oracle for paged-KV decode attention (float64, plain loops).

TEST INFRASTRUCTURE ONLY. Only tests/, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package; the library under
``paged_kv_cache_60_gb300`` never does, and the two share no code.

* ``decode_ref.c``  -- attention by its definition, per (request, KV head,
  head range, token range), plus the split merge; built with gcc + OpenMP.
  ``attend_multi`` applies it per query token of the general decode step:
  several query tokens per request (each draft sees the history and the
  drafts before it), a sliding window, attention sinks; ``attend_sparse``
  over a list of token positions per request (top-k sparse decode).
* ``sched_ref.py``  -- the integer split-KV scheduling metadata.
* ``append_ref.py`` -- appending one new token per request into its page slot,
  with the e4m3 encoder (per-head scales, or the 656-byte latent token).

Parity pins are in tests/test_oracle.py, tests/test_sched_oracle.py and
tests/test_oracle_append.py.
"""
import ctypes
import os
import subprocess
import threading

import numpy as np
import torch

from .sched_ref import CHUNK, SchedRef, sched_ref, part_segments, split_token_ranges, auto_num_parts  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "decode_ref.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libdecode_ref.so")
_lock = threading.Lock()
_lib = None


class RefDesc(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("H_kv", ctypes.c_int32), ("G", ctypes.c_int32),
                ("D_qk", ctypes.c_int32), ("D_v", ctypes.c_int32), ("P", ctypes.c_int32),
                ("max_pages", ctypes.c_int32), ("num_pages", ctypes.c_int32),
                ("kv_dtype", ctypes.c_int32), ("pad", ctypes.c_int32),
                ("softmax_scale", ctypes.c_double)]


def build_oracle(force: bool = False) -> str:
    """Compile decode_ref.c (gcc, -O2, OpenMP). Returns the .so path."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-std=c11", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build_oracle())
            P = ctypes.c_void_p
            lib.ref_attend_units.restype = ctypes.c_int
            lib.ref_attend_units.argtypes = [ctypes.POINTER(RefDesc), P, P, P, P, P, P, P,
                                             ctypes.c_int, P, P, ctypes.c_int64, P, ctypes.c_int64]
            lib.ref_attend_lists.restype = ctypes.c_int
            lib.ref_attend_lists.argtypes = [ctypes.POINTER(RefDesc), P, P, P, P, P, P, ctypes.c_int, P, P,
                                             P, ctypes.c_int64, P, ctypes.c_int64]
            lib.ref_combine.restype = None
            lib.ref_combine.argtypes = [ctypes.c_int, ctypes.c_int, P, P, P, P]
            lib.ref_e4m3_value.restype = ctypes.c_double
            lib.ref_e4m3_value.argtypes = [ctypes.c_uint8]
            lib.ref_bf16_value.restype = ctypes.c_double
            lib.ref_bf16_value.argtypes = [ctypes.c_uint16]
            lib.ref_num_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def num_threads() -> int:
    return _load().ref_num_threads()


def e4m3_value(code: int) -> float:
    return _load().ref_e4m3_value(code)


def bf16_value(bits: int) -> float:
    return _load().ref_bf16_value(bits)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _kv_tag(w):
    return int(w.spec.kv_dtype)


def attend_units(w, units, q64=None):
    """Run the oracle on units [(b, h, g0, g1, t0, t1)] of workload ``w``
    (t1 = -1 means L_b). Returns (out [n, g1-g0, D_v] f64, lse [n, g1-g0] f64)
    with every unit padded to the widest head range."""
    lib = _load()
    s = w.spec
    units = [tuple(int(x) for x in u) for u in units]
    n = len(units)
    ng = max((u[3] - u[2]) for u in units) if n else 1
    if q64 is None:
        q64 = w.q.to(torch.float64).contiguous()
    d = RefDesc(B=s.B, H_kv=s.H_kv, G=s.G, D_qk=s.D_qk, D_v=s.D_v, P=s.page_size,
                max_pages=w.max_pages_per_seq, num_pages=w.num_pages, kv_dtype=_kv_tag(w),
                pad=0, softmax_scale=w.softmax_scale)
    u_arr = torch.tensor(units, dtype=torch.int32).reshape(n, 6).contiguous()
    out = torch.zeros(n, ng, s.D_v, dtype=torch.float64)
    lse = torch.zeros(n, ng, dtype=torch.float64)
    kp = w.k_pool.contiguous()
    vp = w.v_pool.contiguous() if w.v_pool is not None else None
    ks = w.k_scale.contiguous() if w.k_scale is not None else None
    vs = w.v_scale.contiguous() if w.v_scale is not None else None
    bt = w.block_table.contiguous()
    sl = w.cache_seqlens.contiguous()
    bad = lib.ref_attend_units(ctypes.byref(d), _ptr(q64), _ptr(kp), _ptr(vp), _ptr(ks), _ptr(vs),
                               _ptr(bt), _ptr(sl), n, _ptr(u_arr), _ptr(out), ng * s.D_v,
                               _ptr(lse), ng)
    if bad:
        raise ValueError(f"oracle: {bad} unit(s) read a page id outside the pool")
    return out, lse


def attend(w, heads=None):
    """Full attention for every (b, h) (or the given list of (b, h)).
    Returns out [B, H_q, D_v] and lse [B, H_q] (float64; NaN where not computed)."""
    s = w.spec
    if heads is None:
        heads = [(b, h) for b in range(s.B) for h in range(s.H_kv)]
    units = [(b, h, 0, s.G, 0, -1) for (b, h) in heads]
    o, l = attend_units(w, units)
    out = torch.full((s.B, s.H_q, s.D_v), float("nan"), dtype=torch.float64)
    lse = torch.full((s.B, s.H_q), float("nan"), dtype=torch.float64)
    for i, (b, h) in enumerate(heads):
        out[b, h * s.G:(h + 1) * s.G] = o[i]
        lse[b, h * s.G:(h + 1) * s.G] = l[i]
    return out, lse


def attend_multi(w, heads=None):
    """The general decode step: s_q query tokens per request, an optional
    sliding window and optional attention sinks. Returns out [B, s_q, H_q, D_v]
    and lse [B, s_q, H_q] (float64; NaN where not computed).

    * Drafts (s_q > 1; linear speculative-decoding verification, XQA page,
      section "投机解码:XQA 的第二个工作负载": the drafts form a chain, so each
      sees the history and the drafts before it): the request's last s_q
      tokens are the drafts, already in the cache (L_b counts them); draft j
      is at position L_b - s_q + j and sees the tokens up to it. w.q is
      [B, s_q, H_q, D_qk] (or [B, H_q, D_qk] when s_q = 1).
    * Sliding window W > 0 (XQA page, section "分页 KV:页号怎么变成 TMA 坐标"):
      a query token sees only the last W tokens up to and including itself.
    * Sinks (XQA page, section "一个容易漏掉的细节:attention sink"): one logit
      per query head, w.sinks[hq], in the units of the scores sigma q.k, that
      joins the softmax denominator and carries no value:
      lse = ln(e^sink + sum_t e^{s_t}), out = sum_t e^{s_t - lse} v_t. A row
      that sees no token has out = 0 and lse = sink (-inf without sinks).
    """
    s = w.spec
    sq = s.s_q
    W = s.window
    if heads is None:
        heads = [(b, h) for b in range(s.B) for h in range(s.H_kv)]
    out = torch.full((s.B, sq, s.H_q, s.D_v), float("nan"), dtype=torch.float64)
    lse = torch.full((s.B, sq, s.H_q), float("nan"), dtype=torch.float64)
    q = w.q.view(s.B, sq, s.H_q, s.D_qk)
    for j in range(sq):
        units = []
        for (b, h) in heads:
            hi = max(0, w.lengths[b] - sq + 1 + j)
            lo = max(0, hi - W) if W > 0 else 0
            units.append((b, h, 0, s.G, lo, hi))
        o, l = attend_units(w, units, q64=q[:, j].to(torch.float64).contiguous())
        for i, (b, h) in enumerate(heads):
            out[b, j, h * s.G:(h + 1) * s.G] = o[i]
            lse[b, j, h * s.G:(h + 1) * s.G] = l[i]
    if getattr(w, "sinks", None) is not None:
        sink = w.sinks.to(torch.float64).view(1, 1, s.H_q).expand_as(lse)
        done = ~torch.isnan(lse)
        tot = torch.logaddexp(lse, sink)
        fac = torch.where(torch.isneginf(lse), torch.zeros_like(lse), torch.exp(lse - tot))
        out = torch.where(done.unsqueeze(-1), out * fac.unsqueeze(-1), out)
        lse = torch.where(done, tot, lse)
    return out, lse


def attend_sparse(w, indices=None, heads=None):
    """Sparse (top-k) decode, the FlashMLA page's decode call with `indices`:
    request b attends over the token positions indices[b, :] (int32 [B, topk];
    defaults to w.indices). Entries outside [0, L_b) -- the -1 padding of a
    short request, or a stale position -- are skipped; a position listed twice
    is two terms. Returns out [B, H_q, D_v] and lse [B, H_q] (float64; NaN
    where not computed; lse -inf and out 0 for a request with no valid entry)."""
    lib = _load()
    s = w.spec
    if indices is None:
        indices = w.indices
    idx = indices.to(torch.int32).cpu()
    if heads is None:
        heads = [(b, h) for b in range(s.B) for h in range(s.H_kv)]
    toks, units = [], []
    for (b, h) in heads:
        L = w.lengths[b]
        lst = [int(t) for t in idx[b].tolist() if 0 <= int(t) < L]
        units.append((b, h, 0, s.G, len(toks), len(lst)))
        toks.extend(lst)
    q64 = w.q.to(torch.float64).contiguous()
    d = RefDesc(B=s.B, H_kv=s.H_kv, G=s.G, D_qk=s.D_qk, D_v=s.D_v, P=s.page_size,
                max_pages=w.max_pages_per_seq, num_pages=w.num_pages, kv_dtype=_kv_tag(w),
                pad=0, softmax_scale=w.softmax_scale)
    n = len(units)
    u_arr = torch.tensor(units, dtype=torch.int32).reshape(n, 6).contiguous()
    t_arr = torch.tensor(toks if toks else [0], dtype=torch.int32)
    o = torch.zeros(n, s.G, s.D_v, dtype=torch.float64)
    l = torch.zeros(n, s.G, dtype=torch.float64)
    kp = w.k_pool.contiguous()
    vp = w.v_pool.contiguous() if w.v_pool is not None else None
    ks = w.k_scale.contiguous() if w.k_scale is not None else None
    vs = w.v_scale.contiguous() if w.v_scale is not None else None
    bt = w.block_table.contiguous()
    bad = lib.ref_attend_lists(ctypes.byref(d), _ptr(q64), _ptr(kp), _ptr(vp), _ptr(ks), _ptr(vs), _ptr(bt),
                               n, _ptr(u_arr), _ptr(t_arr), _ptr(o), s.G * s.D_v, _ptr(l), s.G)
    if bad:
        raise ValueError(f"oracle: {bad} unit(s) read a page id outside the pool")
    out = torch.full((s.B, s.H_q, s.D_v), float("nan"), dtype=torch.float64)
    lse = torch.full((s.B, s.H_q), float("nan"), dtype=torch.float64)
    for i, (b, h) in enumerate(heads):
        out[b, h * s.G:(h + 1) * s.G] = o[i]
        lse[b, h * s.G:(h + 1) * s.G] = l[i]
    return out, lse


def combine(o_parts: torch.Tensor, lse_parts: torch.Tensor):
    """Merge partials of one query head: o_parts [n, D] f64, lse_parts [n] f64."""
    lib = _load()
    o_parts = o_parts.to(torch.float64).contiguous()
    lse_parts = lse_parts.to(torch.float64).contiguous()
    n, D = o_parts.shape
    out = torch.zeros(D, dtype=torch.float64)
    lse = torch.zeros(1, dtype=torch.float64)
    lib.ref_combine(n, D, _ptr(o_parts), _ptr(lse_parts), _ptr(out), _ptr(lse))
    return out, float(lse[0])


def attend_split_combine(w, ref: SchedRef):
    """Oracle split-then-combine over the token ranges that ``ref`` assigns:
    every split computed on its own, then merged. Returns out, lse like attend()."""
    s = w.spec
    ranges = split_token_ranges(ref, w.lengths, w.spec.window, w.spec.s_q)
    units, index = [], []
    for b in range(s.B):
        for h in range(s.H_kv):
            for si, r in enumerate(ranges[b]):
                t0, t1 = r
                units.append((b, h, 0, s.G, t0, t1))
                index.append((b, h, si))
    o, l = attend_units(w, units) if units else (None, None)
    out = torch.zeros(s.B, s.H_q, s.D_v, dtype=torch.float64)
    lse = torch.full((s.B, s.H_q), float("-inf"), dtype=torch.float64)
    for b in range(s.B):
        for h in range(s.H_kv):
            sel = [i for i, (bb, hh, _) in enumerate(index) if bb == b and hh == h]
            for g in range(s.G):
                if not sel:
                    continue
                ob, lb = combine(o[sel, g], l[sel, g])
                out[b, h * s.G + g] = ob
                lse[b, h * s.G + g] = lb
    return out, lse
