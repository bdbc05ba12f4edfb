"""Helpers for the GPU tests: move a workload to the device, call the library
through its C ABI binding, read back the scheduling metadata."""
import ctypes
import os

import torch

import paged_kv_cache_60_gb300 as da
from paged_kv_cache_60_gb300 import build as dabuild

OUT_TOL = 2e-2      # max |out - oracle| (bf16 output, fp32 accumulation)
LSE_TOL = 1e-4      # max |lse - oracle|


def ensure_built():
    dabuild.build()
    return da.load_library()


TRACE_DIR = os.path.join(os.path.dirname(os.path.dirname(dabuild.LIB_PATH)), "_build_trace")
_trace_lib = None


def debug_build_library():
    """The library compiled with -DDA_PAGE_TRACE into its own directory (built
    once per process): it adds decode_attn_debug_page_trace,
    decode_attn_debug_wait_limit and decode_attn_debug_stall to the product
    entry points."""
    global _trace_lib
    if _trace_lib is None:
        path = dabuild.build(extra_flags=("-DDA_PAGE_TRACE",), out_dir=TRACE_DIR)
        lib = da.load_library(path)
        lib.decode_attn_debug_page_trace.argtypes = [ctypes.c_void_p, ctypes.c_int32]
        lib.decode_attn_debug_page_trace.restype = ctypes.c_int
        lib.decode_attn_debug_wait_limit.argtypes = [ctypes.c_uint64]
        lib.decode_attn_debug_wait_limit.restype = ctypes.c_int
        lib.decode_attn_debug_stall.argtypes = [ctypes.c_int32]
        lib.decode_attn_debug_stall.restype = ctypes.c_int
        _trace_lib = lib
    return _trace_lib


def device_sms() -> int:
    return torch.cuda.get_device_properties(0).multi_processor_count


def auto_slots(spec) -> int:
    """SM slots the library's automatic partition counts for a GQA workload:
    the bf16 D = 64 build for three or four query tokens runs two CTAs per SM."""
    two = spec.kv_dtype == 0 and spec.D_qk == 64 and spec.s_q in (3, 4)
    return device_sms() * (2 if two else 1)


def make_desc(w, splits=None, num_sms=0):
    s = w.spec
    return da.Desc.make(B=s.B, H_kv=s.H_kv, G=s.G, D_qk=s.D_qk, D_v=s.D_v, page_size=s.page_size,
                        max_pages_per_seq=w.max_pages_per_seq, num_pages=w.num_pages, kv_dtype=s.kv_dtype,
                        splits=s.splits if splits is None else splits, num_sms=num_sms,
                        softmax_scale=s.softmax_scale, s_q=s.s_q, window=s.window, topk=s.topk)


class DeviceWorkload:
    def __init__(self, w, dev="cuda"):
        self.w = w
        self.q = w.q.to(dev)
        self.k_pool = w.k_pool.to(dev)
        self.v_pool = w.v_pool.to(dev) if w.v_pool is not None else None
        self.k_scale = w.k_scale.to(dev) if w.k_scale is not None else None
        self.v_scale = w.v_scale.to(dev) if w.v_scale is not None else None
        self.block_table = w.block_table.to(dev)
        self.cache_seqlens = w.cache_seqlens.to(dev)
        self.sinks = w.sinks.to(dev) if getattr(w, "sinks", None) is not None else None
        self.indices = w.indices.to(dev) if getattr(w, "indices", None) is not None else None


def run(w, splits=None, num_sms=0, dw=None, meta=None, desc=None, out=None, lse=None, stream=None):
    """Run sched_meta + fwd; returns (out bf16 [B,H_q,D_v], lse f32 [B,H_q], meta, desc)."""
    ensure_built()
    dw = dw or DeviceWorkload(w)
    desc = desc or make_desc(w, splits, num_sms)
    s = w.spec
    if meta is None:
        meta = torch.empty(da.sched_meta_bytes(desc), dtype=torch.uint8, device="cuda")
        da.sched_meta(desc, dw.cache_seqlens, meta, stream=stream)
    rows = (s.B, s.H_q) if s.s_q == 1 else (s.B, s.s_q, s.H_q)
    if out is None:
        out = torch.full(rows + (s.D_v,), float("nan"), dtype=torch.bfloat16, device="cuda")
    if lse is None:
        lse = torch.full(rows, float("nan"), dtype=torch.float32, device="cuda")
    da.fwd(desc, dw.q, dw.k_pool, dw.v_pool, dw.k_scale, dw.v_scale, dw.block_table, dw.cache_seqlens,
           meta, out, lse, stream=stream, sinks=dw.sinks, indices=dw.indices)
    return out, lse, meta, desc


def read_meta(meta, desc):
    offs = da.meta_offsets(desc)
    m = meta.cpu()

    def i32(a, n):
        return m[offs[a]:offs[a] + 4 * n].view(torch.int32).tolist()
    header = i32(0, 16)
    nparts = header[5]
    recs = m[offs[1]:offs[1] + 32 * nparts].view(torch.int32).view(nparts, 8).tolist()
    B = desc.B
    return dict(header=header, parts=[tuple(p[:4]) for p in recs], part_extra=[tuple(p[4:]) for p in recs],
                chunk_offset=i32(2, B + 1),
                split_offset=i32(3, B + 1), num_splits=i32(4, B))


def expected_part_extra(ref, seqlens, max_len):
    """The four cached per-part fields, derived from the oracle's arrays."""
    out = []
    for (b0, s0, c0, c1) in ref.parts:
        if b0 < 0:
            out.append((0, 0, 0, 0))
        else:
            out.append((ref.chunk_offset[b0], min(max(seqlens[b0], 0), max_len), ref.split_offset[b0],
                        ref.num_splits[b0]))
    return out


def max_err(out, lse, ref_out, ref_lse, heads=None, G=None):
    """max |out - ref| and max |lse - ref| over finite reference entries;
    -inf lse must match exactly."""
    o = out.float().cpu().double()
    l = lse.float().cpu().double()
    sel = ~torch.isnan(ref_lse)
    if heads is not None:
        pass
    ro = ref_out[sel]
    rl = ref_lse[sel]
    oo = o[sel]
    ll = l[sel]
    ninf = torch.isneginf(rl)
    assert torch.equal(torch.isneginf(ll), ninf), "lse -inf pattern differs"
    e_out = (oo - ro).abs().max().item() if ro.numel() else 0.0
    fin = ~ninf
    e_lse = (ll[fin] - rl[fin]).abs().max().item() if fin.any() else 0.0
    if torch.isnan(oo).any():
        e_out = float("inf")
    return e_out, e_lse
