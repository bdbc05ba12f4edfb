"""Paged-KV decode attention for GB300 (sm_103a).

A thin Python binding over the C ABI in include/decode_attn.h. The entry
points keep the C names without the ``decode_attn_`` prefix; each one only
marshals arguments (tensor data pointers, the current CUDA stream) and calls
the shared library, which runs every step in its own CUDA kernels. There is no
fallback: if the library is missing or was built for another machine, the
import raises.

    desc = Desc.make(B=..., H_kv=..., G=..., D_qk=..., D_v=..., page_size=...,
                     max_pages_per_seq=..., num_pages=..., kv_dtype=KV_BF16)
    meta = torch.empty(sched_meta_bytes(desc), dtype=torch.uint8, device="cuda")
    sched_meta(desc, cache_seqlens, meta)
    fwd(desc, q, k_pool, v_pool, k_scale, v_scale, block_table, cache_seqlens, meta, out, lse)
"""
import ctypes
import os

from . import build as _build_mod

KV_BF16 = 0
KV_FP8 = 1
KV_MLA656 = 2

DA_OK = 0
DA_ERR_NULL = -1
DA_ERR_DIMS = -2
DA_ERR_UNSUPPORTED = -3
DA_ERR_ALIGN = -4
DA_ERR_SPLITS = -5
DA_ERR_META_SIZE = -6
DA_ERR_CUDA = -7
DA_ERR_SCALE = -8

DA_DEV_BAD_PAGE = 1
DA_DEV_SEQ_TOO_LONG = 2
DA_DEV_NEG_LEN = 4
DA_DEV_TIMEOUT = 8
DA_DEV_META_MISMATCH = 16

LIB_PATH = _build_mod.LIB_PATH


class Desc(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("H_kv", ctypes.c_int32), ("G", ctypes.c_int32),
                ("D_qk", ctypes.c_int32), ("D_v", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("max_pages_per_seq", ctypes.c_int32), ("num_pages", ctypes.c_int32),
                ("kv_dtype", ctypes.c_int32), ("splits", ctypes.c_int32), ("num_sms", ctypes.c_int32),
                ("softmax_scale", ctypes.c_float), ("s_q", ctypes.c_int32), ("window", ctypes.c_int32),
                ("topk", ctypes.c_int32)]

    @classmethod
    def make(cls, B, H_kv, G, D_qk, D_v, page_size, max_pages_per_seq, num_pages, kv_dtype=KV_BF16,
             splits=0, num_sms=0, softmax_scale=0.0, s_q=1, window=0, topk=0):
        return cls(B, H_kv, G, D_qk, D_v, page_size, max_pages_per_seq, num_pages, kv_dtype, splits,
                   num_sms, softmax_scale, s_q, window, topk)


class LaunchOpts(ctypes.Structure):
    _fields_ = [("use_pdl", ctypes.c_int32), ("main_begin", ctypes.c_void_p), ("main_end", ctypes.c_void_p),
                ("sinks", ctypes.c_void_p), ("indices", ctypes.c_void_p)]


class DecodeAttnError(RuntimeError):
    pass


_libs = {}


def load_library(path: str = LIB_PATH):
    """Load the shared library (raises if it has not been built). Each path is
    loaded once; the default path is the one every entry point below uses
    unless it is given another handle (``lib=``)."""
    if path in _libs:
        return _libs[path]
    if not os.path.exists(path):
        raise DecodeAttnError(f"CUDA library not built: {path} (run paged_kv_cache_60_gb300/build.py)")
    lib = ctypes.CDLL(path)
    P, I32, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    DP = ctypes.POINTER(Desc)
    lib.decode_attn_sched_meta_bytes.argtypes = [DP, ctypes.POINTER(SZ)]
    lib.decode_attn_meta_offsets.argtypes = [DP, ctypes.POINTER(SZ)]
    lib.decode_attn_num_parts.argtypes = [DP, ctypes.POINTER(I32)]
    lib.decode_attn_sched_meta.argtypes = [DP, P, P, SZ, P]
    lib.decode_attn_fwd.argtypes = [DP, P, P, P, P, P, P, P, P, SZ, P, P, P]
    lib.decode_attn_fwd_ex.argtypes = [DP, P, P, P, P, P, P, P, P, SZ, P, P, ctypes.POINTER(LaunchOpts), P]
    lib.decode_attn_get_error.argtypes = [P, ctypes.POINTER(I32), P]
    lib.decode_attn_append_kv.argtypes = [DP, P, P, ctypes.c_int64, P, P, P, P, P, P, P, P]
    lib.decode_attn_strerror.argtypes = [ctypes.c_int]
    lib.decode_attn_strerror.restype = ctypes.c_char_p
    for f in ("decode_attn_sched_meta_bytes", "decode_attn_meta_offsets", "decode_attn_num_parts",
              "decode_attn_sched_meta", "decode_attn_fwd", "decode_attn_fwd_ex", "decode_attn_get_error",
              "decode_attn_append_kv"):
        getattr(lib, f).restype = ctypes.c_int
    _libs[path] = lib
    return lib


def strerror(code: int) -> str:
    return load_library().decode_attn_strerror(int(code)).decode()


def _check(rc: int):
    if rc != DA_OK:
        raise DecodeAttnError(f"decode_attn error {rc}: {strerror(rc)}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def sched_meta_bytes(desc: Desc) -> int:
    n = ctypes.c_size_t(0)
    _check(load_library().decode_attn_sched_meta_bytes(ctypes.byref(desc), ctypes.byref(n)))
    return n.value


def meta_offsets(desc: Desc):
    offs = (ctypes.c_size_t * 8)()
    _check(load_library().decode_attn_meta_offsets(ctypes.byref(desc), offs))
    return list(offs)


def num_parts(desc: Desc) -> int:
    n = ctypes.c_int32(0)
    _check(load_library().decode_attn_num_parts(ctypes.byref(desc), ctypes.byref(n)))
    return n.value


def sched_meta(desc: Desc, cache_seqlens, meta, stream=None, lib=None):
    _check((lib or load_library()).decode_attn_sched_meta(ctypes.byref(desc), _ptr(cache_seqlens), _ptr(meta),
                                                 meta.numel() * meta.element_size(), _stream(stream)))


def fwd(desc: Desc, q, k_pool, v_pool, k_scale, v_scale, block_table, cache_seqlens, meta, out, lse,
        stream=None, use_pdl=True, main_begin=None, main_end=None, sinks=None, indices=None, lib=None):
    lib = lib or load_library()
    args = (ctypes.byref(desc), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(k_scale), _ptr(v_scale),
            _ptr(block_table), _ptr(cache_seqlens), _ptr(meta), meta.numel() * meta.element_size(),
            _ptr(out), _ptr(lse))
    if use_pdl and main_begin is None and main_end is None and sinks is None and indices is None:
        _check(lib.decode_attn_fwd(*args, _stream(stream)))
    else:
        def ev(e):
            if e is None:
                return None
            if not e.cuda_event:     # torch creates events lazily, at their first record
                e.record()
            return ctypes.c_void_p(e.cuda_event)
        opts = LaunchOpts(1 if use_pdl else 0, ev(main_begin), ev(main_end),
                          None if sinks is None else ctypes.c_void_p(sinks.data_ptr()),
                          None if indices is None else ctypes.c_void_p(indices.data_ptr()))
        _check(lib.decode_attn_fwd_ex(*args, ctypes.byref(opts), _stream(stream)))


def fwd_static_scratch(desc: Desc, q, k_pool, v_pool, k_scale, v_scale, block_table, cache_seqlens, out, lse,
                       stream=None):
    """sched_meta + fwd without any caller scratch, for callers that cannot
    allocate device memory; see decode_attn_fwd_static_scratch in the header
    (fixed 16 MiB library buffer, first call per device before any capture,
    overlapping calls race)."""
    lib = load_library()
    f = lib.decode_attn_fwd_static_scratch
    if f.restype is not ctypes.c_int:
        P = ctypes.c_void_p
        f.argtypes = [ctypes.POINTER(Desc), P, P, P, P, P, P, P, P, P, P]
        f.restype = ctypes.c_int
    _check(f(ctypes.byref(desc), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(k_scale), _ptr(v_scale),
             _ptr(block_table), _ptr(cache_seqlens), _ptr(out), _ptr(lse), _stream(stream)))


def append_kv(desc: Desc, k_new, v_new, positions, block_table, k_pool, v_pool, k_scale=None, v_scale=None,
              device_error=None, new_row_stride=0, stream=None, lib=None):
    """Write each request's new token (bf16 rows of k_new / v_new, v_new None
    for the 656-byte token) into slot positions[b] % page_size of page
    block_table[b][positions[b] // page_size], quantising for e4m3 pools;
    see decode_attn_append_kv in the header. ``device_error``: optional
    device int32 tensor that receives the error bits."""
    _check((lib or load_library()).decode_attn_append_kv(
        ctypes.byref(desc), _ptr(k_new), _ptr(v_new), int(new_row_stride), _ptr(positions), _ptr(block_table),
        _ptr(k_pool), _ptr(v_pool), _ptr(k_scale), _ptr(v_scale), _ptr(device_error), _stream(stream)))


def get_error(meta, stream=None) -> int:
    e = ctypes.c_int32(0)
    _check(load_library().decode_attn_get_error(_ptr(meta), ctypes.byref(e), _stream(stream)))
    return e.value


__all__ = ["Desc", "LaunchOpts", "DecodeAttnError", "load_library", "strerror", "sched_meta_bytes",
           "meta_offsets", "num_parts", "sched_meta", "fwd", "fwd_static_scratch", "append_kv", "get_error", "KV_BF16", "KV_FP8", "KV_MLA656"]
