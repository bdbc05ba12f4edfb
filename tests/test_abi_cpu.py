"""C ABI checks that need no GPU: the library builds and loads, exports every
function include/decode_attn.h declares, and rejects bad arguments on the host
with the documented codes before any CUDA call."""
import ctypes
import os
import re

import pytest

import paged_kv_cache_60_gb300 as da
from paged_kv_cache_60_gb300 import build as dabuild
from oracle.sched_ref import auto_num_parts

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    dabuild.build()
    return da.load_library()


def _header_functions():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            # declarations of the page-trace test build are not in the product library
            src = re.sub(r"#ifdef DA_PAGE_TRACE.*?#endif", "", src, flags=re.S)
            names |= set(re.findall(r"\b(decode_attn_\w+)\s*\(", src))
    return sorted(names)


def test_library_exports_every_declared_function(lib):
    names = _header_functions()
    assert len(names) >= 8
    for n in names:
        assert hasattr(lib, n), n


def _desc(**kw):
    base = dict(B=4, H_kv=2, G=8, D_qk=128, D_v=128, page_size=16, max_pages_per_seq=10, num_pages=40,
                kv_dtype=da.KV_BF16, splits=0, num_sms=152)
    base.update(kw)
    return da.Desc.make(**base)


def test_sched_meta_bytes_and_parts_host_only(lib):
    d = _desc()
    n = da.sched_meta_bytes(d)
    offs = da.meta_offsets(d)
    assert offs[7] == n and offs[0] == 0 and offs[1] == 128
    assert all(o % 16 == 0 for o in offs)
    assert offs[5] % 256 == 0 and offs[6] % 256 == 0
    assert da.num_parts(d) == auto_num_parts(152, 2, 1) == 76
    parts = 76
    max_splits = parts + 4
    assert offs[6] - offs[5] >= max_splits * 16 * 4
    assert n - offs[6] >= max_splits * 16 * 128 * 4
    d2 = _desc(splits=8)
    assert da.num_parts(d2) == 32


@pytest.mark.parametrize("field,value,code", [
    ("B", 0, -2), ("H_kv", 0, -2), ("page_size", 12, -3), ("G", 4, -3), ("D_qk", 96, -3),
    ("splits", -1, -5), ("kv_dtype", 7, -3), ("max_pages_per_seq", 0, -2),
])
def test_bad_desc_codes(lib, field, value, code):
    d = _desc(**{field: value})
    n = ctypes.c_size_t(0)
    assert lib.decode_attn_sched_meta_bytes(ctypes.byref(d), ctypes.byref(n)) == code


def test_fp8_needs_d128_and_mla_shape(lib):
    n = ctypes.c_size_t(0)
    assert lib.decode_attn_sched_meta_bytes(ctypes.byref(_desc(kv_dtype=da.KV_FP8, D_qk=64, D_v=64)),
                                            ctypes.byref(n)) == -3
    assert lib.decode_attn_sched_meta_bytes(ctypes.byref(_desc(kv_dtype=da.KV_FP8)), ctypes.byref(n)) == 0


def test_fwd_rejects_null_and_misaligned_before_launch(lib):
    d = _desc()
    n = da.sched_meta_bytes(d)
    P = ctypes.c_void_p
    good = P(0x10000)
    bad = P(0x10008)
    args = lambda q=good, meta=good: (ctypes.byref(d), q, good, good, None, None, good, good, meta, n,  # noqa: E731
                                      good, good, None)
    assert lib.decode_attn_fwd(*args(q=None)) == -1
    assert lib.decode_attn_fwd(*args(q=bad)) == -4
    assert lib.decode_attn_fwd(ctypes.byref(d), good, good, good, None, None, good, good, good, n - 16,
                               good, good, None) == -6
    dq = _desc(kv_dtype=da.KV_FP8)
    nq = da.sched_meta_bytes(dq)
    assert lib.decode_attn_fwd(ctypes.byref(dq), good, good, good, None, None, good, good, good, nq,
                               good, good, None) == -8


def test_strerror_is_total(lib):
    for c in range(-10, 2):
        assert isinstance(da.strerror(c), str) and da.strerror(c)


def test_append_rejects_bad_arguments_before_launch(lib):
    P = ctypes.c_void_p
    g = P(0x10000)
    f = lib.decode_attn_append_kv

    def call(d, k_new=g, v_new=g, stride=0, pos=g, bt=g, kp=g, vp=g, ks=None, vs=None, err=None):
        return f(ctypes.byref(d), k_new, v_new, stride, pos, bt, kp, vp, ks, vs, err, None)

    d = _desc()
    assert call(d, k_new=None) == -1
    assert call(d, v_new=None) == -1
    assert call(d, vp=None) == -1
    assert call(d, k_new=P(0x10008)) == -4
    assert call(d, err=P(0x10002)) == -4
    assert call(d, stride=100) == -2            # below the row of H_kv * D values
    assert call(d, stride=2 * 128 + 4) == -2    # not a multiple of 8 elements
    assert call(_desc(D_qk=100, D_v=100)) == -3
    assert call(_desc(D_qk=128, D_v=64)) == -3
    assert call(_desc(B=0)) == -2
    assert call(_desc(kv_dtype=da.KV_FP8)) == -8
    dm = _desc(kv_dtype=da.KV_MLA656, H_kv=1, G=128, D_qk=576, D_v=512)
    assert call(dm) == -3                        # the latent token takes no v_new
    assert call(dm, v_new=None, vp=P(0x20000)) == -3
    assert call(_desc(kv_dtype=da.KV_MLA656, H_kv=2, G=128, D_qk=576, D_v=512), v_new=None, vp=None) == -3


def test_s_q_limits_and_partial_sizes(lib):
    n = ctypes.c_size_t(0)

    def rc(**kw):
        return lib.decode_attn_sched_meta_bytes(ctypes.byref(_desc(**kw)), ctypes.byref(n))
    assert rc(s_q=0) == 0 and rc(s_q=1) == 0 and rc(s_q=2) == 0
    assert rc(s_q=3) == 0 and rc(s_q=4) == 0 and rc(s_q=5) == -3   # up to 4 query tokens
    assert rc(D_qk=64, D_v=64, s_q=4) == 0 and rc(D_qk=64, D_v=64, s_q=5) == -3
    assert rc(kv_dtype=da.KV_FP8, s_q=4) == 0 and rc(kv_dtype=da.KV_FP8, s_q=5) == -3
    assert rc(s_q=-1) == -2
    # the split partials hold one row per (draft, query head)
    o1, o2 = da.meta_offsets(_desc()), da.meta_offsets(_desc(s_q=2))
    assert o1[:6] == o2[:6]
    assert (o2[6] - o2[5]) >= 2 * (o1[6] - o1[5]) - 256
    assert (o2[7] - o2[6]) >= 2 * (o1[7] - o1[6]) - 256


def test_window_topk_sinks_argument_checks(lib):
    n = ctypes.c_size_t(0)

    def rc(**kw):
        return lib.decode_attn_sched_meta_bytes(ctypes.byref(_desc(**kw)), ctypes.byref(n))
    assert rc(window=-1) == -2
    assert rc(window=4096) == 0
    assert rc(topk=64) == -3                       # sparse decode is for the 656-byte format
    assert rc(topk=-1) == -2
    # sparse decode without a position list, and sinks with the latent format: refused before launch
    d = _desc(kv_dtype=da.KV_MLA656, H_kv=1, G=128, D_qk=576, D_v=512, topk=64)
    if lib.decode_attn_sched_meta_bytes(ctypes.byref(d), ctypes.byref(n)) == 0:
        P = ctypes.c_void_p
        g = P(0x10000)
        opts = da.LaunchOpts(1, None, None, None, None)
        assert lib.decode_attn_fwd_ex(ctypes.byref(d), g, g, None, None, None, g, g, g, n.value, g, g,
                                      ctypes.byref(opts), None) == -1
        dm = _desc(kv_dtype=da.KV_MLA656, H_kv=1, G=128, D_qk=576, D_v=512)
        nm = ctypes.c_size_t(0)
        assert lib.decode_attn_sched_meta_bytes(ctypes.byref(dm), ctypes.byref(nm)) == 0
        opts = da.LaunchOpts(1, None, None, g, None)
        assert lib.decode_attn_fwd_ex(ctypes.byref(dm), g, g, None, None, None, g, g, g, nm.value, g, g,
                                      ctypes.byref(opts), None) == -3
    # misaligned sinks pointer
    d = _desc()
    nb = da.sched_meta_bytes(d)
    g = ctypes.c_void_p(0x10000)
    opts = da.LaunchOpts(1, None, None, ctypes.c_void_p(0x10002), None)
    assert lib.decode_attn_fwd_ex(ctypes.byref(d), g, g, g, None, None, g, g, g, nb, g, g, ctypes.byref(opts),
                                  None) == -4
