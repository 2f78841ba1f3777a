"""The C-ABI library builds for sm_103a, loads without a GPU and exports every
symbol include/dsa.h declares; host-side validation answers without a device."""
import ctypes
import os
import re

import pytest

from sparse_mla_attention_dsa_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def _declared_symbols():
    text = open(os.path.join(ROOT, "include", "dsa.h")).read()
    return sorted(set(re.findall(r"DSA_API\s+[\w\s\*]+?\b(dsa_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = _declared_symbols()
    assert {"dsa_sparse_attn_fwd", "dsa_sparse_attn_fwd_fp8kv", "dsa_sparse_attn_fwd_fp4kv",
            "dsa_sparse_attn_fwd_paged", "dsa_sparse_attn_fwd_workspace_size", "dsa_read_device_status",
            "dsa_status_string", "dsa_kernels_per_call"} <= set(names)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_symbols():
        assert hasattr(lib, name), name
    assert set(_declared_symbols()) == set(_lib.SIGNATURES)


def test_status_strings(lib):
    for code, name in _lib.STATUS.items():
        assert lib.dsa_status_string(code).decode() == name
    assert lib.dsa_status_string(99).decode() == "DSA_ERR_UNKNOWN"
    assert lib.dsa_kernels_per_call() == 3


def test_host_validation_needs_no_device(lib):
    f = lib.dsa_sparse_attn_fwd
    null = ctypes.c_void_p(0)
    args = lambda s_q, h_q, s_kv, topk, scale=0.1: (null, null, null, s_q, h_q, s_kv, topk, ctypes.c_float(scale),
                                                    null, null, null, ctypes.c_size_t(0), null)
    assert f(*args(0, 16, 10, 4)) == 0               # nothing to do
    assert f(*args(-1, 16, 10, 4)) == 1              # negative s_q
    assert f(*args(2, 0, 10, 4)) == 1                # h_q out of range
    assert f(*args(2, 129, 10, 4)) == 1
    assert f(*args(2, 16, -1, 4)) == 1
    assert f(*args(2, 16, 10, 0)) == 1               # topk < 1
    assert f(*args(2, 16, 10, 4, float("nan"))) == 1
    assert f(*args(2, 16, 10, 4)) == 1               # null data pointers
    bad = ctypes.c_void_p(0x1008)                     # 8-byte aligned only
    assert f(bad, bad, bad, 2, 16, 10, 4, ctypes.c_float(0.1), bad, bad, bad, ctypes.c_size_t(0), null) == 3
    assert lib.dsa_sparse_attn_fwd_workspace_size(-1, 16, 4, 0) == 0
    assert lib.dsa_sparse_attn_fwd_workspace_size(4, 16, 4, 7) == 0


def test_fp4_and_paged_host_validation_needs_no_device(lib):
    null = ctypes.c_void_p(0)
    f4 = lib.dsa_sparse_attn_fwd_fp4kv
    assert f4(null, null, null, 0, 16, 10, 4, ctypes.c_float(0.1), null, null, null, ctypes.c_size_t(0), null) == 0
    assert f4(null, null, null, 2, 129, 10, 4, ctypes.c_float(0.1), null, null, null, ctypes.c_size_t(0), null) == 1
    assert f4(null, null, null, 2, 16, 10, 4, ctypes.c_float(0.1), null, null, null, ctypes.c_size_t(0), null) == 1

    pg = lib.dsa_sparse_attn_fwd_paged
    ok_ptr = ctypes.c_void_p(0x1000)

    def call(fmt=0, seq=ok_ptr, table=ok_ptr, s_q=2, n_seq=1, max_pages=4, page=16):
        return pg(fmt, null, null, null, seq, table, s_q, 16, 64, 4, n_seq, max_pages, page, ctypes.c_float(0.1),
                  null, null, null, ctypes.c_size_t(0), null)

    assert call(fmt=3) == 1                                   # unknown KV format
    assert call(n_seq=0) == 1 and call(max_pages=0) == 1 and call(page=0) == 1
    assert call(n_seq=1 << 20, max_pages=1 << 12) == 1        # table of 2^32 entries
    assert call(seq=null) == 1 and call(table=null) == 1      # tables needed when there are tokens
    assert call(seq=ctypes.c_void_p(0x1002)) == 3             # int32 tables need 4-byte alignment
    assert call(s_q=0, seq=null, table=null) == 0             # nothing to do
    assert call() == 1                                        # passes the table checks, then null data pointers


def test_host_pipeline_validation_needs_no_device(lib):
    null = ctypes.c_void_p(0)
    h = ctypes.c_void_p(0x1000)
    f = lib.dsa_sparse_attn_fwd_host

    def call(fmt=0, s_q=8, h_q=16, s_kv=64, topk=4, scale=0.1, chunk=4, ptr=h, buf=h, nbytes=1 << 30):
        return f(fmt, ptr, ptr, ptr, s_q, h_q, s_kv, topk, ctypes.c_float(scale), ptr, ptr, buf,
                 ctypes.c_size_t(nbytes), chunk, null)

    assert call(fmt=3) == 1                       # unknown KV format
    assert call(s_q=-1) == 1 and call(h_q=129) == 1 and call(topk=0) == 1 and call(chunk=0) == 1
    assert call(scale=float("nan")) == 1
    assert call(s_q=0, ptr=null, buf=null) == 0   # nothing to do
    assert call(ptr=null) == 1                    # null host buffers
    assert call() == 2                            # valid, but no sm_103 device here: no size, nothing launched
    for bad in ((3, 8, 16, 64, 4, 4), (0, 0, 16, 64, 4, 4), (0, 8, 16, 64, 4, 0), (0, 8, 200, 64, 4, 4)):
        assert lib.dsa_sparse_attn_fwd_host_device_bytes(*bad) == 0


def test_projection_validation_needs_no_device(lib):
    null = ctypes.c_void_p(0)
    h = ctypes.c_void_p(0x1000)
    f = lib.dsa_out_proj
    ws = lib.dsa_out_proj_workspace_size()
    assert ws >= (1 << 20)

    def call(s_q=4, h_q=2, d_model=16, o=h, w=h, x=null, y=h, buf=h, nbytes=ws):
        return f(o, w, x, s_q, h_q, d_model, y, buf, ctypes.c_size_t(nbytes), null)

    assert call(s_q=0, o=null, w=null, y=null, buf=null) == 0      # nothing to do
    assert call(d_model=12) == 1 and call(d_model=0) == 1 and call(h_q=0) == 1 and call(h_q=129) == 1
    assert call(s_q=-1) == 1 and call(o=null) == 1 and call(y=null) == 1
    assert call(x=ctypes.c_void_p(0x1008)) == 3                     # residual not 16-byte aligned
    assert call(nbytes=ws - 1) == 6 and call(buf=null) == 6          # workspace
    fused = lib.dsa_sparse_attn_fwd_oproj
    args = [null, null, null, 2, 16, 10, 4, ctypes.c_float(0.1), h, null, 16, h, h, h, h, ctypes.c_size_t(1 << 30), null]
    assert fused(3, *args) == 1                                      # unknown KV format
    bad_d = list(args); bad_d[10] = 20
    assert fused(0, *bad_d) == 1                                     # d_model not a multiple of 8
    assert fused(0, *args) == 2                                      # valid, but no sm_103 device here
