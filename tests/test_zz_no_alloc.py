"""The allocation-free forward entry point against the regular one.

`dsa_sparse_attn_fwd_noalloc` serves callers that cannot allocate device memory
(for instance code running inside an allocator of its own, or a plugin that is
handed only its input and output buffers): it runs the same forward on a
scratch array built into the library instead of a caller workspace.  This file
runs last so that a stop at the first failure has already run every other test.
"""
import ctypes

import pytest
import torch

from sparse_mla_attention_dsa_gb300 import _lib
from sparse_mla_attention_dsa_gb300 import workloads as W

from . import _parity as P

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_mla_attention_dsa_gb300 import build
    build.build()
    return _lib.load()


def _noalloc(lib, wl):
    q, kv, idx = wl.q.cuda(), wl.kv.cuda(), wl.indices.cuda()
    out = torch.empty((wl.s_q, wl.h_q, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((wl.s_q, wl.h_q), dtype=torch.float32, device="cuda")
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    st = lib.dsa_sparse_attn_fwd_noalloc(p(q), p(kv), p(idx), wl.s_q, wl.h_q, wl.s_kv, wl.topk,
                                         ctypes.c_float(wl.sm_scale), p(out), p(lse),
                                         ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, _lib.STATUS.get(st, st)
    torch.cuda.synchronize()
    return out, lse


def test_noalloc_matches_the_workspace_entry_point_on_two_calls(lib):
    from sparse_mla_attention_dsa_gb300 import api
    # two calls in a row on different shapes: the second sees whatever the first left in the scratch
    cases = [W.small_random(101, 300, 128, 4096, 256, invalid_frac=0.02),   # tokens split across SM pairs
             W.small_random(102, 9, 64, 1500, 190, invalid_frac=0.1)]
    for wl in cases:
        out_n, lse_n = _noalloc(lib, wl)
        out_r, lse_r = api.dsa_sparse_attn_fwd(wl.q.cuda(), wl.kv.cuda(), wl.indices.cuda(), wl.sm_scale,
                                               check_status=True)
        torch.cuda.synchronize()
        ok, rep = P.compare(out_n, lse_n, out_r.double().cpu().numpy(), lse_r.double().cpu().numpy(), "bf16")
        assert ok, rep


def test_noalloc_rejects_sizes_beyond_its_scratch(lib):
    null = ctypes.c_void_p(16)
    st = lib.dsa_sparse_attn_fwd_noalloc(null, null, null, 8193, 128, 10, 4, ctypes.c_float(0.1), null, null,
                                         ctypes.c_void_p(0))
    assert _lib.STATUS[st] == "DSA_ERR_WORKSPACE"
