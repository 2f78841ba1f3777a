"""GPU parity of the output projection with residual (y = O . W_o + x) against the float64 oracle.

The projection alone is fed seeded bf16 inputs; the forward-plus-projection entry point is compared with
the oracle's own forward followed by its projection.  Tolerance: max|y - y_ref| <= rel * max|y_ref - x|
+ 2^-8 * max|y_ref|, i.e. relative to the projected term (so a wrong or missing product cannot hide under
the residual) plus one bf16 rounding of y; rel = 1e-2 for the projection alone (fp32 accumulation) and
2e-2 after the forward, whose bf16 output error (within the forward's own tolerance) passes through W_o.
"""
import numpy as np
import pytest
import torch

from oracle import dsa_oracle as O
from oracle import out_proj as OP
from sparse_mla_attention_dsa_gb300 import workloads as W

from . import _parity as P

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_mla_attention_dsa_gb300 import build
    build.build()


def _close(y, ref, rel, x=None):
    yd = y.float().cpu().numpy().astype(np.float64)
    xd = 0.0 if x is None else x.float().cpu().numpy().astype(np.float64)
    err = float(np.max(np.abs(yd - ref)))
    bound = rel * float(np.max(np.abs(ref - xd))) + 2.0 ** -8 * float(np.max(np.abs(ref)))
    assert np.all(np.isfinite(yd))
    assert err <= bound, (err, bound)


@pytest.mark.parametrize("s_q,h_q,d_model,residual", [
    (37, 16, 64, True),
    (128, 128, 256, True),
    (5, 3, 8, False),
    (300, 64, 1024, True),
])
def test_projection_alone(s_q, h_q, d_model, residual):
    from sparse_mla_attention_dsa_gb300 import api
    w_o, x, o = W.oproj_inputs(31 + s_q, s_q, h_q, d_model, out_sigma=1.0)
    y = api.dsa_out_proj(o.cuda(), w_o.cuda(), x.cuda() if residual else None)
    torch.cuda.synchronize()
    ref = OP.out_proj(P.bits(o), P.bits(w_o), P.bits(x) if residual else None)
    _close(y, ref, 1e-2, x if residual else None)


def test_projection_in_place_residual():
    from sparse_mla_attention_dsa_gb300 import api
    w_o, x, o = W.oproj_inputs(41, 64, 32, 128, out_sigma=1.0)
    xd = x.cuda()
    api.dsa_out_proj(o.cuda(), w_o.cuda(), xd, y=xd)
    torch.cuda.synchronize()
    _close(xd, OP.out_proj(P.bits(o), P.bits(w_o), P.bits(x)), 1e-2, x)


@pytest.mark.parametrize("kv_format", ["bf16", "fp8"])
def test_forward_then_projection(kv_format):
    from sparse_mla_attention_dsa_gb300 import api
    wl = W.small_random(61, 9, 64, 3000, 300, kv_format=kv_format, invalid_frac=0.05)
    w_o, x, _ = W.oproj_inputs(62, wl.s_q, wl.h_q, 256)
    fmt = {"bf16": api.KV_BF16, "fp8": api.KV_FP8}[kv_format]
    y, out, lse = api.dsa_sparse_attn_fwd_oproj(wl.q.cuda(), wl.kv.cuda(), wl.indices.cuda(), wl.sm_scale,
                                                w_o.cuda(), x.cuda(), kv_format=fmt, check_status=True)
    torch.cuda.synchronize()
    ref_out, ref_lse = P.oracle(wl)
    ok, rep = P.compare(out, lse, ref_out, ref_lse, kv_format)
    assert ok, rep
    _close(y, OP.out_proj_f64(ref_out, P.bits(w_o), P.bits(x)), 2e-2, x)


def test_bad_arguments_are_refused():
    from sparse_mla_attention_dsa_gb300 import _lib, api
    lib = _lib.load()
    null = None
    ws = torch.empty(int(lib.dsa_out_proj_workspace_size()), dtype=torch.uint8, device="cuda")
    o = torch.zeros((4, 2, 512), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((1024, 12), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((4, 12), dtype=torch.bfloat16, device="cuda")
    P_ = lambda t: __import__("ctypes").c_void_p(t.data_ptr() if t is not None else 0)
    assert lib.dsa_out_proj(P_(o), P_(w), P_(null), 4, 2, 12, P_(y), P_(ws), ws.numel(), None) == 1  # d_model % 8
    assert lib.dsa_out_proj(P_(o), P_(w), P_(null), 4, 2, 16, P_(y), P_(ws), 1024, None) == 6        # workspace


@pytest.mark.slow
def test_prefill_with_projection_full_size_sampled():
    from sparse_mla_attention_dsa_gb300 import api
    wl = W.prefill_oproj()
    m = wl.meta
    y, out, lse = api.dsa_sparse_attn_fwd_oproj(wl.q.cuda(), wl.kv.cuda(), wl.indices.cuda(), wl.sm_scale,
                                                m["w_o"].cuda(), m["x"].cuda(), check_status=True)
    torch.cuda.synchronize()
    tokens = [0, 1, 1000, 2047, 4095]
    ref_out, ref_lse = P.oracle(wl, tokens)
    ok, rep = P.compare(out[tokens], lse[tokens], ref_out, ref_lse)
    assert ok, rep
    ref_y = OP.out_proj_f64(ref_out, P.bits(m["w_o"]), P.bits(m["x"][tokens]))
    _close(y[tokens], ref_y, 2e-2, m["x"][tokens])
