"""Helpers for GPU-vs-oracle parity tests (tolerances written here, used by every test).

Tolerances: lse within 2e-3 absolute; out max-abs error <= 1e-2 * max|out_ref| + 1e-3
for a bf16 KV cache and <= 3e-2 * max|out_ref| for an FP8 or FP4 cache (the oracle is
fed the dequantised rows, so the quantised-cache bound covers the bf16 rounding of P
and of the dequantised values before the tensor cores).
"""
import numpy as np
import torch

from oracle import dsa_oracle as O

LSE_ABS = 2e-3
OUT_REL_BF16, OUT_ABS_BF16 = 1e-2, 1e-3
OUT_REL_FP8, OUT_ABS_FP8 = 3e-2, 0.0


def bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def kv_raw(wl) -> np.ndarray:
    return bits(wl.kv) if wl.kv_format == "bf16" else wl.kv.numpy()


def oracle(wl, tokens=None):
    tokens = list(range(wl.s_q)) if tokens is None else list(tokens)
    return O.sparse_mla_fwd_sampled(bits(wl.q), kv_raw(wl), wl.kv_format, wl.indices.numpy(), wl.sm_scale, tokens)


def oracle_paged(wl, tokens=None):
    """The definition over a paged workload: logical positions -> pool rows by the oracle's own translation."""
    from oracle import paged as PG
    tokens = list(range(wl.s_q)) if tokens is None else list(tokens)
    rows = PG.logical_to_rows(wl.indices.numpy(), wl.meta["seq_of_token"].numpy(), wl.meta["block_table"].numpy(),
                              wl.meta["page_size"], wl.kv.shape[0])
    return O.sparse_mla_fwd_sampled(bits(wl.q), kv_raw(wl), wl.kv_format, rows, wl.sm_scale, tokens)


def run_gpu_paged(wl, device="cuda"):
    from sparse_mla_attention_dsa_gb300 import api
    fmt = {"bf16": api.KV_BF16, "fp8": api.KV_FP8, "fp4": api.KV_FP4}[wl.kv_format]
    out, lse = api.dsa_sparse_attn_fwd_paged(wl.q.to(device), wl.kv.to(device), wl.indices.to(device),
                                             wl.meta["seq_of_token"].to(device), wl.meta["block_table"].to(device),
                                             wl.meta["page_size"], wl.sm_scale, kv_format=fmt, check_status=True)
    torch.cuda.synchronize()
    return out, lse


def run_gpu(wl, device="cuda"):
    from sparse_mla_attention_dsa_gb300 import api
    q = wl.q.to(device)
    kv = wl.kv.to(device)
    idx = wl.indices.to(device)
    fn = {"bf16": api.dsa_sparse_attn_fwd, "fp8": api.dsa_sparse_attn_fwd_fp8kv,
          "fp4": api.dsa_sparse_attn_fwd_fp4kv}[wl.kv_format]
    out, lse = fn(q, kv, idx, wl.sm_scale, check_status=True)
    torch.cuda.synchronize()
    return out, lse


def compare(out_gpu, lse_gpu, ref_out, ref_lse, kv_format="bf16"):
    """Returns (ok, report) for GPU outputs (torch, any device) against float64 references."""
    o = out_gpu.float().cpu().numpy().astype(np.float64)
    l = lse_gpu.float().cpu().numpy().astype(np.float64)
    fin = np.isfinite(ref_lse)
    rep = {}
    ok = bool(np.array_equal(np.isfinite(l), fin))
    rep["lse_inf_match"] = ok
    if fin.any():
        rep["lse_err"] = float(np.max(np.abs(l[fin] - ref_lse[fin])))
        ok &= rep["lse_err"] <= LSE_ABS
    ok &= bool(np.all(np.isneginf(l[~fin])))
    ref_max = float(np.max(np.abs(ref_out), initial=0.0))
    rep["out_err"] = float(np.max(np.abs(o - ref_out), initial=0.0))
    rep["out_ref_max"] = ref_max
    rel, ab = (OUT_REL_BF16, OUT_ABS_BF16) if kv_format == "bf16" else (OUT_REL_FP8, OUT_ABS_FP8)
    rep["out_bound"] = rel * ref_max + ab
    ok &= rep["out_err"] <= rep["out_bound"]
    ok &= bool(np.all(np.isfinite(o)))
    return ok, rep
