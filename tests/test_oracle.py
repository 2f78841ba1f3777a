"""Pins of the CPU oracle against facts that do not come from the oracle itself.

The forward's definition is "Ascend Sparse Attention Forward 算法与优化技术简析",
section "数学建模"; the blockwise algorithm is section "计算流程".  Each test
below fixes the oracle to something independent: a hand-derived example, closed
forms, invariants of the definition, a brute-force formulation over all KV rows
with multiplicities computed by torch's float64 routines, or library decoders.
"""
import math
import os

import numpy as np
import pytest
import torch

from oracle import dsa_oracle as O
from oracle import emu as E
from oracle import formats as F
from sparse_mla_attention_dsa_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _f64(wl):
    return O.q_to_f64(_bits(wl.q)), O.kv_to_f64(wl.kv.numpy() if wl.kv_format == "fp8" else _bits(wl.kv), wl.kv_format)


# --------------------------------------------------------------------------- formats

def test_bf16_decoder_matches_torch_on_all_patterns():
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    mine = F.bf16_bits_to_f64(pats)
    ref = torch.from_numpy(pats.view(np.int16)).view(torch.bfloat16).double().numpy()
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(mine[ok], ref[ok])


def test_e4m3_decoder_matches_torch_on_all_256_codes():
    codes = np.arange(256, dtype=np.uint8)
    mine = F.e4m3_to_f64(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(mine[ok], ref[ok])
    # the format's fixed points
    assert F.e4m3_to_f64(np.array([0x7E], np.uint8))[0] == 448.0
    assert F.e4m3_to_f64(np.array([0x01], np.uint8))[0] == 2.0 ** -9
    assert F.e4m3_to_f64(np.array([0x38], np.uint8))[0] == 1.0
    assert np.isnan(F.e4m3_to_f64(np.array([0xFF], np.uint8))[0])


def test_fp8_row_layout_round_trip():
    rng = np.random.default_rng(5)
    lat = torch.from_numpy(rng.standard_normal((33, 512), dtype=np.float32))
    lat[3, 128:256] = 0.0  # an all-zero group takes scale 1
    rope = torch.from_numpy(rng.standard_normal((33, 64), dtype=np.float32)).to(torch.bfloat16)
    rows = W.quantize_fp8_rows(lat, rope).numpy()
    dec = F.fp8_rows_to_f64(rows)
    # independent route: torch's float8 view, float32 product, torch's bf16 rounding
    codes = torch.from_numpy(rows[:, :512].copy()).view(torch.float8_e4m3fn).float()
    scales = torch.from_numpy(rows[:, 512:528].copy()).view(torch.float32)
    ref_lat = (codes * scales.repeat_interleave(128, dim=1)).to(torch.bfloat16).double()
    assert np.array_equal(dec[:, :512], ref_lat.numpy())
    assert np.array_equal(dec[:, 512:], rope.double().numpy())
    assert scales[3, 1].item() == 1.0
    # e4m3 (3 mantissa bits) then bf16: at most 2^-4 + 2^-8 relative, plus the subnormal step
    err = np.abs(dec[:, :512] - lat.double().numpy())
    bound = np.abs(lat.double().numpy()) * (2.0 ** -4 + 2.0 ** -8) + 2.0 ** -9 * float(scales.max())
    assert np.all(err <= bound)


def test_round_to_bf16_matches_torch():
    rng = np.random.default_rng(7)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 100,
                        np.exp(rng.uniform(-80, 80, 10000)).astype(np.float32),
                        np.array([0.0, -0.0, 1.0, 1.00390625, 1.01171875], np.float32)])
    mine = E.round_to_bf16(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    assert np.array_equal(mine, ref)


# --------------------------------------------------------------------------- the definition

def _golden():
    vals = {}
    with open(os.path.join(GOLDEN, "two_valid_rows.txt")) as f:
        for line in f:
            if line.startswith("#") or line.startswith("key") or not line.strip():
                continue
            k, v = line.split()
            vals[k] = float(v)
    return vals


def test_hand_worked_example():
    g = _golden()
    q = np.zeros((1, 576))
    q[0, 0], q[0, 512] = 1.0, 0.5
    kv = np.zeros((3, 576))
    kv[0, 0], kv[0, 1], kv[0, 511], kv[0, 512] = 2.0, 1.0, -3.0, 5.0
    kv[1, 1], kv[1, 512] = 4.0, -2.0
    kv[2, 0] = 7.0
    out, lse = O.sparse_mla_fwd_token(q, kv, np.array([0, -1, 1, 3]), 0.5)
    assert out.shape == (1, 512)
    assert abs(lse[0] - g["lse"]) < 1e-14
    assert abs(out[0, 0] - g["out0"]) < 1e-14
    assert abs(out[0, 1] - g["out1"]) < 1e-14
    assert abs(out[0, 511] - g["out511"]) < 1e-14
    rest = np.delete(out[0], [0, 1, 511])
    assert np.all(rest == 0.0)


def _dense_torch(q, kv, idx, sm_scale):
    """Brute force over ALL KV rows with multiplicity weights, torch float64."""
    qt, kvt = torch.from_numpy(q), torch.from_numpy(kv)
    s_kv = kv.shape[0]
    idx = np.asarray(idx)
    valid = idx[(idx >= 0) & (idx < s_kv)]
    w = torch.from_numpy(np.bincount(valid, minlength=s_kv).astype(np.float64))
    logits = torch.matmul(qt, kvt.T) * sm_scale + torch.log(w)[None, :]
    lse = torch.logsumexp(logits, dim=-1)
    out = torch.matmul(torch.softmax(logits, dim=-1), kvt[:, :512])
    return out.numpy(), lse.numpy()


@pytest.mark.parametrize("seed,h_q,s_kv,topk,bad", [(0, 16, 256, 64, 0.0), (1, 8, 100, 37, 0.2),
                                                   (2, 3, 40, 40, 0.5), (3, 1, 2000, 300, 0.05)])
def test_definition_matches_dense_bruteforce(seed, h_q, s_kv, topk, bad):
    wl = W.small_random(seed, 3, h_q, s_kv, topk, invalid_frac=bad)
    q, kv = _f64(wl)
    idx = wl.indices.numpy()
    out, lse = O.sparse_mla_fwd(q, kv, idx, wl.sm_scale)
    for t in range(q.shape[0]):
        ro, rl = _dense_torch(q[t], kv, idx[t], wl.sm_scale)
        assert np.allclose(lse[t], rl, rtol=1e-12, atol=1e-12)
        assert np.allclose(out[t], ro, rtol=1e-11, atol=1e-12)


def test_duplicates_count_with_multiplicity():
    rng = np.random.default_rng(3)
    q = rng.standard_normal((4, 576))
    kv = rng.standard_normal((10, 576))
    out, lse = O.sparse_mla_fwd_token(q, kv, np.array([2, 2, 7]), 0.1)
    la, lb = 0.1 * q @ kv[2], 0.1 * q @ kv[7]
    den = 2 * np.exp(la) + np.exp(lb)
    ref = (2 * np.exp(la)[:, None] * kv[2, :512] + np.exp(lb)[:, None] * kv[7, :512]) / den[:, None]
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-13)
    assert np.allclose(lse, np.log(den), rtol=1e-13)


def test_permutation_and_padding_invariance():
    wl = W.small_random(11, 2, 12, 500, 129, invalid_frac=0.1)
    q, kv = _f64(wl)
    idx = wl.indices.numpy().astype(np.int64)
    out, lse = O.sparse_mla_fwd(q, kv, idx, wl.sm_scale)
    rng = np.random.default_rng(0)
    perm = np.stack([rng.permutation(r) for r in idx])
    out_p, lse_p = O.sparse_mla_fwd(q, kv, perm, wl.sm_scale)
    assert np.allclose(out, out_p, rtol=1e-12, atol=1e-13) and np.allclose(lse, lse_p, rtol=1e-13)
    # interleave -1 and out-of-range values
    pad = np.concatenate([idx, np.full((2, 50), -1), np.full((2, 7), 500), np.full((2, 3), 2 ** 31 - 1)], axis=1)
    pad = np.stack([rng.permutation(r) for r in pad])
    out_d, lse_d = O.sparse_mla_fwd(q, kv, pad, wl.sm_scale)
    assert np.allclose(out, out_d, rtol=1e-12, atol=1e-13) and np.allclose(lse, lse_d, rtol=1e-13)


def test_equal_rows_closed_form():
    """All selected rows equal r: out = r[:512], lse = ln(n_valid) + sm_scale * q.r."""
    rng = np.random.default_rng(4)
    q = rng.standard_normal((5, 576))
    r = rng.standard_normal(576)
    kv = rng.standard_normal((64, 576))
    sel = np.array([3, 9, 10, 20, 33, 40, 41])
    kv[sel] = r
    idx = np.concatenate([sel, [-1, -1, 64]])
    out, lse = O.sparse_mla_fwd_token(q, kv, idx, 0.125)
    assert np.allclose(out, np.broadcast_to(r[:512], out.shape), rtol=1e-12, atol=1e-12)
    assert np.allclose(lse, math.log(len(sel)) + 0.125 * q @ r, rtol=1e-13, atol=1e-13)


def test_single_and_two_valid_closed_forms():
    rng = np.random.default_rng(8)
    q = rng.standard_normal((6, 576))
    kv = rng.standard_normal((30, 576))
    out, lse = O.sparse_mla_fwd_token(q, kv, np.array([-1, 17, -1]), 0.2)
    assert np.allclose(out, np.broadcast_to(kv[17, :512], out.shape), rtol=1e-13, atol=1e-13)
    assert np.allclose(lse, 0.2 * q @ kv[17], rtol=1e-13, atol=1e-13)
    out, lse = O.sparse_mla_fwd_token(q, kv, np.array([4, 29]), 0.2)
    l1, l2 = 0.2 * q @ kv[4], 0.2 * q @ kv[29]
    s1 = 1.0 / (1.0 + np.exp(l2 - l1))
    ref = s1[:, None] * kv[4, :512] + (1 - s1)[:, None] * kv[29, :512]
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-13)
    assert np.allclose(lse, np.logaddexp(l1, l2), rtol=1e-13)


def test_no_valid_index_gives_zero_and_minus_inf():
    q = np.ones((3, 576))
    kv = np.ones((5, 576))
    out, lse = O.sparse_mla_fwd_token(q, kv, np.array([-1, 5, 99, -7]), 1.0)
    assert np.all(out == 0.0) and np.all(np.isneginf(lse))
    out, lse = O.sparse_mla_fwd_token(q, np.zeros((0, 576)), np.array([0, 1]), 1.0)
    assert np.all(out == 0.0) and np.all(np.isneginf(lse))


def test_scale_moves_between_q_and_sm_scale():
    wl = W.small_random(21, 2, 4, 64, 32)
    q, kv = _f64(wl)
    idx = wl.indices.numpy()
    a = O.sparse_mla_fwd(q, kv, idx, 0.25)
    b = O.sparse_mla_fwd(q * 0.25, kv, idx, 1.0)
    assert np.allclose(a[0], b[0], rtol=1e-12, atol=1e-13) and np.allclose(a[1], b[1], rtol=1e-12, atol=1e-13)


def test_sampled_route_equals_full_route():
    wl = W.small_random(31, 5, 8, 300, 90, invalid_frac=0.1)
    q, kv = _f64(wl)
    idx = wl.indices.numpy()
    full = O.sparse_mla_fwd(q, kv, idx, wl.sm_scale, tokens=[1, 3, 4])
    samp = O.sparse_mla_fwd_sampled(_bits(wl.q), _bits(wl.kv), "bf16", idx, wl.sm_scale, [1, 3, 4])
    assert np.array_equal(full[0], samp[0]) and np.array_equal(full[1], samp[1])


def test_fp8_definition_uses_dequantised_rows():
    wl = W.small_random(41, 3, 16, 200, 70, kv_format="fp8", q_sigma=2.0)
    q = O.q_to_f64(_bits(wl.q))
    rows = wl.kv.numpy()
    kv = O.kv_to_f64(rows, "fp8")
    idx = wl.indices.numpy()
    out, lse = O.sparse_mla_fwd(q, kv, idx, wl.sm_scale)
    codes = torch.from_numpy(rows[:, :512].copy()).view(torch.float8_e4m3fn).float()
    sc = torch.from_numpy(rows[:, 512:528].copy()).view(torch.float32)
    rope = torch.from_numpy(rows[:, 528:].copy()).view(torch.bfloat16).double()
    lat = (codes * sc.repeat_interleave(128, 1)).to(torch.bfloat16).double()
    kv_t = torch.cat([lat, rope], dim=1).numpy()
    for t in range(3):
        ro, rl = _dense_torch(q[t], kv_t, idx[t], wl.sm_scale)
        assert np.allclose(out[t], ro, rtol=1e-11, atol=1e-12) and np.allclose(lse[t], rl, rtol=1e-12)


# --------------------------------------------------------------------------- the blockwise algorithm

def _tol_ok(out, lse, ref_out, ref_lse, rel=1e-2, abs_=1e-3, lse_abs=2e-3):
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(lse), fin)
    assert np.max(np.abs(lse[fin] - ref_lse[fin]), initial=0.0) <= lse_abs
    return np.max(np.abs(out - ref_out), initial=0.0) <= rel * np.max(np.abs(ref_out), initial=0.0) + abs_


@pytest.mark.parametrize("thres,mode,compact", [(6.0, "any", False), (6.0, "row", False), (0.0, "any", False),
                                                (6.0, "row", True)])
def test_blockwise_reaches_the_definition(thres, mode, compact):
    wl = W.small_random(51, 3, 16, 700, 300, invalid_frac=0.1, q_sigma=2.0)
    q, kv = _f64(wl)
    idx = wl.indices.numpy()
    ref_out, ref_lse = O.sparse_mla_fwd(q, kv, idx, wl.sm_scale)
    out, lse, ev = E.blockwise(q.astype(np.float32), kv.astype(np.float32), idx, wl.sm_scale,
                               thres=thres, rescale=mode, compact=compact)
    assert _tol_ok(out, lse, ref_out, ref_lse)
    assert np.max(np.abs(lse - ref_lse)) < 1e-4
    assert ev.min() >= 1


def test_skip_scale_changes_rounding_only():
    """THRES=6 against THRES=0 (rescale at every block): equal up to float32/bf16 rounding."""
    wl = W.small_random(61, 2, 32, 1024, 512, q_sigma=2.0)
    q, kv = _f64(wl)
    idx = wl.indices.numpy()
    a = E.blockwise(q.astype(np.float32), kv.astype(np.float32), idx, wl.sm_scale, thres=6.0)
    b = E.blockwise(q.astype(np.float32), kv.astype(np.float32), idx, wl.sm_scale, thres=0.0)
    assert a[2].max() < b[2].min()  # skip-scale really skipped some rescales
    scale = np.abs(b[0]).max()
    assert np.max(np.abs(a[0] - b[0])) <= 1e-2 * scale
    assert np.max(np.abs(a[1] - b[1])) <= 1e-4


def test_blockwise_masked_and_empty_blocks():
    wl = W.small_random(71, 2, 8, 300, 256)
    q, kv = _f64(wl)
    idx = wl.indices.numpy().astype(np.int64).copy()
    idx[0, :128] = -1        # two leading fully masked blocks
    idx[1, :] = -1           # nothing valid at all
    ref_out, ref_lse = O.sparse_mla_fwd(q, kv, idx, wl.sm_scale)
    out, lse, _ = E.blockwise(q.astype(np.float32), kv.astype(np.float32), idx, wl.sm_scale)
    assert np.all(out[1] == 0) and np.all(np.isneginf(lse[1]))
    assert _tol_ok(out, lse, ref_out, ref_lse)


def test_a_planted_mistake_is_caught():
    """A dropped rope term in the logits (a plausible slip) breaks the dense pin."""
    wl = W.small_random(81, 1, 4, 64, 40)
    q, kv = _f64(wl)
    idx = wl.indices.numpy()
    q_bad = q.copy()
    q_bad[:, :, 512:] = 0.0
    out_bad, lse_bad = O.sparse_mla_fwd(q_bad, kv, idx, wl.sm_scale)
    ro, rl = _dense_torch(q[0], kv, idx[0], wl.sm_scale)
    assert not np.allclose(lse_bad[0], rl, rtol=1e-6)
