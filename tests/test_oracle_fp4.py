"""Pins of the oracle's FP4 decoders (``oracle/formats.py``).

e2m1 against the format's own value table (OCP FP4: sign, two exponent bits
with bias 1, one mantissa bit), and the 448-byte FP4 row (this library's
reading of the FP4 cache of "Ascend Sparse Attention Forward 算法与优化技术简析",
section "能不能用 1C1V") on a hand-built row whose every byte is chosen.
"""
import numpy as np
import torch

from oracle import dsa_oracle as O
from oracle import formats as F

# the sixteen e2m1 values, written out from the format's definition
E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]


def test_e2m1_decoder_matches_the_value_table():
    got = F.e2m1_to_f64(np.arange(16))
    assert got.tolist() == E2M1
    assert np.array_equal(np.signbit(got), np.signbit(np.array(E2M1)))


def _row(codes_by_channel: dict, scales: list, rope_value: float) -> np.ndarray:
    row = np.zeros(448, dtype=np.uint8)
    for ch, code in codes_by_channel.items():
        row[ch // 2] |= np.uint8(code << (4 * (ch & 1)))  # low nibble = even channel
    row[256:320] = np.array(scales, dtype=np.float32).view(np.uint8)
    row[320:448] = np.full(64, rope_value, dtype=np.float32).astype(np.float32).view(np.uint32).__rshift__(16) \
        .astype(np.uint16).view(np.uint8)
    return row


def test_fp4_row_nibble_order_scale_groups_and_rope():
    scales = [0.5, 2.0] + [1.0] * 14
    row = _row({0: 2, 1: 7, 2: 8, 3: 15, 32: 3, 511: 9}, scales, 1.0)
    got = F.fp4_rows_to_f64(row[None, :])[0]
    want = np.zeros(576)
    want[0], want[1], want[2], want[3] = 0.5 * 1.0, 0.5 * 6.0, -0.0, 0.5 * -6.0  # group 0: scale 0.5
    want[32] = 2.0 * 1.5                                                         # group 1: scale 2
    want[511] = 1.0 * -0.5                                                       # group 15
    want[512:] = 1.0                                                             # rope
    assert np.array_equal(got, want)
    assert np.signbit(got[2])


def test_fp4_product_is_rounded_to_bf16():
    # 1.5 * float32(0.1) is not a bf16 value; the dequantised channel is its bf16 (round to nearest even)
    row = _row({5: 3}, [0.1] + [1.0] * 15, 0.0)
    got = F.fp4_rows_to_f64(row[None, :])[0, 5]
    want = torch.tensor(np.float32(1.5) * np.float32(0.1), dtype=torch.float32).to(torch.bfloat16).double().item()
    assert got == want and got != np.float32(1.5) * np.float32(0.1)


def test_kv_dispatch_knows_fp4():
    row = _row({0: 4}, [1.0] * 16, 2.0)
    assert np.array_equal(O.kv_to_f64(row[None, :], "fp4"), F.fp4_rows_to_f64(row[None, :]))


def test_fp4_definition_uses_dequantised_rows():
    # the FP4 forward through the oracle equals a dense brute force over rows dequantised by a second route:
    # the e2m1 value table above, scales repeated over their 32-channel groups, torch's bf16 rounding
    from sparse_mla_attention_dsa_gb300 import workloads as W
    from tests.test_oracle import _bits, _dense_torch
    wl = W.small_random(43, 3, 16, 200, 70, kv_format="fp4", q_sigma=2.0)
    rows = wl.kv.numpy()
    q = O.q_to_f64(_bits(wl.q))
    idx = wl.indices.numpy()
    out, lse = O.sparse_mla_fwd(q, O.kv_to_f64(rows, "fp4"), idx, wl.sm_scale)
    table = np.array(E2M1)
    codes = np.stack([rows[:, :256] & 0xF, rows[:, :256] >> 4], axis=2).reshape(rows.shape[0], 512)
    scales = rows[:, 256:320].copy().view(np.float32).astype(np.float64)
    lat32 = (table[codes].astype(np.float32) * np.repeat(scales, 32, axis=1).astype(np.float32)).astype(np.float32)
    lat = torch.from_numpy(lat32).to(torch.bfloat16).double().numpy()
    rope = torch.from_numpy(rows[:, 320:].copy()).view(torch.bfloat16).double().numpy()
    kv_t = np.concatenate([lat, rope], axis=1)
    for t in range(3):
        ro, rl = _dense_torch(q[t], kv_t, idx[t], wl.sm_scale)
        assert np.allclose(out[t], ro, rtol=1e-11, atol=1e-12) and np.allclose(lse[t], rl, rtol=1e-12)
