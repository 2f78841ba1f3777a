"""Pins of the output projection with residual (``oracle/out_proj.py``).

"FlashMLA算子Ascend 950移植：从tiling到访存优化全解读", section 3.4: y = O · W_o + x with O the
head-major concatenation of a token's attention output.  Pinned by a brute-force loop on tiny
inputs, by the closed form of a column-selection W_o (catches transposed operands and head
order), by exact additivity over heads and by the residual entering exactly once.
"""
import numpy as np

from oracle import out_proj as OP
from oracle.formats import round_to_bf16


def _bits(x: np.ndarray) -> np.ndarray:
    """float64 values already representable in bf16 -> their bf16 bit patterns."""
    return (np.asarray(x, dtype=np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def _rand_bf16(rng, shape, sigma=1.0):
    return round_to_bf16(rng.standard_normal(shape) * sigma)


def test_brute_force_tiny():
    rng = np.random.default_rng(0)
    s_q, h_q, d_v, d_model = 2, 2, 8, 3
    o = _rand_bf16(rng, (s_q, h_q, d_v))
    w = _rand_bf16(rng, (h_q * d_v, d_model))
    x = _rand_bf16(rng, (s_q, d_model))
    y = OP.out_proj(_bits(o), _bits(w), _bits(x))
    for t in range(s_q):
        for j in range(d_model):
            acc = float(x[t, j])
            for h in range(h_q):
                for d in range(d_v):
                    acc += float(o[t, h, d]) * float(w[h * d_v + d, j])
            assert abs(y[t, j] - acc) <= 1e-12 * max(1.0, abs(acc))


def test_column_selection_closed_form():
    # W_o[k, j] = 1 iff k == sel[j]: y[:, j] = O_cat[:, sel[j]] + x[:, j] exactly; sel crosses heads and
    # is not symmetric, so a transposed W_o or a head-minor concatenation fails it
    rng = np.random.default_rng(1)
    s_q, h_q, d_v, d_model = 5, 3, 512, 7
    o = _rand_bf16(rng, (s_q, h_q, d_v))
    sel = np.array([1500, 0, 513, 1024, 511, 1535, 7])
    w = np.zeros((h_q * d_v, d_model))
    w[sel, np.arange(d_model)] = 1.0
    x = _rand_bf16(rng, (s_q, d_model))
    y = OP.out_proj(_bits(o), _bits(w), _bits(x))
    heads, cols = sel // d_v, sel % d_v
    expect = o[:, heads, cols] + x
    assert np.array_equal(y, expect)


def test_additive_over_heads_and_residual_once():
    rng = np.random.default_rng(2)
    s_q, h_q, d_v, d_model = 4, 4, 512, 16
    o = _rand_bf16(rng, (s_q, h_q, d_v))
    w = _rand_bf16(rng, (h_q * d_v, d_model), sigma=0.05)
    x = _rand_bf16(rng, (s_q, d_model))
    full = OP.out_proj(_bits(o), _bits(w))
    parts = np.zeros_like(full)
    for h in range(h_q):
        oh = np.zeros_like(o)
        oh[:, h] = o[:, h]
        parts += OP.out_proj(_bits(oh), _bits(w))
    assert np.allclose(full, parts, rtol=0, atol=1e-12)
    with_x = OP.out_proj(_bits(o), _bits(w), _bits(x))
    assert np.allclose(with_x - full, x, rtol=0, atol=1e-12)
    assert np.array_equal(OP.out_proj_f64(o, _bits(w), _bits(x)), with_x)
