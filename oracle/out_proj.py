"""Output projection with residual after the attention, in float64 (test infrastructure only).

"FlashMLA算子Ascend 950移植：从tiling到访存优化全解读", section 3.4 (输出投影与残差合并): once a
token's attention output O is formed, it is multiplied by the output projection weight of the
linear layer that follows, and the block's input (the residual) is added:

    y = O · W_o + x

Readings (the page gives no shapes for the latent multi-head case):
  * O of one token is the head-major concatenation of the attention output out[t, h, :512],
    a vector of h_q * 512 values (out is bf16, as the forward writes it);
  * W_o is [h_q * 512, d_model] (bf16), x and y are [s_q, d_model];
  * the product and the sum are exact here (float64); no residual means x = 0.
"""
from __future__ import annotations

import numpy as np

from .formats import bf16_bits_to_f64


def out_proj(o_bits: np.ndarray, w_bits: np.ndarray, x_bits: np.ndarray | None = None) -> np.ndarray:
    """o_bits bf16 bits [s_q, h_q, d_v], w_bits bf16 bits [h_q * d_v, d_model], x_bits bf16 bits [s_q, d_model]
    or None  ->  y float64 [s_q, d_model]."""
    s_q = o_bits.shape[0]
    o = bf16_bits_to_f64(o_bits).reshape(s_q, -1)
    w = bf16_bits_to_f64(w_bits)
    assert o.shape[1] == w.shape[0], (o.shape, w.shape)
    y = o @ w
    if x_bits is not None:
        y = y + bf16_bits_to_f64(x_bits)
    return y


def out_proj_f64(o: np.ndarray, w_bits: np.ndarray, x_bits: np.ndarray | None = None) -> np.ndarray:
    """The same with a float64 attention output o [s_q, h_q, d_v] (the oracle's own forward result)."""
    s_q = o.shape[0]
    y = o.reshape(s_q, -1) @ bf16_bits_to_f64(w_bits)
    if x_bits is not None:
        y = y + bf16_bits_to_f64(x_bits)
    return y
