"""The sparse MLA forward by its definition, in float64 (test infrastructure only).

Follows "Ascend Sparse Attention Forward 算法与优化技术简析", section "数学建模":
for one query token with Q[h_q, d_qk], KV[s_kv, d_qk], indices[topk], sm_scale

    gathered_kv = KV.index_select(indices)          [topk, d_qk]
    P   = Q @ gathered_kv^T                         [h_q, topk]
    S   = softmax(P * sm_scale, dim=-1)             [h_q, topk]
    out = S @ gathered_kv[:, :d_v]                  [h_q, d_v]

plus lse = log(sum(exp(P * sm_scale))) per head (the page names lse as an
output in section "计算流程"; the natural log is used).

Readings where the pages are silent:
  * an index outside [0, s_kv) (the -1 marker included) is excluded exactly:
    it contributes to neither the normaliser nor the output;
  * a token with no valid index gives out = 0 and lse = -inf;
  * duplicate indices each count (index_select semantics).

The softmax is taken in full over the valid slots (no blocking, no online
update): m = max logit, Z = sum exp(logit - m), lse = m + ln Z,
out = sum exp(logit - lse) * row[:d_v].
"""
from __future__ import annotations

import numpy as np

from .formats import bf16_bits_to_f64, fp4_rows_to_f64, fp8_rows_to_f64

D_QK = 576
D_V = 512


def sparse_mla_fwd_token(q: np.ndarray, kv: np.ndarray, idx: np.ndarray, sm_scale: float, d_v: int = D_V):
    """One query token.  q [h_q, d_qk] f64, kv [s_kv, d_qk] f64, idx [topk] ints.

    Returns (out [h_q, d_v] f64, lse [h_q] f64).
    """
    s_kv = kv.shape[0]
    idx = np.asarray(idx, dtype=np.int64)
    valid = (idx >= 0) & (idx < s_kv)
    j = idx[valid]
    h_q = q.shape[0]
    if j.size == 0:
        return np.zeros((h_q, d_v)), np.full(h_q, -np.inf)
    g = kv[j]                                  # gathered_kv [n_valid, d_qk]
    logits = (q @ g.T) * sm_scale              # [h_q, n_valid]
    m = logits.max(axis=1, keepdims=True)
    z = np.exp(logits - m).sum(axis=1, keepdims=True)
    lse = m + np.log(z)                        # [h_q, 1]
    s = np.exp(logits - lse)                   # softmax weights
    out = s @ g[:, :d_v]
    return out, lse[:, 0]


def sparse_mla_fwd(q: np.ndarray, kv: np.ndarray, indices: np.ndarray, sm_scale: float,
                   tokens=None, d_v: int = D_V):
    """All (or the listed) query tokens.  q [s_q, h_q, d_qk] f64, kv [s_kv, d_qk] f64.

    Returns (out [n, h_q, d_v] f64, lse [n, h_q] f64) for the n selected tokens.
    """
    tokens = range(q.shape[0]) if tokens is None else list(tokens)
    outs, lses = [], []
    for t in tokens:
        o, l = sparse_mla_fwd_token(q[t], kv, indices[t], sm_scale, d_v)
        outs.append(o)
        lses.append(l)
    h_q = q.shape[1]
    if not outs:
        return np.zeros((0, h_q, d_v)), np.zeros((0, h_q))
    return np.stack(outs), np.stack(lses)


# --- helpers that turn stored inputs (raw bits) into float64 -----------------

def q_to_f64(q_bits: np.ndarray) -> np.ndarray:
    """bf16 query bits (uint16/int16 [s_q, h_q, 576]) -> float64."""
    return bf16_bits_to_f64(q_bits)


def kv_to_f64(kv_raw: np.ndarray, kv_format: str) -> np.ndarray:
    """KV cache bytes -> float64 [s_kv, 576] (bf16 bits, 656-byte FP8 rows or 448-byte FP4 rows)."""
    if kv_format == "bf16":
        return bf16_bits_to_f64(kv_raw)
    if kv_format == "fp8":
        return fp8_rows_to_f64(kv_raw)
    if kv_format == "fp4":
        return fp4_rows_to_f64(kv_raw)
    raise ValueError(kv_format)


def gathered_kv_f64(kv_raw: np.ndarray, kv_format: str, rows: np.ndarray) -> np.ndarray:
    """Dequantise only the listed rows (for large caches); returns [len(rows), 576]."""
    return kv_to_f64(kv_raw[rows], kv_format)


def sparse_mla_fwd_sampled(q_bits: np.ndarray, kv_raw: np.ndarray, kv_format: str, indices: np.ndarray,
                           sm_scale: float, tokens, d_v: int = D_V):
    """The definition on a sample of tokens of a large workload.

    Only the rows that the sampled tokens name are decoded; the index list is
    remapped onto that row subset, which leaves every gathered row unchanged.
    """
    tokens = list(tokens)
    s_kv = kv_raw.shape[0]
    h_q = q_bits.shape[1]
    outs = np.zeros((len(tokens), h_q, d_v))
    lses = np.zeros((len(tokens), h_q))
    for n, t in enumerate(tokens):
        idx = np.asarray(indices[t], dtype=np.int64)
        valid = (idx >= 0) & (idx < s_kv)
        rows, inv = np.unique(idx[valid], return_inverse=True)
        sub = gathered_kv_f64(kv_raw, kv_format, rows)
        local = np.full(idx.shape, -1, dtype=np.int64)
        local[valid] = inv
        o, l = sparse_mla_fwd_token(q_to_f64(q_bits[t]), sub, local, sm_scale, d_v)
        outs[n] = o
        lses[n] = l
    return outs, lses
