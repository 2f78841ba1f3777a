"""The pages' blockwise online-softmax algorithm, emulated on the CPU (test only).

Follows "Ascend Sparse Attention Forward 算法与优化技术简析", section "计算流程"
(steps 1 to 8) in its own notation, in float32:

  1. cut the topk indices into blocks of B_TOPK;
  2. keep running_max, running_max_for_softmax and running_sumexp [h_q]
     (initial -inf, -inf, 0) and out_accum [h_q, d_v], all float32;
  3. per block: gather the block's KV rows; P = Q @ gathered_kv^T; cur_max =
     row max; running_max = max(running_max, cur_max); if some row has
     running_max - running_max_for_softmax > RESCALE_THRES (6), multiply
     out_accum and running_sumexp by exp(running_max_for_softmax -
     running_max) and set running_max_for_softmax = running_max ("skip
     scale": otherwise nothing is rescaled); S = exp(P - running_max_for_
     softmax); out_accum += S.to(bf16) @ gathered_kv[:, :d_v];
     running_sumexp += S.sum(-1).

Readings where the section is silent (each is also listed in the design notes):
  * the max and exp act on the scaled logits P * sm_scale, so the threshold of
    6 is in natural-log units of scaled logits;
  * the end result is out = out_accum / running_sumexp and
    lse = running_max_for_softmax + ln(running_sumexp);
  * an index outside [0, s_kv) is masked: its S is exactly 0 and it never
    raises cur_max; while every slot so far was masked (running_max = -inf)
    nothing is rescaled;
  * running_sumexp accumulates the float32 S before the bf16 cast;
  * ``rescale="any"`` updates every row when some row triggers (the section's
    vector formulas); ``rescale="row"`` updates only the rows that trigger.
    Both are exact; they differ in rounding only;
  * ``compact=True`` first removes masked slots from the index list and then
    cuts blocks, which only regroups the same terms.
"""
from __future__ import annotations

import numpy as np

from .formats import round_to_bf16  # noqa: F401  (re-exported for tests)

D_V = 512


def blockwise_token(q32: np.ndarray, kv32: np.ndarray, idx: np.ndarray, sm_scale: float, b_topk: int = 64,
                    thres: float = 6.0, rescale: str = "any", compact: bool = False, d_v: int = D_V):
    """One token through the blockwise algorithm.

    q32 [h_q, d_qk] and kv32 [s_kv, d_qk] hold the bf16 input values as float32.
    Returns (out f32 [h_q, d_v], lse f32 [h_q], n_rescale_events).
    """
    s_kv = kv32.shape[0]
    h_q = q32.shape[0]
    idx = np.asarray(idx, dtype=np.int64)
    valid_all = (idx >= 0) & (idx < s_kv)
    if compact:
        idx = idx[valid_all]
        valid_all = np.ones(idx.shape, dtype=bool)
    running_max = np.full(h_q, -np.inf, dtype=np.float32)
    rmfs = np.full(h_q, -np.inf, dtype=np.float32)
    sumexp = np.zeros(h_q, dtype=np.float32)
    out_accum = np.zeros((h_q, d_v), dtype=np.float32)
    scale = np.float32(sm_scale)
    events = 0
    for k0 in range(0, idx.size, b_topk):
        blk = idx[k0:k0 + b_topk]
        valid = valid_all[k0:k0 + b_topk]
        g = np.zeros((blk.size, kv32.shape[1]), dtype=np.float32)
        g[valid] = kv32[blk[valid]]
        p = (q32 @ g.T).astype(np.float32) * scale
        p[:, ~valid] = -np.inf
        cur_max = p.max(axis=1)
        running_max = np.maximum(running_max, cur_max)
        with np.errstate(invalid="ignore"):
            trig = (running_max - rmfs) > np.float32(thres)
        if trig.any():
            events += 1
            rows = np.isfinite(running_max) if rescale == "any" else trig
            alpha = np.exp(rmfs[rows] - running_max[rows]).astype(np.float32)
            out_accum[rows] *= alpha[:, None]
            sumexp[rows] *= alpha
            rmfs[rows] = running_max[rows]
        with np.errstate(invalid="ignore"):
            s = np.exp(p - rmfs[:, None]).astype(np.float32)
        s[:, ~valid] = 0.0
        s[~np.isfinite(rmfs)] = 0.0
        out_accum += round_to_bf16(s) @ g[:, :d_v]
        sumexp += s.sum(axis=1, dtype=np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        out = np.where(sumexp[:, None] > 0, out_accum / sumexp[:, None], 0.0).astype(np.float32)
        lse = np.where(sumexp > 0, rmfs + np.log(sumexp), -np.inf).astype(np.float32)
    return out, lse, events


def blockwise(q32: np.ndarray, kv32: np.ndarray, indices: np.ndarray, sm_scale: float, tokens=None, **kw):
    """All (or the listed) tokens; returns (out [n,h_q,d_v], lse [n,h_q], events [n])."""
    tokens = range(q32.shape[0]) if tokens is None else list(tokens)
    res = [blockwise_token(q32[t], kv32, indices[t], sm_scale, **kw) for t in tokens]
    return (np.stack([r[0] for r in res]), np.stack([r[1] for r in res]), np.array([r[2] for r in res]))
