"""The seeded input generators follow the recipes they state (structure only: no attention arithmetic).

Checked on reduced sizes of the same generators: value distributions (bf16 normal draws), index structure
(distinct, causal, per-sequence ranges, the -1 pattern, ragged counts and local windows), FP8/FP4 row
layouts, the paged pool and the projection weights' scale.
"""
import math

import numpy as np
import torch

from sparse_mla_attention_dsa_gb300 import workloads as W


def _distinct_rows(idx: np.ndarray) -> bool:
    return all(len(set(r[r >= 0].tolist())) == int((r >= 0).sum()) for r in idx)


def test_prefill_causal_structure():
    wl = W.prefill_causal(seed=2, s_q=64, h_q=8, s_kv=4160, topk=2048)
    idx = wl.indices.numpy()
    base = wl.s_kv - wl.s_q
    assert (idx == -1).sum(axis=1).tolist() == [102] * wl.s_q          # round(5 % of 2048) slots masked
    for t in range(wl.s_q):
        v = idx[t][idx[t] >= 0]
        assert v.size == 1946 and v.max() <= base + t and v.min() >= 0  # causal: up to the query's position
    assert _distinct_rows(idx)
    assert abs(float(wl.q.float().std()) - 1.0) < 0.02 and wl.q.dtype == torch.bfloat16
    assert math.isclose(wl.sm_scale, 1 / 24)


def test_decode_structure():
    wl = W.decode_bf16(seed=1, n_seq=4, h_q=8, s_kv_per_seq=4096, topk=2048)
    idx = wl.indices.numpy()
    for b in range(4):
        assert idx[b].min() >= b * 4096 and idx[b].max() < (b + 1) * 4096  # its own sequence's rows
    assert _distinct_rows(idx) and (idx >= 0).all()


def test_long_prefill_structure():
    wl = W.long_prefill(seed=4, s_q=48, h_q=8, s_kv=8192, topk=2048)
    idx = wl.indices.numpy()
    base = wl.s_kv - wl.s_q
    nv = (idx >= 0).sum(axis=1)
    assert nv.min() >= 256 and nv.max() <= 2048
    for t in range(wl.s_q):
        n = int(nv[t])
        assert (idx[t, n:] == -1).all()                                  # tail-padded
        v = idx[t, :n]
        assert v.max() <= base + t
        c = int(round(0.7 * n))
        lo = max(0, base + t + 1 - (-(-c // 512)) * 512)
        assert int((v >= lo).sum()) == min(c, base + t + 1 - lo)        # the local share sits in the windows
    assert _distinct_rows(idx)


def test_quantised_rows_layout():
    wl8 = W.small_random(1, 2, 4, 50, 8, kv_format="fp8")
    wl4 = W.small_random(1, 2, 4, 50, 8, kv_format="fp4")
    assert wl8.kv.dtype == torch.uint8 and tuple(wl8.kv.shape) == (50, 656)
    assert wl4.kv.dtype == torch.uint8 and tuple(wl4.kv.shape) == (50, 448)
    s8 = wl8.kv.numpy()[:, 512:528].copy().view(np.float32)
    s4 = wl4.kv.numpy()[:, 256:320].copy().view(np.float32)
    assert (s8 > 0).all() and (s4 > 0).all()                            # per-group scales are positive


def test_paged_pool_and_table():
    wl = W.small_paged(3, 10, 4, 3, 5, 16, 40, unmapped_frac=0.2)
    table = wl.meta["block_table"].numpy()
    mapped = table[table >= 0]
    assert len(set(mapped.tolist())) == mapped.size                     # no page shared by two sequences
    assert mapped.max() < wl.kv.shape[0] // wl.meta["page_size"]
    assert ((table < 0).sum(axis=1) == 1).all()                         # round(0.2 * 5) unmapped per sequence


def test_projection_weights_scale():
    w_o, x, o = W.oproj_inputs(5, 4, 8, 64)
    k = 8 * 512
    assert tuple(w_o.shape) == (k, 64) and tuple(x.shape) == (4, 64) and tuple(o.shape) == (4, 8, 512)
    assert abs(float(w_o.float().std()) * math.sqrt(k) - 1.0) < 0.05
