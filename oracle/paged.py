"""Paged KV cache: logical positions of a sequence -> rows of the page pool.

TEST INFRASTRUCTURE ONLY (see the package header).

"Flash Attention Infer算子性能优化", section "优化Paged Attention路径": with a
paged cache, a sequence's KV lives in fixed-size pages of a shared pool and is
reached through a block table that lists, per sequence, the physical page of
each logical page (the sequence length is rounded up to whole pages).  The
forward itself is unchanged: once every index is turned into a pool row, the
definition in ``dsa_oracle`` applies as is.

Readings (the page gives no formulas):
  * index v of a token of sequence s is a logical position in that sequence;
    its logical page is v // page_size, its offset v % page_size;
  * the pool row is block_table[s, v // page_size] * page_size + v % page_size;
  * v is invalid (contributes nothing, like -1 in the flat layout) when v < 0,
    v // page_size >= max_pages, the table entry is negative (page not
    mapped), the sequence id is outside [0, n_seq), or the row is outside the
    pool.
"""
from __future__ import annotations

import numpy as np


def logical_to_rows(indices: np.ndarray, seq_of_token: np.ndarray, block_table: np.ndarray, page_size: int,
                    n_rows: int) -> np.ndarray:
    """indices int [s_q, topk] (logical positions), seq_of_token int [s_q], block_table int [n_seq, max_pages]
    -> int64 [s_q, topk] pool rows, -1 where the position does not resolve to a row of the pool."""
    indices = np.asarray(indices, dtype=np.int64)
    seq = np.asarray(seq_of_token, dtype=np.int64)
    table = np.asarray(block_table, dtype=np.int64)
    n_seq, max_pages = table.shape
    out = np.full(indices.shape, -1, dtype=np.int64)
    for t in range(indices.shape[0]):
        s = int(seq[t])
        if s < 0 or s >= n_seq:
            continue
        for j in range(indices.shape[1]):
            v = int(indices[t, j])
            if v < 0:
                continue
            page, offset = divmod(v, page_size)
            if page >= max_pages:
                continue
            phys = int(table[s, page])
            if phys < 0:
                continue
            row = phys * page_size + offset
            if row < n_rows:
                out[t, j] = row
    return out
