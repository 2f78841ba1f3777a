"""Pins of the paged-cache translation of the oracle (``oracle/paged.py``).

"Flash Attention Infer算子性能优化", section "优化Paged Attention路径": the KV of a
sequence is reached through a block table of physical pages.  The translation
is pinned by a hand-worked table (``tests/golden/paged_table.txt``), by the
closed form of an identity table, and end to end: a forward over a shuffled
page pool equals the forward over the same sequences stored contiguously.
"""
import os

import numpy as np

from oracle import dsa_oracle as O
from oracle import paged as PG

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden():
    tables, tokens, page_size, n_rows = {}, [], None, None
    with open(os.path.join(GOLDEN, "paged_table.txt"), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("page_size"):
                page_size = int(line.split()[1])
            elif line.startswith("n_rows"):
                n_rows = int(line.split()[1])
            elif line.startswith("table"):
                head, vals = line.split(":")
                tables[int(head.split()[1])] = [int(v) for v in vals.split()]
            elif line.startswith("token"):
                head, rest = line.split(":")
                seq = int(head.split()[3])
                pos, rows = rest.split("->")
                tokens.append((seq, [int(v) for v in pos.split()], [int(v) for v in rows.split()]))
    table = np.array([tables[k] for k in sorted(tables)], dtype=np.int64)
    return page_size, n_rows, table, tokens


def test_hand_worked_table():
    page_size, n_rows, table, tokens = _read_golden()
    idx = np.array([t[1] for t in tokens])
    seq = np.array([t[0] for t in tokens])
    want = np.array([t[2] for t in tokens])
    got = PG.logical_to_rows(idx, seq, table, page_size, n_rows)
    assert np.array_equal(got, want)


def test_identity_table_is_the_flat_layout():
    # sequence s stored contiguously at rows [s * L, (s + 1) * L), L = max_pages * page_size
    rng = np.random.default_rng(0)
    n_seq, max_pages, page = 3, 5, 8
    L = max_pages * page
    table = np.arange(n_seq * max_pages).reshape(n_seq, max_pages)
    seq = rng.integers(0, n_seq, size=7)
    idx = rng.integers(-1, L + 4, size=(7, 11))
    got = PG.logical_to_rows(idx, seq, table, page, n_seq * L)
    want = np.where((idx >= 0) & (idx < L), seq[:, None] * L + idx, -1)
    assert np.array_equal(got, want)


def test_rows_outside_the_pool_and_unknown_sequences_are_invalid():
    table = np.array([[0, 9]])
    got = PG.logical_to_rows(np.array([[0, 3, 4, 7]]), np.array([0]), table, 4, 38)  # page 9 = rows 36..39
    assert got.tolist() == [[0, 3, 36, -1]]
    assert PG.logical_to_rows(np.array([[0, 1]]), np.array([1]), table, 4, 64).tolist() == [[-1, -1]]
    assert PG.logical_to_rows(np.array([[0, 1]]), np.array([-1]), table, 4, 64).tolist() == [[-1, -1]]


def test_forward_over_a_shuffled_pool_equals_the_contiguous_forward():
    rng = np.random.default_rng(1)
    n_seq, max_pages, page, h_q = 3, 4, 8, 4
    L = max_pages * page
    flat = rng.standard_normal((n_seq * L, 576))           # sequence s at rows [s * L, (s + 1) * L)
    perm = rng.permutation(n_seq * max_pages)              # logical page (s, p) -> physical page perm[s * max_pages + p]
    pool = np.empty_like(flat)
    for s in range(n_seq):
        for p_ in range(max_pages):
            ph = perm[s * max_pages + p_]
            pool[ph * page:(ph + 1) * page] = flat[(s * max_pages + p_) * page:(s * max_pages + p_ + 1) * page]
    table = perm.reshape(n_seq, max_pages)
    s_q, topk = 5, 9
    seq = rng.integers(0, n_seq, size=s_q)
    idx = rng.integers(-1, L, size=(s_q, topk))
    q = rng.standard_normal((s_q, h_q, 576))
    out_p, lse_p = O.sparse_mla_fwd(q, pool, PG.logical_to_rows(idx, seq, table, page, len(pool)), 0.05)
    flat_idx = np.where(idx >= 0, seq[:, None] * L + idx, -1)
    out_f, lse_f = O.sparse_mla_fwd(q, flat, flat_idx, 0.05)
    assert np.allclose(out_p, out_f, rtol=0, atol=1e-12) and np.allclose(lse_p, lse_f, rtol=0, atol=1e-12)
