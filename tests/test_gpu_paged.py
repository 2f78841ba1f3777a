"""GPU parity of the paged-cache forward (``dsa_sparse_attn_fwd_paged``) against the oracle.

The oracle turns logical positions into pool rows with its own translation
(``oracle/paged.py``) and then applies the definition; the GPU resolves them in
its index-loading step.  Cases cover several pages per block and blocks per
page, a page size that is not a power of two, unmapped pages, -1 slots,
positions past the block table, both KV formats, tokens cut across CTA pairs,
and the full-size decode shape with its pages scattered over the pool.
"""
import numpy as np
import pytest
import torch

from sparse_mla_attention_dsa_gb300 import workloads as W

from . import _parity as P

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_mla_attention_dsa_gb300 import build
    build.build()


def _check(wl, tokens=None, out=None, lse=None):
    if out is None:
        out, lse = P.run_gpu_paged(wl)
    tokens = list(range(wl.s_q)) if tokens is None else list(tokens)
    ref_out, ref_lse = P.oracle_paged(wl, tokens)
    ok, rep = P.compare(out[tokens], lse[tokens], ref_out, ref_lse, wl.kv_format)
    assert ok, rep
    return rep


@pytest.mark.parametrize("s_q,h_q,n_seq,max_pages,page_size,topk,unmapped,bad,past", [
    (7, 128, 3, 12, 64, 300, 0.0, 0.0, 0),     # plain: several blocks, ragged tail
    (9, 64, 4, 40, 16, 257, 0.25, 0.05, 3),    # small pages, unmapped pages, -1 slots, positions past the table
    (5, 16, 2, 9, 48, 190, 0.1, 0.1, 1),       # page size not a power of two
    (3, 128, 1, 3, 256, 640, 0.0, 0.0, 0),     # one sequence, pages larger than a block
])
def test_paged_bf16(s_q, h_q, n_seq, max_pages, page_size, topk, unmapped, bad, past):
    _check(W.small_paged(31 + s_q, s_q, h_q, n_seq, max_pages, page_size, topk, unmapped_frac=unmapped,
                         invalid_frac=bad, past_end=past))


def test_paged_fp8():
    _check(W.small_paged(41, 6, 128, 3, 20, 32, 300, kv_format="fp8", unmapped_frac=0.1, invalid_frac=0.05,
                         past_end=2))


def test_paged_tokens_split_across_pairs():
    # 300 tokens x 3 blocks over 5 sequences: range boundaries cut many tokens
    wl = W.small_paged(42, 300, 64, 5, 24, 32, 384, unmapped_frac=0.05)
    _check(wl, tokens=range(0, 300, 7))


def test_identity_table_gives_the_flat_result_exactly():
    # an identity block table over one sequence: the same rows in the same order as the flat call
    from sparse_mla_attention_dsa_gb300 import api
    wl = W.small_random(43, 11, 128, 2048, 300, invalid_frac=0.05)
    q, kv, idx = wl.q.cuda(), wl.kv.cuda(), wl.indices.cuda()
    seq = torch.zeros(wl.s_q, dtype=torch.int32, device="cuda")
    table = torch.arange(2048 // 64, dtype=torch.int32, device="cuda").view(1, -1)
    out_p, lse_p = api.dsa_sparse_attn_fwd_paged(q, kv, idx, seq, table, 64, wl.sm_scale, check_status=True)
    out_f, lse_f = api.dsa_sparse_attn_fwd(q, kv, idx, wl.sm_scale, check_status=True)
    torch.cuda.synchronize()
    assert torch.equal(out_p, out_f) and torch.equal(lse_p, lse_f)


@pytest.mark.slow
def test_decode_paged_full_size_sampled():
    wl = W.decode_paged()
    out, lse = P.run_gpu_paged(wl)
    _check(wl, tokens=[0, 1, 30, 63], out=out, lse=lse)


def test_paged_dynamic_token_scheduling():
    # 640 tokens: pairs take whole tokens from the shared counter
    wl = W.small_paged(81, 640, 16, 8, 12, 32, 200, unmapped_frac=0.1, invalid_frac=0.05)
    out, lse = P.run_gpu_paged(wl)
    tokens = list(range(0, 640, 29))
    ref_out, ref_lse = P.oracle_paged(wl, tokens)
    ok, rep = P.compare(out[tokens], lse[tokens], ref_out, ref_lse, wl.kv_format)
    assert ok, rep
