"""GPU parity: the CUDA library (called through its C ABI) against the float64 oracle.

Small cases compare every output element; the full-size workloads compare a
sample of tokens that the oracle computes one by one.  Cases span several
index blocks of 128, ragged tails (topk % 128 != 0), -1 and out-of-range slots,
fully masked tokens, duplicates, h_q < 128, and enough tokens that the work
sequence is cut across CTA pairs (exercising the merge of split tokens).
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
        out, lse = P.run_gpu(wl)
    tokens = list(range(wl.s_q)) if tokens is None else list(tokens)
    ref_out, ref_lse = P.oracle(wl, tokens)
    ok, rep = P.compare(out[tokens], lse[tokens], ref_out, ref_lse, wl.kv_format)
    assert ok, rep
    return rep


def test_tiny_workload():
    _check(W.tiny())


@pytest.mark.parametrize("s_q,h_q,s_kv,topk,bad", [
    (3, 128, 700, 64, 0.0),      # exactly one block
    (3, 128, 700, 65, 0.0),      # one full block + a 1-row tail
    (5, 128, 3000, 200, 0.1),    # ragged tail and -1 slots
    (4, 64, 5000, 2048, 0.05),   # many blocks, h_q = 64
    (6, 16, 300, 127, 0.3),      # h_q = 16, heavy masking
    (2, 100, 900, 333, 0.0),     # h_q not a power of two
    (2, 1, 50, 1, 0.0),          # a single index, a single head
])
def test_small_shapes(s_q, h_q, s_kv, topk, bad):
    _check(W.small_random(s_q * 1000 + topk, s_q, h_q, s_kv, topk, invalid_frac=bad))


def test_masked_blocks_and_empty_tokens():
    wl = W.small_random(7, 4, 128, 2000, 300)
    idx = wl.indices.clone()
    idx[0, :] = -1                 # no valid slot: out = 0, lse = -inf
    idx[1, :200] = -1              # leading masked slots (three blocks' worth)
    idx[2, ::2] = 2000             # out of range counts as masked
    idx[3, 100:] = idx[3, :1]      # duplicates count with multiplicity
    wl.indices = idx
    rep = _check(wl)
    out, lse = P.run_gpu(wl)
    assert torch.all(out[0] == 0) and torch.all(torch.isneginf(lse[0]))


def test_no_kv_rows():
    wl = W.small_random(9, 3, 16, 10, 8)
    wl.kv = wl.kv[:0]
    out, lse = P.run_gpu(wl)
    assert torch.all(out == 0) and torch.all(torch.isneginf(lse))


def test_scheduler_splits_tokens_across_pairs():
    # 300 tokens x 4 blocks: range boundaries cut many tokens; all must merge exactly
    _check(W.small_random(11, 300, 128, 4096, 256, invalid_frac=0.02), tokens=range(0, 300, 7))


def test_one_token_spread_over_every_pair():
    # 16 blocks < number of CTA pairs: one token cut into many pieces, some pairs idle
    _check(W.small_random(12, 1, 128, 8192, 2048, q_sigma=2.0))


def test_one_token_cut_into_more_pieces_than_a_warp_has_lanes():
    # 100 blocks over every CTA pair: the merge sees one piece per pair (more than 32 and more than 64)
    _check(W.small_random(14, 1, 128, 16384, 12800, q_sigma=2.0))


def test_repeatable_and_no_stray_writes():
    wl = W.small_random(13, 9, 128, 1500, 190, invalid_frac=0.1)
    from sparse_mla_attention_dsa_gb300 import api
    q, kv, idx = wl.q.cuda(), wl.kv.cuda(), wl.indices.cuda()
    pad = 4096
    obuf = torch.full((wl.s_q * wl.h_q * 512 + 2 * pad,), 12345, dtype=torch.int16, device="cuda")
    lbuf = torch.full((wl.s_q * wl.h_q + 2 * pad,), -7.0, dtype=torch.float32, device="cuda")
    out = obuf[pad:pad + wl.s_q * wl.h_q * 512].view(torch.bfloat16).view(wl.s_q, wl.h_q, 512)
    lse = lbuf[pad:pad + wl.s_q * wl.h_q].view(wl.s_q, wl.h_q)
    api.dsa_sparse_attn_fwd(q, kv, idx, wl.sm_scale, out=out, lse=lse, check_status=True)
    o1, l1 = out.clone(), lse.clone()
    api.dsa_sparse_attn_fwd(q, kv, idx, wl.sm_scale, out=out, lse=lse, check_status=True)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), out.view(torch.int16)) and torch.equal(l1, lse)  # deterministic
    assert torch.all(obuf[:pad] == 12345) and torch.all(obuf[-pad:] == 12345)
    assert torch.all(lbuf[:pad] == -7.0) and torch.all(lbuf[-pad:] == -7.0)
    _check(wl, out=out, lse=lse)


def test_rescale_fires_with_wide_logits():
    # sigma = 4 queries: logits spread widely, the skip-scale rescale fires mid-token
    _check(W.small_random(14, 3, 128, 4000, 1024, q_sigma=4.0))


# ---------------------------------------------------------------- FP8-e4m3 KV cache (656-byte rows)

@pytest.mark.parametrize("s_q,h_q,s_kv,topk,bad", [
    (3, 128, 700, 128, 0.0),     # exactly one block
    (3, 128, 900, 129, 0.0),     # one block + a 1-row tail
    (5, 128, 3000, 300, 0.1),    # ragged tail and -1 slots
    (4, 64, 5000, 2048, 0.05),   # many blocks, h_q = 64
    (6, 16, 300, 127, 0.3),      # h_q = 16, heavy masking
])
def test_fp8_small_shapes(s_q, h_q, s_kv, topk, bad):
    _check(W.small_random(s_q * 1000 + topk + 7, s_q, h_q, s_kv, topk, kv_format="fp8", invalid_frac=bad, q_sigma=2.0))


def test_fp8_masked_tokens_and_split_work():
    wl = W.small_random(17, 200, 128, 6000, 512, kv_format="fp8", invalid_frac=0.05, q_sigma=2.0)
    idx = wl.indices.clone()
    idx[3, :] = -1
    idx[5, 100:] = -1
    wl.indices = idx
    _check(wl, tokens=list(range(0, 200, 9)) + [3, 5])


def test_fp8_tiny_decode_shape():
    _check(W.decode_fp8(n_seq=4, s_kv_per_seq=4096, topk=2048))


# ---------------------------------------------------------------- full-size workloads (sampled tokens)

@pytest.mark.slow
def test_prefill_causal_full_size_sampled():
    wl = W.prefill_causal()
    out, lse = P.run_gpu(wl)
    rng = np.random.default_rng(0)
    tokens = sorted(set(rng.choice(wl.s_q, 24, replace=False).tolist()) | {0, wl.s_q - 1})
    _check(wl, tokens=tokens, out=out, lse=lse)


@pytest.mark.slow
def test_decode_bf16_full_size_sampled():
    wl = W.decode_bf16()
    out, lse = P.run_gpu(wl)
    _check(wl, tokens=[0, 1, 17, 40, 63], out=out, lse=lse)


@pytest.mark.slow
def test_long_prefill_full_size_sampled():
    wl = W.long_prefill()
    out, lse = P.run_gpu(wl)
    rng = np.random.default_rng(1)
    tokens = sorted(set(rng.choice(wl.s_q, 24, replace=False).tolist()) | {0, wl.s_q - 1})
    _check(wl, tokens=tokens, out=out, lse=lse)


@pytest.mark.slow
def test_decode_fp8_full_size_sampled():
    wl = W.decode_fp8()
    out, lse = P.run_gpu(wl)
    _check(wl, tokens=[0, 1, 50, 99, 127], out=out, lse=lse)


# ---------------------------------------------------------------- FP4 (e2m1) KV cache

@pytest.mark.parametrize("s_q,h_q,s_kv,topk,bad", [
    (4, 128, 600, 300, 0.0),
    (9, 64, 2000, 257, 0.1),
    (3, 16, 300, 129, 0.0),
])
def test_fp4_small_shapes(s_q, h_q, s_kv, topk, bad):
    _check(W.small_random(51 + s_q, s_q, h_q, s_kv, topk, kv_format="fp4", invalid_frac=bad, q_sigma=2.0))


def test_fp4_masked_tokens_and_split_work():
    wl = W.small_random(55, 200, 128, 4096, 512, kv_format="fp4", invalid_frac=0.05, q_sigma=2.0)
    wl.indices[3] = -1  # a token with no valid slot
    _check(wl, tokens=list(range(0, 200, 9)) + [3])


@pytest.mark.slow
def test_decode_fp4_full_size_sampled():
    wl = W.decode_fp4()
    out, lse = P.run_gpu(wl)
    _check(wl, tokens=[0, 1, 50, 99, 127], out=out, lse=lse)


# ---------------------------------------------------------------- whole tokens taken from a shared counter
# With at least 8 tokens per SM pair the pairs take whole tokens one by one instead of static shares
# (76 pairs on a GB300: from 608 tokens on).

@pytest.mark.parametrize("kv_format", ["bf16", "fp8"])
def test_dynamic_token_scheduling(kv_format):
    wl = W.small_random(71, 700, 16, 3000, 300, kv_format=kv_format, invalid_frac=0.05,
                        q_sigma=2.0 if kv_format != "bf16" else 1.0)
    wl.indices[5] = -1      # a token with no valid slot
    wl.indices[6, 1:] = -1  # a token with one valid slot
    _check(wl, tokens=list(range(0, 700, 23)) + [5, 6, 699])


def test_dynamic_scheduling_is_repeatable_and_complete():
    from sparse_mla_attention_dsa_gb300 import api
    wl = W.small_random(72, 1000, 16, 2000, 130)
    q, kv, idx = wl.q.cuda(), wl.kv.cuda(), wl.indices.cuda()
    out = torch.full((wl.s_q, wl.h_q, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((wl.s_q, wl.h_q), float("nan"), device="cuda")
    api.dsa_sparse_attn_fwd(q, kv, idx, wl.sm_scale, out=out, lse=lse, check_status=True)
    o1, l1 = out.clone(), lse.clone()
    assert not torch.isnan(o1.float()).any() and not torch.isnan(l1).any()  # every token written
    api.dsa_sparse_attn_fwd(q, kv, idx, wl.sm_scale, out=out, lse=lse, check_status=True)
    torch.cuda.synchronize()
    # a token's result does not depend on which pair took it
    assert torch.equal(o1.view(torch.int16), out.view(torch.int16)) and torch.equal(l1, lse)
    _check(wl, tokens=range(0, 1000, 37), out=o1, lse=l1)
