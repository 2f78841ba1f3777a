"""GPU parity of the host-buffer entry point (token chunks pipelined through the GPU) against the oracle.

The chunks are separate forward calls, so the split of tokens across CTA pairs differs from one call over
all tokens: results are held to the oracle's tolerances, not to bit equality with the device entry point.
Cases cover a ragged last chunk, one-token chunks, a chunk larger than s_q, every KV format, pageable and
page-locked host memory, a device buffer that is too small, and an empty KV.
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


def _fmt(wl):
    from sparse_mla_attention_dsa_gb300 import api
    return {"bf16": api.KV_BF16, "fp8": api.KV_FP8, "fp4": api.KV_FP4}[wl.kv_format]


def _run_host(wl, chunk, pinned=True):
    from sparse_mla_attention_dsa_gb300 import api
    q, kv, idx = (t.pin_memory() if pinned else t.contiguous() for t in (wl.q, wl.kv, wl.indices))
    out, lse = api.dsa_sparse_attn_fwd_host(q, kv, idx, wl.sm_scale, kv_format=_fmt(wl), chunk_tokens=chunk)
    assert not out.is_cuda and not lse.is_cuda
    return out, lse


def _check(wl, out, lse, tokens=None):
    tokens = list(range(wl.s_q)) if tokens is None else list(tokens)
    ref_out, ref_lse = P.oracle(wl, tokens)
    ok, rep = P.compare(out[tokens], lse[tokens], ref_out, ref_lse, wl.kv_format)
    assert ok, rep


@pytest.mark.parametrize("chunk", [1, 8, 37, 64])
def test_bf16_chunks(chunk):
    # 37 tokens: chunks of 8 leave a ragged 5-token tail; 37 and 64 are a single chunk
    wl = W.small_random(101, 37, 128, 3000, 300, invalid_frac=0.05)
    out, lse = _run_host(wl, chunk)
    _check(wl, out, lse)


@pytest.mark.parametrize("kv_format", ["fp8", "fp4"])
def test_quantised_kv(kv_format):
    wl = W.small_random(102, 29, 64, 2000, 257, kv_format=kv_format, invalid_frac=0.05, q_sigma=2.0)
    out, lse = _run_host(wl, 6)
    _check(wl, out, lse)


def test_pageable_host_memory():
    wl = W.small_random(103, 20, 32, 900, 129)
    out, lse = _run_host(wl, 7, pinned=False)
    _check(wl, out, lse)


def test_agrees_with_device_entry_point():
    wl = W.small_random(104, 300, 128, 4096, 256, invalid_frac=0.02)
    out_h, lse_h = _run_host(wl, 64)
    out_d, lse_d = P.run_gpu(wl)
    assert torch.allclose(lse_h, lse_d.cpu(), atol=1e-4, rtol=0)
    assert torch.allclose(out_h.float(), out_d.float().cpu(), atol=2e-2, rtol=2e-2)
    _check(wl, out_h, lse_h, tokens=range(0, 300, 11))


def test_masked_tokens_and_empty_kv():
    wl = W.small_random(105, 9, 16, 500, 64)
    wl.indices[2] = -1
    out, lse = _run_host(wl, 4)
    _check(wl, out, lse)
    assert torch.all(out[2] == 0) and torch.all(torch.isneginf(lse[2]))
    wl.kv = wl.kv[:0]
    out, lse = _run_host(wl, 4)
    assert torch.all(out == 0) and torch.all(torch.isneginf(lse))


def test_device_buffer_too_small_is_refused_before_any_copy():
    from sparse_mla_attention_dsa_gb300 import _lib, api
    wl = W.small_random(106, 8, 16, 300, 32)
    need = api.dsa_sparse_attn_fwd_host_device_bytes(api.KV_BF16, 8, 16, 300, 32, 4)
    assert need > 0
    buf = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    out = torch.full((8, 16, 512), 7.0, dtype=torch.bfloat16)
    lse = torch.full((8, 16), 7.0)
    with pytest.raises(_lib.DsaError) as e:
        api.dsa_sparse_attn_fwd_host(wl.q, wl.kv, wl.indices, wl.sm_scale, out=out, lse=lse, device_buffer=buf,
                                     chunk_tokens=4)
    assert e.value.code == 6
    assert torch.all(out == 7.0) and torch.all(lse == 7.0)


@pytest.mark.slow
def test_prefill_causal_full_size_sampled():
    wl = W.prefill_causal()
    out, lse = _run_host(wl, 256)
    rng = np.random.default_rng(3)
    tokens = sorted(set(rng.choice(wl.s_q, 16, replace=False).tolist()) | {0, 255, 256, wl.s_q - 1})
    _check(wl, out, lse, tokens)
