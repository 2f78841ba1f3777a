"""Python binding of the C ABI (include/dsa.h): argument marshalling only.

Each function takes torch CUDA tensors, checks dtypes/shapes/contiguity,
allocates missing outputs and the workspace with torch, and calls the C entry
point of the same name on the current (or given) stream.  Every step of the
computation runs in the library's CUDA kernels; there is no other code path.
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib

D_QK = 576
D_V = 512
FP8_ROW_BYTES = 656
KV_BF16 = 0
KV_FP8 = 1
KV_FP4 = 2
FP4_ROW_BYTES = 448


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream_handle(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def dsa_sparse_attn_fwd_workspace_size(s_q: int, h_q: int, topk: int, kv_format: int = KV_BF16) -> int:
    return int(_lib.load().dsa_sparse_attn_fwd_workspace_size(s_q, h_q, topk, kv_format))


def _check(q, kv, indices, kv_format):
    if not (q.is_cuda and kv.is_cuda and indices.is_cuda):
        raise ValueError("q, kv and indices must be CUDA tensors")
    _check_shapes(q, kv, indices, kv_format)


def _check_shapes(q, kv, indices, kv_format):
    if q.dtype != torch.bfloat16 or q.dim() != 3 or q.shape[2] != D_QK or not q.is_contiguous():
        raise ValueError("q must be a contiguous bf16 tensor [s_q, h_q, 576]")
    if kv_format == KV_BF16:
        if kv.dtype != torch.bfloat16 or kv.dim() != 2 or kv.shape[1] != D_QK or not kv.is_contiguous():
            raise ValueError("kv must be a contiguous bf16 tensor [s_kv, 576]")
    else:
        nb = FP8_ROW_BYTES if kv_format == KV_FP8 else FP4_ROW_BYTES
        if kv.dtype != torch.uint8 or kv.dim() != 2 or kv.shape[1] != nb or not kv.is_contiguous():
            raise ValueError(f"kv must be a contiguous uint8 tensor [s_kv, {nb}] of quantised rows")
    if indices.dtype != torch.int32 or indices.dim() != 2 or indices.shape[0] != q.shape[0] or not indices.is_contiguous():
        raise ValueError("indices must be a contiguous int32 tensor [s_q, topk]")


def _forward(fn_name, kv_format, q, kv, indices, sm_scale, out=None, lse=None, workspace=None, stream=None,
             check_status=False):
    _check(q, kv, indices, kv_format)
    lib = _lib.load()
    s_q, h_q, _ = q.shape
    s_kv = kv.shape[0]
    topk = indices.shape[1]
    if out is None:
        out = torch.empty((s_q, h_q, D_V), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((s_q, h_q), dtype=torch.float32, device=q.device)
    ws_bytes = int(lib.dsa_sparse_attn_fwd_workspace_size(s_q, h_q, topk, kv_format))
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=q.device)
    st = getattr(lib, fn_name)(_ptr(q), _ptr(kv), _ptr(indices), s_q, h_q, s_kv, topk, ctypes.c_float(sm_scale),
                               _ptr(out), _ptr(lse), _ptr(workspace), ctypes.c_size_t(workspace.numel()),
                               _stream_handle(stream))
    if st != 0:
        raise _lib.DsaError(st, fn_name)
    if check_status:
        dsa_read_device_status(workspace, stream)
    return out, lse


def dsa_sparse_attn_fwd(q, kv, indices, sm_scale, out=None, lse=None, workspace=None, stream=None,
                        check_status=False):
    """Sparse MLA forward with a bf16 KV cache.  Returns (out bf16 [s_q,h_q,512], lse f32 [s_q,h_q])."""
    return _forward("dsa_sparse_attn_fwd", KV_BF16, q, kv, indices, sm_scale, out, lse, workspace, stream,
                    check_status)


def dsa_sparse_attn_fwd_fp8kv(q, kv_fp8, indices, sm_scale, out=None, lse=None, workspace=None, stream=None,
                              check_status=False):
    """Sparse MLA forward with an FP8 KV cache of 656-byte rows."""
    return _forward("dsa_sparse_attn_fwd_fp8kv", KV_FP8, q, kv_fp8, indices, sm_scale, out, lse, workspace, stream,
                    check_status)


def dsa_sparse_attn_fwd_paged(q, kv_pool, indices, seq_of_token, block_table, page_size, sm_scale, kv_format=KV_BF16,
                              out=None, lse=None, workspace=None, stream=None, check_status=False):
    """Sparse MLA forward over a paged KV cache: indices [s_q, topk] are logical positions in each token's
    sequence (seq_of_token int32 [s_q]); block_table int32 [n_seq, max_pages] gives the physical page of each
    logical page of the pool kv_pool (page k = rows [k * page_size, (k + 1) * page_size))."""
    _check(q, kv_pool, indices, kv_format)
    for name, t in (("seq_of_token", seq_of_token), ("block_table", block_table)):
        if not t.is_cuda or t.dtype != torch.int32 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous int32 CUDA tensor")
    if seq_of_token.dim() != 1 or seq_of_token.shape[0] != q.shape[0] or block_table.dim() != 2:
        raise ValueError("seq_of_token must be [s_q] and block_table [n_seq, max_pages]")
    lib = _lib.load()
    s_q, h_q, _ = q.shape
    topk = indices.shape[1]
    n_seq, max_pages = block_table.shape
    if out is None:
        out = torch.empty((s_q, h_q, D_V), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((s_q, h_q), dtype=torch.float32, device=q.device)
    ws_bytes = int(lib.dsa_sparse_attn_fwd_workspace_size(s_q, h_q, topk, kv_format))
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=q.device)
    st = lib.dsa_sparse_attn_fwd_paged(kv_format, _ptr(q), _ptr(kv_pool), _ptr(indices), _ptr(seq_of_token),
                                       _ptr(block_table), s_q, h_q, kv_pool.shape[0], topk, n_seq, max_pages,
                                       page_size, ctypes.c_float(sm_scale), _ptr(out), _ptr(lse), _ptr(workspace),
                                       ctypes.c_size_t(workspace.numel()), _stream_handle(stream))
    if st != 0:
        raise _lib.DsaError(st, "dsa_sparse_attn_fwd_paged")
    if check_status:
        dsa_read_device_status(workspace, stream)
    return out, lse


def dsa_sparse_attn_fwd_fp4kv(q, kv_fp4, indices, sm_scale, out=None, lse=None, workspace=None, stream=None,
                              check_status=False):
    """Sparse MLA forward with an FP4 (e2m1) KV cache of 448-byte rows."""
    return _forward("dsa_sparse_attn_fwd_fp4kv", KV_FP4, q, kv_fp4, indices, sm_scale, out, lse, workspace, stream,
                    check_status)


def dsa_read_device_status(workspace, stream=None) -> int:
    """Synchronise the stream and raise if a kernel reported a device-side timeout."""
    st = int(_lib.load().dsa_read_device_status(_ptr(workspace), _stream_handle(stream)))
    if st != 0:
        raise _lib.DsaError(st, "device status")
    return st


def dsa_status_string(code: int) -> str:
    return _lib.load().dsa_status_string(code).decode()


def dsa_kernels_per_call() -> int:
    return int(_lib.load().dsa_kernels_per_call())


def dsa_set_timing_events(before=None, after=None) -> None:
    """Have later forward calls record two torch.cuda.Event objects around the attention kernel.

    Both events must already exist on the device (record them once first); pass
    no arguments to switch the hook off.
    """
    if before is None or after is None:
        _lib.load().dsa_set_timing_events(ctypes.c_void_p(0), ctypes.c_void_p(0))
        return
    _lib.load().dsa_set_timing_events(ctypes.c_void_p(before.cuda_event), ctypes.c_void_p(after.cuda_event))


def dsa_sparse_attn_fwd_noalloc(q, kv, indices, sm_scale, out, lse, stream=None):
    """The bf16 forward without a workspace, for callers that cannot allocate device memory.

    The library uses its own built-in scratch array instead (limits: s_q <= 8192,
    h_q <= 128).  `out` and `lse` must be given (nothing is allocated here).
    Calls that overlap on the GPU share that array and race; serialise them.
    """
    _check(q, kv, indices, KV_BF16)
    s_q, h_q, _ = q.shape
    st = _lib.load().dsa_sparse_attn_fwd_noalloc(_ptr(q), _ptr(kv), _ptr(indices), s_q, h_q, kv.shape[0],
                                                 indices.shape[1], ctypes.c_float(sm_scale), _ptr(out), _ptr(lse),
                                                 _stream_handle(stream))
    if st != 0:
        raise _lib.DsaError(st, "dsa_sparse_attn_fwd_noalloc")
    return out, lse


def dsa_sparse_attn_fwd_host_device_bytes(kv_format: int, s_q: int, h_q: int, s_kv: int, topk: int,
                                          chunk_tokens: int) -> int:
    return int(_lib.load().dsa_sparse_attn_fwd_host_device_bytes(kv_format, s_q, h_q, s_kv, topk, chunk_tokens))


def dsa_sparse_attn_fwd_host(q, kv, indices, sm_scale, kv_format=KV_BF16, out=None, lse=None, device_buffer=None,
                             chunk_tokens=256, device=None, stream=None):
    """The forward from host (CPU) tensors, token chunks pipelined through the GPU (upload, compute and
    download overlap).  Pinned tensors (``tensor.pin_memory()``) let the copies overlap; the call returns
    when ``out`` and ``lse`` (host tensors) hold the result.  ``device_buffer`` is a uint8 CUDA tensor of at
    least ``dsa_sparse_attn_fwd_host_device_bytes(...)`` bytes (allocated here when not given)."""
    for name, t in (("q", q), ("kv", kv), ("indices", indices)):
        if t.is_cuda:
            raise ValueError(f"{name} must be a host tensor")
    _check_shapes(q, kv, indices, kv_format)
    lib = _lib.load()
    s_q, h_q, _ = q.shape
    s_kv, topk = kv.shape[0], indices.shape[1]
    if out is None:
        out = torch.empty((s_q, h_q, D_V), dtype=torch.bfloat16, pin_memory=q.is_pinned())
    if lse is None:
        lse = torch.empty((s_q, h_q), dtype=torch.float32, pin_memory=q.is_pinned())
    if out.is_cuda or lse.is_cuda or out.dtype != torch.bfloat16 or lse.dtype != torch.float32 \
            or tuple(out.shape) != (s_q, h_q, D_V) or tuple(lse.shape) != (s_q, h_q) \
            or not out.is_contiguous() or not lse.is_contiguous():
        raise ValueError("out / lse must be contiguous host tensors bf16 [s_q, h_q, 512] / f32 [s_q, h_q]")
    need = int(lib.dsa_sparse_attn_fwd_host_device_bytes(kv_format, s_q, h_q, s_kv, topk, chunk_tokens))
    if device_buffer is None and s_q > 0:
        dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
        device_buffer = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    nbytes = device_buffer.numel() if device_buffer is not None else 0
    st = lib.dsa_sparse_attn_fwd_host(kv_format, _ptr(q), _ptr(kv), _ptr(indices), s_q, h_q, s_kv, topk,
                                      ctypes.c_float(sm_scale), _ptr(out), _ptr(lse), _ptr(device_buffer),
                                      ctypes.c_size_t(nbytes), chunk_tokens, _stream_handle(stream))
    if st != 0:
        raise _lib.DsaError(st, "dsa_sparse_attn_fwd_host")
    return out, lse


def dsa_out_proj(out, w_o, x=None, y=None, workspace=None, stream=None):
    """y = out . W_o + x: out bf16 [s_q, h_q, 512] (a forward's output), w_o bf16 [h_q * 512, d_model],
    x bf16 [s_q, d_model] or None.  Returns y bf16 [s_q, d_model]."""
    s_q, h_q = out.shape[0], out.shape[1]
    d_model = w_o.shape[1]
    _check_oproj(out, w_o, x, s_q, h_q, d_model)
    lib = _lib.load()
    if y is None:
        y = torch.empty((s_q, d_model), dtype=torch.bfloat16, device=out.device)
    if workspace is None:
        workspace = torch.empty(dsa_out_proj_workspace_size(), dtype=torch.uint8, device=out.device)
    st = lib.dsa_out_proj(_ptr(out), _ptr(w_o), _ptr(x), s_q, h_q, d_model, _ptr(y), _ptr(workspace),
                          ctypes.c_size_t(workspace.numel()), _stream_handle(stream))
    if st != 0:
        raise _lib.DsaError(st, "dsa_out_proj")
    return y


def _check_oproj(out, w_o, x, s_q, h_q, d_model):
    if out.dtype != torch.bfloat16 or out.dim() != 3 or out.shape[2] != D_V or not out.is_contiguous():
        raise ValueError("out must be a contiguous bf16 tensor [s_q, h_q, 512]")
    if w_o.dtype != torch.bfloat16 or w_o.dim() != 2 or w_o.shape[0] != h_q * D_V or not w_o.is_contiguous():
        raise ValueError("w_o must be a contiguous bf16 tensor [h_q * 512, d_model]")
    if x is not None and (x.dtype != torch.bfloat16 or tuple(x.shape) != (s_q, d_model) or not x.is_contiguous()):
        raise ValueError("x must be a contiguous bf16 tensor [s_q, d_model]")


def dsa_sparse_attn_fwd_oproj(q, kv, indices, sm_scale, w_o, x=None, kv_format=KV_BF16, out=None, lse=None, y=None,
                              workspace=None, stream=None, check_status=False):
    """The forward, then y = out . W_o + x on the same stream.  Returns (y, out, lse)."""
    _check(q, kv, indices, kv_format)
    lib = _lib.load()
    s_q, h_q, _ = q.shape
    topk = indices.shape[1]
    d_model = w_o.shape[1]
    if out is None:
        out = torch.empty((s_q, h_q, D_V), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((s_q, h_q), dtype=torch.float32, device=q.device)
    if y is None:
        y = torch.empty((s_q, d_model), dtype=torch.bfloat16, device=q.device)
    _check_oproj(out, w_o, x, s_q, h_q, d_model)
    if workspace is None:
        nb = int(lib.dsa_sparse_attn_fwd_oproj_workspace_size(s_q, h_q, topk, kv_format))
        workspace = torch.empty(max(nb, 256), dtype=torch.uint8, device=q.device)
    st = lib.dsa_sparse_attn_fwd_oproj(kv_format, _ptr(q), _ptr(kv), _ptr(indices), s_q, h_q, kv.shape[0], topk,
                                       ctypes.c_float(sm_scale), _ptr(w_o), _ptr(x), d_model, _ptr(out), _ptr(lse),
                                       _ptr(y), _ptr(workspace), ctypes.c_size_t(workspace.numel()),
                                       _stream_handle(stream))
    if st != 0:
        raise _lib.DsaError(st, "dsa_sparse_attn_fwd_oproj")
    if check_status:
        dsa_read_device_status(workspace, stream)
    return y, out, lse


def dsa_sparse_attn_fwd_oproj_workspace_size(s_q: int, h_q: int, topk: int, kv_format: int = KV_BF16) -> int:
    return int(_lib.load().dsa_sparse_attn_fwd_oproj_workspace_size(s_q, h_q, topk, kv_format))


def dsa_out_proj_workspace_size() -> int:
    return int(_lib.load().dsa_out_proj_workspace_size())
