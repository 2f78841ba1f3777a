"""ctypes loader for the in-tree CUDA library (argument types of every C entry point)."""
from __future__ import annotations

import ctypes
import os

from .build import LIB_PATH

# Every symbol include/dsa.h declares, with (restype, argtypes).
_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_S = ctypes.c_size_t
SIGNATURES = {
    "dsa_sparse_attn_fwd_workspace_size": (_S, [_I, _I, _I, _I]),
    "dsa_sparse_attn_fwd": (_I, [_P, _P, _P, _I, _I, _I, _I, _F, _P, _P, _P, _S, _P]),
    "dsa_sparse_attn_fwd_fp8kv": (_I, [_P, _P, _P, _I, _I, _I, _I, _F, _P, _P, _P, _S, _P]),
    "dsa_sparse_attn_fwd_fp4kv": (_I, [_P, _P, _P, _I, _I, _I, _I, _F, _P, _P, _P, _S, _P]),
    "dsa_read_device_status": (_I, [_P, _P]),
    "dsa_status_string": (ctypes.c_char_p, [_I]),
    "dsa_kernels_per_call": (_I, []),
    "dsa_set_timing_events": (None, [_P, _P]),
    "dsa_sparse_attn_fwd_noalloc": (_I, [_P, _P, _P, _I, _I, _I, _I, _F, _P, _P, _P]),
    "dsa_sparse_attn_fwd_paged": (_I, [_I, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P, _P, _P, _S, _P]),
    "dsa_sparse_attn_fwd_host_device_bytes": (_S, [_I, _I, _I, _I, _I, _I]),
    "dsa_sparse_attn_fwd_host": (_I, [_I, _P, _P, _P, _I, _I, _I, _I, _F, _P, _P, _P, _S, _I, _P]),
    "dsa_out_proj_workspace_size": (_S, []),
    "dsa_out_proj": (_I, [_P, _P, _P, _I, _I, _I, _P, _P, _S, _P]),
    "dsa_sparse_attn_fwd_oproj_workspace_size": (_S, [_I, _I, _I, _I]),
    "dsa_sparse_attn_fwd_oproj": (_I, [_I, _P, _P, _P, _I, _I, _I, _I, _F, _P, _P, _I, _P, _P, _P, _P, _S, _P]),
}

STATUS = {0: "DSA_OK", 1: "DSA_ERR_INVALID_ARG", 2: "DSA_ERR_UNSUPPORTED", 3: "DSA_ERR_MISALIGNED", 4: "DSA_ERR_CUDA",
          5: "DSA_ERR_DEVICE_TIMEOUT", 6: "DSA_ERR_WORKSPACE"}

_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the library (once).  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(f"CUDA library not built: {path} is missing (run sparse_mla_attention_dsa_gb300.build)")
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


class DsaError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {STATUS.get(code, code)}")
        self.code = code
