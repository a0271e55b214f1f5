"""ctypes loader for the in-tree CUDA library libtd.so (no fallback: a missing library is an error)."""
from __future__ import annotations

import ctypes
import os
import threading

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_build", "libtd.so")

# the exported symbols, as declared in include/td.h
SYMBOLS = (
    "td_status_string",
    "td_version",
    "td_last_cuda_error",
    "td_decode_workspace_bytes",
    "td_split_plan",
    "td_rope_kv_append",
    "td_rope_append_attn",
    "td_spec_accept",
    "td_spec_workspace_bytes",
    "td_quantize_q8",
    "td_kv_append_q8",
    "td_decode_attn_q8",
    "td_verify_attn_q8",
    "td_prefill_attn",
    "td_kv_append",
    "td_decode_attn",
    "td_verify_attn",
    "td_lse_merge",
    "td_decode_attn_noalloc",
    "td_selftest_wait_timeout",
)

_lock = threading.Lock()
_lib = None


class TDError(RuntimeError):
    """A td_* call returned a status other than TD_OK."""

    def __init__(self, func: str, status: int, message: str):
        super().__init__(f"{func} failed: {message} (status {status})")
        self.status = status


def _declare(lib):
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.td_status_string.argtypes = [i]
    lib.td_status_string.restype = ctypes.c_char_p
    lib.td_version.argtypes = []
    lib.td_version.restype = ctypes.c_char_p
    lib.td_last_cuda_error.argtypes = []
    lib.td_last_cuda_error.restype = i
    lib.td_decode_workspace_bytes.argtypes = [i, i, i, i, i, i, i]
    lib.td_decode_workspace_bytes.restype = sz
    lib.td_split_plan.argtypes = [i, i, i, i, i, i, i, i, vp, vp, vp, vp]
    lib.td_split_plan.restype = i
    lib.td_rope_kv_append.argtypes = [i, vp, vp, i, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, vp, vp]
    lib.td_rope_kv_append.restype = i
    lib.td_rope_append_attn.argtypes = [i, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, i, vp, vp, vp,
                                        sz, vp, vp]
    lib.td_rope_append_attn.restype = i
    lib.td_spec_accept.argtypes = [vp, vp, vp, vp, i, i, i, f, vp, vp, vp, sz, vp, vp]
    lib.td_spec_workspace_bytes.argtypes = [i, i, i]
    lib.td_spec_workspace_bytes.restype = sz
    ll = ctypes.c_longlong
    lib.td_quantize_q8.argtypes = [i, vp, ll, i, vp, vp, vp]
    lib.td_quantize_q8.restype = i
    lib.td_kv_append_q8.argtypes = [i, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, vp, vp]
    lib.td_kv_append_q8.restype = i
    lib.td_decode_attn_q8.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, vp, vp, sz, vp, vp]
    lib.td_decode_attn_q8.restype = i
    lib.td_verify_attn_q8.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp, vp, vp, sz, vp, vp]
    lib.td_verify_attn_q8.restype = i
    lib.td_prefill_attn.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, f, vp, vp, vp, vp]
    lib.td_prefill_attn.restype = i
    lib.td_spec_accept.restype = i
    lib.td_kv_append.argtypes = [i, vp, vp, vp, vp, vp, i, i, i, i, i, i, vp, vp]
    lib.td_kv_append.restype = i
    lib.td_decode_attn.argtypes = [i, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, vp, vp, sz, vp, vp]
    lib.td_decode_attn.restype = i
    lib.td_verify_attn.argtypes = [i, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp, vp, vp, sz, vp, vp]
    lib.td_verify_attn.restype = i
    lib.td_lse_merge.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, vp, vp, vp]
    lib.td_lse_merge.restype = i
    lib.td_decode_attn_noalloc.argtypes = [i, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, vp, vp, vp]
    lib.td_decode_attn_noalloc.restype = i
    lib.td_selftest_wait_timeout.argtypes = [ll, vp, vp, vp]
    lib.td_selftest_wait_timeout.restype = i
    return lib


def lib():
    """The loaded library; raises if it has not been built (run the package's build())."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise RuntimeError(
                        f"CUDA library not built ({LIB_PATH} missing); run "
                        "`python -m decode_attention_split_gb300.build` first")
                _lib = _declare(ctypes.CDLL(LIB_PATH))
    return _lib


def check(func: str, status: int) -> None:
    if status != 0:
        msg = lib().td_status_string(status).decode()
        if status == 4:
            msg += f" (cudaError {lib().td_last_cuda_error()})"
        raise TDError(func, status, msg)
