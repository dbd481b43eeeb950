"""ctypes handle on libpkv.so: loads the in-tree library and declares the C signatures of
include/pkv.h.  No arithmetic happens here."""
from __future__ import annotations

import ctypes
import os
import re
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libpkv.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "pkv.h")

_lock = threading.Lock()
_lib = None


class PkvDims(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32),
        ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("block_size", ctypes.c_int32),
        ("num_blocks", ctypes.c_int32),
        ("max_blocks_per_seq", ctypes.c_int32),
    ]


class PkvError(RuntimeError):
    """A call into libpkv returned a non-zero status."""

    def __init__(self, func: str, status: int, text: str):
        super().__init__(f"{func}: status {status}: {text}")
        self.status = status


def header_constants() -> dict:
    """#define NAME value pairs of include/pkv.h (status and device-error codes)."""
    out = {}
    with open(HEADER) as f:
        for m in re.finditer(r"^#define\s+(PKV_\w+)\s+([-+*() 0-9]+?)\s*(?:/\*.*)?$", f.read(), re.M):
            out[m.group(1)] = int(eval(m.group(2), {"__builtins__": {}}, {}))  # integer literal arithmetic only
    return out


def header_functions() -> list:
    """Names of the functions include/pkv.h declares."""
    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\*?(pkv_\w+)\s*\(", text, re.M)))


def load():
    """Load libpkv.so; raises if it was not built (there is no fallback path)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`"
                " (the CUDA library is required; there is no CPU fallback)")
        lib = ctypes.CDLL(LIB_PATH)
        P, I32, I64, SZ, F32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
        U32 = ctypes.c_uint32
        D = ctypes.POINTER(PkvDims)
        sig = {
            "pkv_kv_append": (I32, [P, P, P, P, P, I64, D, P, P]),
            "pkv_kv_append_q8": (I32, [P, P, P, P, P, P, P, I64, D, P, P]),
            "pkv_prefill_window_scores": (I32, [P, I32, P, I32, P, P, P, P, I32, F32, D, P, P]),
            "pkv_decode_workspace_bytes": (SZ, [D]),
            "pkv_paged_decode_attention_q8": (I32, [P, P, P, P, P, P, P, P, F32, I32, P, SZ, D, U32, P, P]),
            "pkv_paged_decode_attention": (I32, [P, P, P, P, P, P, F32, I32, P, SZ, D, U32, P, P]),
            "pkv_paged_decode_attention_append": (I32, [P, P, P, P, P, P, P, P, F32, I32, P, SZ, D, U32, P, P]),
            "pkv_paged_decode_attention_scores": (I32, [P, P, P, P, I32, P, P, P, P, P, P, P, F32, I32, P, SZ,
                                                        D, U32, P, P]),
            "pkv_kv_rolling_admit": (I32, [P, P, P, P, P, P, P, P, P, I32, I32, I32, D, U32, P, P]),
            "pkv_paged_decode_attention_scores_q8": (I32, [P, P, P, P, I32, P, P, P, P, P, P, P, F32, I32, P,
                                                           SZ, D, U32, P, P]),
            "pkv_paged_decode_attention_append_q8": (I32, [P, P, P, P, P, P, P, P, P, P, F32, I32, P, SZ, D, U32,
                                                           P, P]),
            "pkv_sparse_decode_attention_q8": (I32, [P, P, P, P, P, P, P, P, P, P, I32, F32, P, SZ, D, U32, P, P]),
            "pkv_kv_compact_q8": (I32, [P, P, P, P, P, I32, I32, P, P, P, P, P, P, P, P, I32, D, U32, P, P]),
            "pkv_kv_rolling_admit_q8": (I32, [P, P, P, P, P, P, P, P, P, P, P, I32, I32, I32, D, U32, P, P]),
            "pkv_sparse_decode_workspace_bytes": (SZ, [D, I32]),
            "pkv_sparse_decode_attention": (I32, [P, P, P, P, P, P, P, P, I32, F32, P, SZ, D, U32, P, P]),
            "pkv_kv_select_topk": (I32, [P, P, P, I32, P, I32, I32, I32, D, U32, P, P]),
            "pkv_kv_compact": (I32, [P, P, P, I32, I32, P, P, P, P, P, P, I32, D, U32, P, P]),
            "pkv_paged_decode_attention_fixed_scratch": (I32, [P, P, P, P, P, P, F32, I32, D, P, P]),
            "pkv_read_error": (I32, [P, I32, P]),
            "pkv_device_alias": (I32, [P, ctypes.POINTER(ctypes.c_void_p)]),
            "pkv_status_string": (ctypes.c_char_p, [I32]),
            "pkv_device_error_string": (ctypes.c_char_p, [I32]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def check(func: str, status: int) -> None:
    if status != 0:
        text = load().pkv_status_string(status).decode()
        raise PkvError(func, status, text)
