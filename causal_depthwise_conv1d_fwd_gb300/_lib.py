"""ctypes loader for libccv.so, the CUDA library behind include/ccv.h.

There is no fallback: if the library has not been built, loading raises.
"""
from __future__ import annotations

import ctypes
import os
import re

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libccv.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "ccv.h")

P = ctypes.c_void_p
I64 = ctypes.c_int64
I32 = ctypes.c_int


class PagedStream(ctypes.Structure):
    """struct ccv_paged_stream of include/ccv.h."""
    _fields_ = [("x", P), ("x_stride_t", I64), ("weight", P), ("w_stride_c", I64),
                ("w_stride_w", I64), ("out", P), ("out_stride_t", I64), ("off_s", I32),
                ("ws", I32)]


# Argument lists, in the order of the declarations in include/ccv.h.
SIGNATURES = {
    "ccv_status_string": ([I32], ctypes.c_char_p),
    "ccv_version": ([], I32),
    "ccv_fwd": ([P, I64, I64, P, I64, I64, P, I64, I64, P,
                 P, I64, I64, I64, I32, I32, P, I32, P, P,
                 I32, I32, I32, I32, I32, P, P], I32),
    "ccv_update": ([P, I64, I64, I64, P, I64, I64, I64, P, I64, I64, P,
                    P, I64, I64, I64, I32, I32, P, I32, I32, I32,
                    I32, I32, I32, P, P], I32),
    "ccv_update_spec": ([P, I64, I64, I64, P, I64, I64, I64, P, I64, I64, P,
                         P, I64, I64, I64, I32, I32, P, P,
                         P, I64, I64, I64, I64, I32, P, I64, I64, I32,
                         I32, I32, I32, I32, I32, I32, P, P], I32),
    "paged_sconv_seq_metadata": ([P, I32, I32, I32, P, P, I32, P], I32),
    "paged_sconv_fwd": ([P, I64, P, I64, I64, I64, I32, I32, I32, I32,
                         P, I64, I64, P, I64, P, P, P, P, I64, I32, I32,
                         P, I32, I32, I32, I32, I32, I32, P, P], I32),
    "paged_sconv_fwd_with_metadata": ([P, I64, P, I64, I64, I64, I32, I32, I32, I32,
                                       P, I64, I64, P, I64, P, P, I32, I32, P, P,
                                       P, P, I64, I32, I32, I32, I32, I32, I32, I32, I32,
                                       P, P], I32),
    "paged_sconv_fwd_streams": ([P, I32, P, I64, I64, I64, I32, I32, I32, I32,
                                 P, P, P, P, I64, I32, I32, P, I32, I32, I32, I32, P, P], I32),
}

_LIB = None


class CcvError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


def load():
    """Load libccv.so once.  Raises if it has not been built."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"libccv.so is not built ({LIB_PATH} missing); build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _LIB = lib
    return _LIB


def status_string(status: int) -> str:
    return load().ccv_status_string(int(status)).decode()


def declared_functions():
    """Names of the functions declared in include/ccv.h."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)
