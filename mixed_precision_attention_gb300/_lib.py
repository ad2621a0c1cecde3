"""ctypes loader for libapa.so (the C ABI declared in include/apa.h).

There is no fallback: if the library has not been built, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_lib", "libapa.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "apa.h")

APA_OK = 0
_lock = threading.Lock()
_lib = None

P, I, F, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
_SIGS = {
    "apa_attention": (I, [P, P, P, I, I, I, I, I, I, I, F, P, P, P, P]),
    "apa_attention_ws": (I, [P, P, P, I, I, I, I, I, I, I, F, P, P, P, P, SZ, P]),
    "apa_attention_host": (I, [P, P, P, I, I, I, I, I, I, I, F, P, P, P, P]),
    "apa_attention_paged": (I, [P, P, P, I, P, I, I, I, I, I, I, I, I, F, P, P, P, P]),
    "apa_workspace_bytes": (SZ, [I, I, I, I, I, I, F]),
    "apa_attention_ex": (I, [P, P, P, I, I, I, I, I, I, I, F, ctypes.c_uint, P, P, P, P, SZ, P]),
    "apa_workspace_bytes_ex": (SZ, [I, I, I, I, I, I, F, ctypes.c_uint]),
    "apa_workspace_operands": (I, [I, I, I, I, I, I, F, ctypes.c_uint, P, P, P, P, P, P]),
    "apa_quantize_ex": (I, [P, P, P, I, I, I, I, I, I, ctypes.c_uint, P, P, P, P, P, P, P, P]),
    "apa_quantize": (I, [P, P, P, I, I, I, I, I, I, P, P, P, P, P, P, P]),
    "apa_quantize_noalloc": (I, [P, P, P, I, I, I, I, I, I, P, P, P, P, P, P, P]),
    "apa_quantize_noalloc_scratch_bytes": (SZ, [I, I, I, I, I]),
    "apa_kv_blob_bytes": (SZ, [I, I, I, I]),
    "apa_q_blob_bytes": (SZ, [I, I, I, I, I]),
    "apa_check_error": (I, [P]),
    "apa_stage_timing": (I, [I]),
    "apa_stage_timing_read": (I, [P, P]),
    "apa_status_string": (ctypes.c_char_p, [I]),
}


class ApaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


def declared_functions() -> list[str]:
    """Names of the functions include/apa.h declares."""
    with open(HEADER) as f:
        text = f.read()
    return re.findall(r"^\s*(?:int|size_t|const char\*)\s+(apa_\w+)\s*\(", text, flags=re.M)


def load():
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                                   "mixed_precision_attention_gb300.build.build() (nvcc, sm_103a)")
            lib = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in _SIGS.items():
                fn = getattr(lib, name)
                fn.restype, fn.argtypes = res, args
            _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load().apa_status_string(int(status)).decode()


def check(status: int, what: str):
    if status != APA_OK:
        raise ApaError(status, what)
