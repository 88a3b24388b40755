"""ctypes binding of the C ABI in include/mla.h (argument marshalling only).

Loads ``_build/libmla_gb300.so`` from this package. There is no fallback: if
the library is missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
# MLA_GB300_LIB names another build of the library to load instead (the
# bounds-checked debug variant, for its tests).
LIB_PATH = os.environ.get("MLA_GB300_LIB") or os.path.join(_HERE, "_build", "libmla_gb300.so")

MLA_OK, MLA_ERR_INVALID_ARG, MLA_ERR_UNSUPPORTED, MLA_ERR_WORKSPACE, MLA_ERR_CUDA, \
    MLA_ERR_TIMEOUT, MLA_ERR_BAD_INDEX, MLA_ERR_CHECK = range(8)
STATUS_NAMES = {0: "MLA_OK", 1: "MLA_ERR_INVALID_ARG", 2: "MLA_ERR_UNSUPPORTED",
                3: "MLA_ERR_WORKSPACE", 4: "MLA_ERR_CUDA", 5: "MLA_ERR_TIMEOUT",
                6: "MLA_ERR_BAD_INDEX", 7: "MLA_ERR_CHECK"}
OP_PREFILL, OP_DECODE, OP_INDEX_TOPK, OP_SPARSE_DECODE, OP_CACHE_APPEND, \
    OP_LATENT_DECODE, OP_PREFILL_INDEX_TOPK, OP_SPARSE_PREFILL_LATENT, OP_INDEX_TOPK_FP8, \
    OP_GATHER_PROBE = range(10)
DEBUG_WAIT_LIMIT_NS, DEBUG_STALL_STAGE, DEBUG_SPARSE_CHUNK, DEBUG_PREFILL_CTAS = 1, 2, 3, 4
NOALLOC_SCRATCH_BYTES = 16 << 20

# Every symbol include/mla.h declares, with (restype, argtypes).
_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_Z = ctypes.c_size_t
SIGNATURES = {
    "mla_prefill": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _P, _Z, _P]),
    "mla_decode": (_I, [_P, _P, _P, _P, _I, _I, _I, _P, _P, _F, _P, _Z, _P]),
    "mla_decode_noalloc": (_I, [_P, _P, _P, _P, _I, _I, _I, _P, _P, _F, _P]),
    "dsa_index_topk": (_I, [_P, _P, _P, _P, _I, _I, ctypes.c_int64, _I, _I, _P, _P, _P, _Z,
                            _P]),
    "dsa_sparse_decode": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _P, _P, _F, _P, _Z, _P]),
    "mla_cache_append": (_I, [_P, _P, _P, _P, _P, ctypes.c_int64, _I, _I, _I, _I, _P]),
    "mla_prefill_chunk": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _P, _Z, _P]),
    "mla_decode_cached": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _F, _P, _Z, _P]),
    "mla_decode_latent": (_I, [_P, _P, _P, ctypes.c_int64, _I, _I, _I, _P, _P, _P, _P, _F, _P,
                               _Z, _P]),
    "dsa_prefill_index_topk": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _Z, _P]),
    "mla_sparse_prefill_latent": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _F, _P, _Z,
                                       _P]),
    "dsa_quantize_index_keys": (_I, [_P, _P, _P, ctypes.c_int64, _P]),
    "dsa_index_topk_fp8": (_I, [_P, _P, _P, _P, _P, _I, _I, ctypes.c_int64, _I, _I, _P, _P, _P,
                                _Z, _P]),
    "mla_quantize_latent_cache": (_I, [_P, _P, ctypes.c_int64, _P]),
    "mla_decode_latent_fp8": (_I, [_P, _P, _P, ctypes.c_int64, _I, _I, _I, _P, _P, _P, _P, _F,
                                   _P, _Z, _P]),
    "mla_sparse_prefill_latent_fp8": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _F, _P,
                                           _Z, _P]),
    "mla_workspace_size": (_Z, [_I, _I, _I, _I, _I]),
    "mla_check_device_status": (_I, [_P]),
    "mla_last_error": (ctypes.c_char_p, []),
    "mla_debug_set": (_I, [_I, ctypes.c_longlong]),
    "mla_timing_enable": (_I, [_I]),
    "mla_timing_read": (_I, [_I, ctypes.POINTER(ctypes.c_double),
                             ctypes.POINTER(ctypes.c_longlong)]),
    "mla_gather_probe_blocks": (_I, []),
    "mla_gather_probe": (_I, [_P, _P, _P, _P, _I, _I, _I, _P, _P]),
}

_lock = threading.Lock()
_lib = None


class MlaError(RuntimeError):
    def __init__(self, status: int, message: str):
        self.status = status
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")


def load(path: str | None = None):
    """Load (once) and bind the library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None or path is not None:
            p = path or LIB_PATH
            if not os.path.exists(p):
                raise RuntimeError(f"{p} is missing: build it with "
                                   "`python -m mla_family_attention_gb300.build`")
            lib = ctypes.CDLL(p)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            if path is not None:
                return lib
            _lib = lib
    return _lib


def check(status: int, lib=None):
    if status != MLA_OK:
        msg = (lib or load()).mla_last_error()
        raise MlaError(status, msg.decode() if msg else "")
