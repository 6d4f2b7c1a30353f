"""ctypes binding of libtq.so (the C ABI in include/tq.h): argument marshalling only.

Every computation happens in the library's CUDA kernels.  If the library is missing or
cannot be loaded, the first call raises -- there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtq.so")

TQ_TURBO2 = 2
TQ_TURBO3 = 3
TQ_BLOCK_VALUES = 128
# TQ_NOALLOC_SCRATCH_BYTES of tq.h: the fixed scratch of tq_attn_decode_noalloc
NOALLOC_SCRATCH_BYTES = 8 << 20

STATUS_NAMES = {
    0: "TQ_OK", 1: "TQ_ERR_INVALID_ARGUMENT", 2: "TQ_ERR_UNSUPPORTED", 3: "TQ_ERR_NOT_INITIALIZED",
    4: "TQ_ERR_WORKSPACE_TOO_SMALL", 5: "TQ_ERR_CUDA", 6: "TQ_ERR_DEVICE_TIMEOUT",
    7: "TQ_ERR_OUT_OF_RANGE",
}


class TQError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)}")


class TqCache(ctypes.Structure):
    """Mirror of struct tq_cache."""
    _fields_ = [
        ("type", ctypes.c_int32),
        ("n_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("page_tokens", ctypes.c_int32),
        ("base", ctypes.c_void_p),
        ("capacity_tokens", ctypes.c_int64),
        ("n_seqs", ctypes.c_int32),
        ("max_pages_per_seq", ctypes.c_int32),
        ("page_table", ctypes.c_void_p),
        ("n_pages", ctypes.c_int64),
        ("rotation_signs", ctypes.c_uint32 * 4),
        ("norm_correction", ctypes.c_int32),
    ]


_lib = None

# name -> (restype, argtypes); the list of exported symbols the header declares
SIGNATURES = {
    "tq_block_bytes": (ctypes.c_size_t, [ctypes.c_int]),
    "tq_row_bytes": (ctypes.c_size_t, [ctypes.c_int, ctypes.c_int, ctypes.c_int]),
    "tq_codebook_init": (ctypes.c_int, [ctypes.c_int, ctypes.c_int]),
    "tq_codebook_get": (ctypes.c_int, [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]),
    "tq_encode": (ctypes.c_int, [ctypes.POINTER(TqCache), ctypes.c_void_p, ctypes.c_int64,
                                 ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                 ctypes.c_int64, ctypes.c_void_p]),
    "tq_encode_kv": (ctypes.c_int, [ctypes.POINTER(TqCache), ctypes.POINTER(TqCache),
                                    ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                    ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
                                    ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                                    ctypes.c_void_p]),
    "tq_decode": (ctypes.c_int, [ctypes.POINTER(TqCache), ctypes.c_int32, ctypes.c_int64,
                                 ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]),
    "tq_attn_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                  ctypes.c_int64]),
    "tq_attn_decode": (ctypes.c_int, [ctypes.POINTER(TqCache), ctypes.POINTER(TqCache),
                                      ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                      ctypes.c_int64, ctypes.c_float, ctypes.c_void_p,
                                      ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "tq_attn_decode_append": (ctypes.c_int, [ctypes.POINTER(TqCache), ctypes.POINTER(TqCache),
                                             ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                             ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                             ctypes.c_int64, ctypes.c_float, ctypes.c_void_p,
                                             ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "tq_attn_decode_noalloc": (ctypes.c_int, [ctypes.POINTER(TqCache), ctypes.POINTER(TqCache),
                                              ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                              ctypes.c_void_p, ctypes.c_int64, ctypes.c_float,
                                              ctypes.c_void_p, ctypes.c_void_p]),
    "tq_attn_prefill": (ctypes.c_int, [ctypes.POINTER(TqCache), ctypes.POINTER(TqCache),
                                       ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                                       ctypes.c_int64, ctypes.c_int, ctypes.c_float,
                                       ctypes.c_void_p, ctypes.c_void_p]),
    "tq_inject_wait_timeout": (ctypes.c_int, [ctypes.c_int]),
    "tq_device_status": (ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32)]),
    "tq_status_str": (ctypes.c_char_p, [ctypes.c_int]),
}


def load(path: str | None = None):
    """Load libtq.so (once).  Raises if it is missing: the CUDA path is the only path."""
    global _lib
    if _lib is not None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"{p} is missing: build it with rotated_bit_kv_tq_gb300.build.build() "
                           "(there is no CPU fallback)")
    lib = ctypes.CDLL(p)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def check(status: int, what: str):
    if status != 0:
        raise TQError(status, what)
