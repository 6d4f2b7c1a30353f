"""Oracle for the rotated, bit-packed KV cache (turbo3 / turbo2).

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import this package.  It wraps the plain
single-threaded C oracle in ``tq_oracle.c`` (see ``tq_oracle.h`` for what each
function follows and how it is pinned) and never touches the CUDA library.

Sources, by title and section:
  * "llama.cpp に TurboQuant を実装" (TurboQuant in llama.cpp, openalchemy.io):
    "What TurboQuant does differently", "How small does it get",
    "Why the KV cache is so heavy".
  * kenji.blog C++ inference-engine article, section 8 (attention, KV cache);
    kenji.blog TinyLLaMA article, sections 4.3 (GQA) and 7 (KV cache).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tq_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

TURBO2 = 2
TURBO3 = 3
BLOCK = 128


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc: -O2, no FMA contraction, no fast-math."""
    if force or not os.path.exists(_LIB_PATH) or (
        os.path.getmtime(_LIB_PATH) < max(os.path.getmtime(_SRC),
                                           os.path.getmtime(os.path.join(_HERE, "tq_oracle.h")))):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
                               "-Wall", "-Wextra", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB_PATH)
    P = ctypes.c_void_p
    i64, i32, dbl = ctypes.c_int64, ctypes.c_int, ctypes.c_double
    lib.oracle_block_bytes.restype = ctypes.c_size_t
    lib.oracle_block_bytes.argtypes = [i32]
    lib.oracle_kv_bytes.restype = ctypes.c_uint64
    lib.oracle_kv_bytes.argtypes = [ctypes.c_uint64] * 6
    lib.oracle_f16_to_f32.restype = ctypes.c_float
    lib.oracle_f16_to_f32.argtypes = [ctypes.c_uint16]
    lib.oracle_f32_to_f16.restype = ctypes.c_uint16
    lib.oracle_f32_to_f16.argtypes = [ctypes.c_float]
    lib.oracle_fwht_f32.argtypes = [P, i32]
    lib.oracle_fwht_f64.argtypes = [P, i32]
    lib.oracle_codebook.restype = i32
    lib.oracle_codebook.argtypes = [i32, i32, P, P, P]
    lib.oracle_encode_block.argtypes = [i32, P, P, P]
    lib.oracle_decode_block.argtypes = [i32, P, P, P]
    lib.oracle_unpack_block.argtypes = [i32, P, P, P]
    lib.oracle_encode_rows.argtypes = [i32, P, i64, i32, i32, i64, P, P]
    lib.oracle_decode_rows.argtypes = [i32, P, i64, i32, i32, P, P]
    lib.oracle_dense_attention.argtypes = [P, P, P, i64, i32, i32, i32, dbl, P]
    lib.oracle_attn_decode.argtypes = [i32, i32, P, P, P, i64, i32, i32, i32, dbl, P, P, P]
    lib.oracle_attn_prefill.argtypes = [i32, i32, P, P, P, i64, i64, i32, i32, i32, dbl, P, P, P]
    lib.oracle_encode_block_v.argtypes = [i32, P, P, P, P, P]
    lib.oracle_decode_block_v.argtypes = [i32, P, P, P, P]
    lib.oracle_encode_rows_v.argtypes = [i32, P, i64, i32, i32, i64, P, P, P, P]
    lib.oracle_decode_rows_v.argtypes = [i32, P, i64, i32, i32, P, P, P]
    lib.oracle_attn_decode_v.argtypes = [i32, i32, P, P, P, i64, i32, i32, i32, dbl, P, P, P, P, P]
    lib.oracle_attn_prefill_v.argtypes = [i32, i32, P, P, P, i64, i64, i32, i32, i32, dbl, P, P,
                                          P, P, P]
    _lib = lib
    return lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def block_bytes(tq_type: int) -> int:
    return int(_load().oracle_block_bytes(tq_type))


def kv_bytes(layers, kv_heads, head_dim, ctx, bytes_num, bytes_den) -> int:
    return int(_load().oracle_kv_bytes(layers, kv_heads, head_dim, ctx, bytes_num, bytes_den))


def f16_to_f32(h: int) -> float:
    return float(_load().oracle_f16_to_f32(h))


def f32_to_f16(f: float) -> int:
    return int(_load().oracle_f32_to_f16(f))


def fwht_f32(x: np.ndarray) -> np.ndarray:
    y = np.ascontiguousarray(x, dtype=np.float32).copy()
    _load().oracle_fwht_f32(_ptr(y), y.size)
    return y


def fwht_f64(x: np.ndarray) -> np.ndarray:
    y = np.ascontiguousarray(x, dtype=np.float64).copy()
    _load().oracle_fwht_f64(_ptr(y), y.size)
    return y


_codebook_cache: dict = {}


def codebook(d: int, levels: int):
    """(centroids_f64, centroids_f32, thresholds_f32, iterations) for dimension d."""
    key = (d, levels)
    if key not in _codebook_cache:
        c64 = np.zeros(levels, np.float64)
        c32 = np.zeros(levels, np.float32)
        t32 = np.zeros(levels - 1, np.float32)
        it = _load().oracle_codebook(d, levels, _ptr(c64), _ptr(c32), _ptr(t32))
        if it < 0:
            raise ValueError("bad codebook arguments")
        _codebook_cache[key] = (c64, c32, t32, it)
    c64, c32, t32, it = _codebook_cache[key]
    return c64.copy(), c32.copy(), t32.copy(), it


def type_codebook(tq_type: int):
    """fp32 centroids and thresholds of a cache type (d = 128)."""
    _, c, t, _ = codebook(BLOCK, 1 << tq_type)
    return c, t


class Variant(ctypes.Structure):
    """oracle_variant: sign bits of the random-sign Hadamard W D (bit i of the 128-bit
    mask, word i // 32, negates coordinate i) and the norm-correction flag."""
    _fields_ = [("signs", ctypes.c_uint32 * 4), ("norm_correction", ctypes.c_int32)]


def variant(signs=None, norm_correction=False):
    """A Variant from a 128-entry 0/1 array (or an int mask) and a flag; None for none."""
    if signs is None and not norm_correction:
        return None
    v = Variant()
    if signs is not None:
        mask = signs if isinstance(signs, int) else sum(int(b) << i for i, b in enumerate(signs))
        for w in range(4):
            v.signs[w] = (mask >> (32 * w)) & 0xFFFFFFFF
    v.norm_correction = 1 if norm_correction else 0
    return v


def _vref(v):
    return ctypes.byref(v) if v is not None else None


def encode_block(tq_type: int, x_f16_bits: np.ndarray, var=None) -> np.ndarray:
    c, t = type_codebook(tq_type)
    x = np.ascontiguousarray(x_f16_bits, dtype=np.uint16)
    assert x.size == BLOCK
    out = np.zeros(block_bytes(tq_type), np.uint8)
    _load().oracle_encode_block_v(tq_type, _ptr(x), _ptr(t), _ptr(c), _vref(var), _ptr(out))
    return out


def decode_block(tq_type: int, blk: np.ndarray, var=None) -> np.ndarray:
    c, _ = type_codebook(tq_type)
    b = np.ascontiguousarray(blk, dtype=np.uint8)
    out = np.zeros(BLOCK, np.float64)
    _load().oracle_decode_block_v(tq_type, _ptr(b), _ptr(c), _vref(var), _ptr(out))
    return out


def unpack_block(tq_type: int, blk: np.ndarray):
    b = np.ascontiguousarray(blk, dtype=np.uint8)
    codes = np.zeros(BLOCK, np.uint8)
    norm = np.zeros(1, np.uint16)
    _load().oracle_unpack_block(tq_type, _ptr(b), _ptr(codes), _ptr(norm))
    return codes, int(norm[0])


def encode_rows(tq_type: int, src_f16: np.ndarray, n_kv_heads: int, head_dim: int,
                src_stride: int | None = None, var=None) -> np.ndarray:
    """src_f16: uint16 (fp16 bits) or float16 array whose first axis is tokens."""
    c, t = type_codebook(tq_type)
    src = np.ascontiguousarray(src_f16).view(np.uint16)
    n_tokens = src.shape[0]
    stride = n_kv_heads * head_dim if src_stride is None else src_stride
    nb = head_dim // BLOCK
    out = np.zeros((n_tokens, n_kv_heads * nb * block_bytes(tq_type)), np.uint8)
    _load().oracle_encode_rows_v(tq_type, _ptr(src), n_tokens, n_kv_heads, head_dim, stride,
                                 _ptr(t), _ptr(c), _vref(var), _ptr(out))
    return out


def decode_rows(tq_type: int, rows: np.ndarray, n_kv_heads: int, head_dim: int,
                var=None) -> np.ndarray:
    c, _ = type_codebook(tq_type)
    r = np.ascontiguousarray(rows, dtype=np.uint8)
    n_tokens = r.shape[0]
    out = np.zeros((n_tokens, n_kv_heads, head_dim), np.float64)
    _load().oracle_decode_rows_v(tq_type, _ptr(r), n_tokens, n_kv_heads, head_dim, _ptr(c),
                                 _vref(var), _ptr(out))
    return out


def dense_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, n_kv_heads: int,
                    scale: float) -> np.ndarray:
    """q [Hq][D], k/v [T][Hkv][D] (any float dtype) -> [Hq][D] float64."""
    q64 = np.ascontiguousarray(q, dtype=np.float64)
    k64 = np.ascontiguousarray(k, dtype=np.float64)
    v64 = np.ascontiguousarray(v, dtype=np.float64)
    hq, d = q64.shape
    out = np.zeros((hq, d), np.float64)
    _load().oracle_dense_attention(_ptr(q64), _ptr(k64), _ptr(v64), k64.shape[0], hq,
                                   n_kv_heads, d, float(scale), _ptr(out))
    return out


def attn_decode(type_k: int, type_v: int, k_rows: np.ndarray, v_rows: np.ndarray,
                q_f16: np.ndarray, n_tokens: int, n_q_heads: int, n_kv_heads: int,
                head_dim: int, scale: float, var_k=None, var_v=None) -> np.ndarray:
    """Attention of one query row over the first n_tokens packed rows -> [Hq][D] f64."""
    ck, _ = type_codebook(type_k)
    cv, _ = type_codebook(type_v)
    kr = np.ascontiguousarray(k_rows, dtype=np.uint8)
    vr = np.ascontiguousarray(v_rows, dtype=np.uint8)
    q = np.ascontiguousarray(q_f16).view(np.uint16)
    out = np.zeros((n_q_heads, head_dim), np.float64)
    _load().oracle_attn_decode_v(type_k, type_v, _ptr(kr), _ptr(vr), _ptr(q), n_tokens, n_q_heads,
                                 n_kv_heads, head_dim, float(scale), _ptr(ck), _ptr(cv),
                                 _vref(var_k), _vref(var_v), _ptr(out))
    return out


def attn_prefill(type_k: int, type_v: int, k_rows: np.ndarray, v_rows: np.ndarray,
                 q_f16: np.ndarray, pos0: int, n_kv_heads: int, head_dim: int,
                 scale: float, var_k=None, var_v=None) -> np.ndarray:
    """Causal attention of a prompt chunk: q_f16 [n_q][Hq][D], query j at position pos0 + j
    over packed rows 0 .. pos0 + j  ->  [n_q][Hq][D] f64."""
    ck, _ = type_codebook(type_k)
    cv, _ = type_codebook(type_v)
    q = np.ascontiguousarray(q_f16).view(np.uint16)
    n_q, n_q_heads = q.shape[0], q.shape[1]
    kr = np.ascontiguousarray(k_rows, dtype=np.uint8)
    vr = np.ascontiguousarray(v_rows, dtype=np.uint8)
    assert kr.shape[0] >= pos0 + n_q and vr.shape[0] >= pos0 + n_q
    out = np.zeros((n_q, n_q_heads, head_dim), np.float64)
    _load().oracle_attn_prefill_v(type_k, type_v, _ptr(kr), _ptr(vr), _ptr(q), pos0, n_q,
                                  n_q_heads, n_kv_heads, head_dim, float(scale), _ptr(ck),
                                  _ptr(cv), _vref(var_k), _vref(var_v), _ptr(out))
    return out

