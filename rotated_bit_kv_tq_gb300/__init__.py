"""GB300 rotated, bit-packed KV cache (turbo3 / turbo2) -- Python binding.

Thin marshalling layer over the C ABI of libtq.so (include/tq.h).  PyTorch supplies
device memory and streams; every step of encode, decode and attention runs in the
library's sm_103a kernels.  There is no CPU fallback: calls raise if the library is
missing.
"""
from __future__ import annotations

import ctypes

from ._lib import (NOALLOC_SCRATCH_BYTES, TQ_BLOCK_VALUES, TQ_TURBO2, TQ_TURBO3, TQError, TqCache,
                   check, load)

__all__ = ["TQ_TURBO2", "TQ_TURBO3", "TQ_BLOCK_VALUES", "NOALLOC_SCRATCH_BYTES", "TQError", "TqCache", "KVCache",
           "block_bytes", "row_bytes", "codebook_init", "codebook_get", "encode", "encode_kv", "decode",
           "attn_workspace_bytes", "attn_decode", "attn_decode_append", "attn_prefill",
           "inject_wait_timeout", "device_status", "load"]


# Pointers and stream handles are passed as plain integers (the argtypes are c_void_p), which
# keeps the per-call host cost of the decode loop low.
def _stream_ptr(stream=None):
    import torch
    if stream is not None:
        return stream.cuda_stream
    raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
    if raw is not None:   # the current stream's handle without building a Stream object
        return raw(torch.cuda.current_device())
    return torch.cuda.current_stream().cuda_stream


def _ptr(t):
    return t.data_ptr() if t is not None else None


def block_bytes(tq_type: int) -> int:
    return int(load().tq_block_bytes(tq_type))


def row_bytes(tq_type: int, n_kv_heads: int, head_dim: int) -> int:
    return int(load().tq_row_bytes(tq_type, n_kv_heads, head_dim))


def codebook_init(tq_type: int, device: int = 0):
    check(load().tq_codebook_init(tq_type, device), "tq_codebook_init")


def codebook_get(tq_type: int):
    import numpy as np
    levels = 1 << tq_type
    c = np.zeros(levels, np.float32)
    t = np.zeros(levels - 1, np.float32)
    check(load().tq_codebook_get(tq_type, c.ctypes.data_as(ctypes.c_void_p),
                                 t.ctypes.data_as(ctypes.c_void_p)), "tq_codebook_get")
    return c, t


class KVCache:
    """One layer's K or V cache: a PyTorch uint8 device buffer plus its tq_cache view.

    Contiguous: ``capacity_tokens`` rows per sequence.  Paged: pass ``page_tokens`` and an
    int32 device ``page_table`` [n_seqs, max_pages]; the pool holds ``n_pages`` pages.
    Variants: ``rotation_signs`` (a 128-bit int or 128 0/1 values: coordinate i negated
    before the rotation, W D) and ``norm_correction`` (store |x| / |c|).
    """

    def __init__(self, tq_type: int, n_kv_heads: int, head_dim: int, *, n_seqs: int = 1,
                 capacity_tokens: int = 0, page_tokens: int = 0, page_table=None,
                 n_pages: int = 0, device=None, buffer=None, rotation_signs=None,
                 norm_correction: bool = False):
        import torch
        self.type, self.n_kv_heads, self.head_dim = tq_type, n_kv_heads, head_dim
        self.row_bytes = row_bytes(tq_type, n_kv_heads, head_dim)
        if self.row_bytes == 0:
            raise TQError(1, "KVCache: bad shape")
        rows = n_pages * page_tokens if page_tokens else n_seqs * capacity_tokens
        if buffer is None:
            buffer = torch.zeros(rows * self.row_bytes, dtype=torch.uint8,
                                 device=device if device is not None else "cuda")
        self.buffer = buffer
        self.page_table = page_table
        self.view = TqCache(tq_type, n_kv_heads, head_dim, page_tokens, buffer.data_ptr(),
                            capacity_tokens, n_seqs, page_table.shape[1] if page_table is not None else 0,
                            page_table.data_ptr() if page_table is not None else None, n_pages)
        if rotation_signs is not None:
            mask = (rotation_signs if isinstance(rotation_signs, int)
                    else sum(int(b) << i for i, b in enumerate(rotation_signs)))
            for w in range(4):
                self.view.rotation_signs[w] = (mask >> (32 * w)) & 0xFFFFFFFF
        self.view.norm_correction = 1 if norm_correction else 0
        self.ref = ctypes.byref(self.view)   # what the C calls take (the view is updated in place)

    @property
    def nbytes(self) -> int:
        return self.buffer.numel()


def encode(cache: KVCache, src, *, seq_ids=None, positions=None, seq_id: int = 0, pos0: int = 0,
           stream=None):
    """src: fp16 device tensor [n_tokens, n_kv_heads*head_dim] (row stride = src.stride(0))."""
    n = src.shape[0]
    stride = src.stride(0) if src.dim() > 1 else cache.n_kv_heads * cache.head_dim
    check(load().tq_encode(cache.ref, _ptr(src), n, stride, _ptr(seq_ids),
                           _ptr(positions), seq_id, pos0, _stream_ptr(stream)), "tq_encode")


def encode_kv(kc: KVCache, vc: KVCache, k_src, v_src, *, seq_ids=None, positions=None,
              seq_id: int = 0, pos0: int = 0, stream=None):
    """K rows into kc and V rows into vc in one launch (same arguments as encode)."""
    n = k_src.shape[0]
    if v_src.shape[0] != n:
        raise TQError(1, "encode_kv: K and V token counts differ")
    ks = k_src.stride(0) if k_src.dim() > 1 else kc.n_kv_heads * kc.head_dim
    vs = v_src.stride(0) if v_src.dim() > 1 else vc.n_kv_heads * vc.head_dim
    check(load().tq_encode_kv(kc.ref, vc.ref, _ptr(k_src),
                              _ptr(v_src), n, ks, vs, _ptr(seq_ids), _ptr(positions), seq_id,
                              pos0, _stream_ptr(stream)), "tq_encode_kv")


def decode(cache: KVCache, seq_id: int, pos0: int, n_tokens: int, out, stream=None):
    check(load().tq_decode(cache.ref, seq_id, pos0, n_tokens, _ptr(out),
                           _stream_ptr(stream)), "tq_decode")


def attn_workspace_bytes(n_seqs: int, n_q_heads: int, head_dim: int, max_seq_len: int) -> int:
    return int(load().tq_attn_workspace_bytes(n_seqs, n_q_heads, head_dim, max_seq_len))


def attn_decode(k: KVCache, v: KVCache, q, seq_lens, max_seq_len: int, out, workspace,
                softmax_scale: float = 0.0, stream=None):
    """q: fp16 [n_seqs, n_q_heads, head_dim]; seq_lens int32 [n_seqs]; out fp32 like q."""
    n_seqs, n_q_heads = q.shape[0], q.shape[1]
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    check(load().tq_attn_decode(k.ref, v.ref, _ptr(q), n_seqs,
                                n_q_heads, _ptr(seq_lens), max_seq_len, softmax_scale, _ptr(out),
                                _ptr(workspace), ws_bytes, _stream_ptr(stream)), "tq_attn_decode")


def attn_decode_append(k: KVCache, v: KVCache, k_new, v_new, q, seq_lens, max_seq_len: int, out,
                       workspace, softmax_scale: float = 0.0, stream=None):
    """One decode step: k_new / v_new fp16 [n_seqs, n_kv_heads, head_dim] go to position
    seq_lens[s] - 1 of sequence s, then attention as attn_decode (seq_lens counts them)."""
    n_seqs, n_q_heads = q.shape[0], q.shape[1]
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    check(load().tq_attn_decode_append(k.ref, v.ref, _ptr(k_new),
                                       _ptr(v_new), _ptr(q), n_seqs, n_q_heads, _ptr(seq_lens),
                                       max_seq_len, softmax_scale, _ptr(out), _ptr(workspace),
                                       ws_bytes, _stream_ptr(stream)), "tq_attn_decode_append")


def attn_prefill(k: KVCache, v: KVCache, q, out, *, pos0: int, seq_id: int = 0,
                 softmax_scale: float = 0.0, stream=None):
    """Causal attention of a prompt chunk: q fp16 [n_q, n_q_heads, head_dim], query j at
    position pos0 + j over cache rows 0 .. pos0 + j of seq_id (its own rows encoded
    first); out fp32 like q."""
    n_q, n_q_heads = q.shape[0], q.shape[1]
    check(load().tq_attn_prefill(k.ref, v.ref, _ptr(q), seq_id,
                                 pos0, n_q, n_q_heads, softmax_scale, _ptr(out),
                                 _stream_ptr(stream)), "tq_attn_prefill")


def inject_wait_timeout(n_calls: int):
    """The next n_calls tensor-core decode-attention launches withhold their tile copies
    and time out their bounded waits (a test of the failure path; no GPU fault)."""
    check(load().tq_inject_wait_timeout(n_calls), "tq_inject_wait_timeout")


def device_status(stream=None) -> int:
    st = ctypes.c_int32(0)
    check(load().tq_device_status(_stream_ptr(stream), ctypes.byref(st)), "tq_device_status")
    return int(st.value)
