"""Seeded synthetic workloads for the rotated, bit-packed KV cache.

This module holds no part of the method's arithmetic: it only draws the fp16 K, V and
query tensors, sequence lengths and page permutations that the tests and the benchmark
feed to both the CUDA library and the oracle.  The pages measure on real models
(Qwen2.5-Coder-14B and a head_dim-256 9B model, "llama.cpp に TurboQuant を実装",
section "Numbers on real models"); no weights are available here, so these draws stand
in for post-RoPE keys and values of those shapes.

Random numbers come from NumPy's Philox counter-based generator (Salmon et al., SC'11),
one independent key per (seed, workload, layer, stream, sequence, chunk), so any token
range of any layer can be regenerated on its own and in any order.

Recipe (all values rounded to fp16, round to nearest even):
  * V[t, h, c] ~ N(0, 1); q[h, c] ~ N(0, 1).
  * K[t, h, c] ~ N(0, 1) * s[h, c] * o[h, c] with s ~ lognormal(0, 0.5) drawn once per
    (layer, KV head, channel) and o = outlier_gain on ``n_outliers`` channels per
    (layer, KV head) picked without replacement, o = 1 elsewhere.  Outlier channels model
    the large KV outliers that motivate the rotation ("Why the KV cache is so heavy").
"""
from __future__ import annotations

import concurrent.futures
import dataclasses
import os

import numpy as np

CHUNK = 64  # tokens per generator key

_STREAMS = {"K": 1, "V": 2, "Q": 3, "scale": 4, "outlier": 5, "lens": 6, "pages": 7}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    wid: int                 # small integer id mixed into every generator key
    layers: int
    n_kv_heads: int
    n_q_heads: int
    head_dim: int
    ctx: int                 # context length (max length for the batched workload)
    types: tuple             # cache types run on this workload (3 = turbo3, 2 = turbo2)
    n_seqs: int = 1
    decode_steps: int = 0
    n_outliers: int = 4
    outlier_gain: float = 10.0
    page_tokens: int = 0     # 0 = contiguous cache
    len_range: tuple = (0, 0)  # batched workload: lengths uniform in [lo, hi]
    seed: int = 0

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads


# The five workloads.  Shapes follow Llama-3-8B, Qwen2.5-14B and a head_dim-256 model.
TINY = Workload("tiny", 0, layers=1, n_kv_heads=2, n_q_heads=8, head_dim=128, ctx=256,
                types=(3,), decode_steps=1)
LLAMA3_8B_32K = Workload("llama3-8b-kv-32k", 1, layers=32, n_kv_heads=8, n_q_heads=32,
                         head_dim=128, ctx=32768, types=(3,), decode_steps=128)
QWEN25_14B_32K = Workload("qwen2.5-14b-kv-32k", 2, layers=48, n_kv_heads=8, n_q_heads=40,
                          head_dim=128, ctx=32768, types=(3, 2), decode_steps=1)
HD256_128K = Workload("hd256-kv-128k", 3, layers=32, n_kv_heads=4, n_q_heads=16, head_dim=256,
                      ctx=131072, types=(2,), decode_steps=1, n_outliers=8, outlier_gain=20.0)
BATCHED_PAGED = Workload("batched-paged-64seq", 4, layers=32, n_kv_heads=8, n_q_heads=32,
                         head_dim=128, ctx=16384, types=(3,), n_seqs=64, decode_steps=128,
                         page_tokens=256, len_range=(1024, 16384))

WORKLOADS = [TINY, LLAMA3_8B_32K, QWEN25_14B_32K, HD256_128K, BATCHED_PAGED]


def _gen(w: Workload, stream: str, layer: int = 0, seq: int = 0, chunk: int = 0,
         extra: int = 0) -> np.random.Generator:
    k0 = ((w.seed & 0xFFFFFFFF) << 32) | ((w.wid & 0xFF) << 24) | ((_STREAMS[stream] & 0xFF) << 16) \
        | (layer & 0xFFFF)
    k1 = ((seq & 0xFFFF) << 48) | ((extra & 0xFFFF) << 32) | (chunk & 0xFFFFFFFF)
    return np.random.Generator(np.random.Philox(key=np.array([k0, k1], dtype=np.uint64)))


def k_channel_gain(w: Workload, layer: int) -> np.ndarray:
    """[n_kv_heads, head_dim] float32 per-channel gain of K (lognormal scale x outliers)."""
    g = _gen(w, "scale", layer)
    s = np.exp(0.5 * g.standard_normal((w.n_kv_heads, w.head_dim))).astype(np.float32)
    go = _gen(w, "outlier", layer)
    for h in range(w.n_kv_heads):
        ch = go.permutation(w.head_dim)[: w.n_outliers]
        s[h, ch] *= np.float32(w.outlier_gain)
    return s


def _fill_chunks(w, layer, kind, t0, n, seq, gain, out, c_lo, c_hi):
    for c in range(c_lo, c_hi):
        g = _gen(w, kind, layer, seq, c)
        x = g.standard_normal((CHUNK, w.n_kv_heads, w.head_dim), dtype=np.float32)
        if gain is not None:
            x *= gain
        lo = max(t0, c * CHUNK)
        hi = min(t0 + n, (c + 1) * CHUNK)
        out[lo - t0: hi - t0] = x[lo - c * CHUNK: hi - c * CHUNK].astype(np.float16)


_POOL = None


def kv_tokens(w: Workload, layer: int, kind: str, t0: int, n: int, seq: int = 0) -> np.ndarray:
    """fp16 [n, n_kv_heads, head_dim] K or V of tokens t0 .. t0+n-1 of one sequence.
    Large ranges are drawn by a thread pool; the result does not depend on it (every
    CHUNK-token piece has its own generator key)."""
    global _POOL
    assert kind in ("K", "V")
    out = np.empty((n, w.n_kv_heads, w.head_dim), np.float16)
    if n == 0:
        return out
    gain = k_channel_gain(w, layer) if kind == "K" else None
    c_first, c_last = t0 // CHUNK, (t0 + n - 1) // CHUNK
    n_chunks = c_last - c_first + 1
    workers = min(16, os.cpu_count() or 1, max(1, n_chunks // 16))
    if workers <= 1:
        _fill_chunks(w, layer, kind, t0, n, seq, gain, out, c_first, c_last + 1)
        return out
    if _POOL is None:
        _POOL = concurrent.futures.ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1))
    bounds = np.linspace(c_first, c_last + 1, workers + 1).astype(int)
    futs = [_POOL.submit(_fill_chunks, w, layer, kind, t0, n, seq, gain, out, int(a), int(b))
            for a, b in zip(bounds[:-1], bounds[1:])]
    for f in futs:
        f.result()
    return out


def query(w: Workload, layer: int, step: int = 0, seq: int = 0) -> np.ndarray:
    """fp16 [n_q_heads, head_dim] query of one decode step."""
    g = _gen(w, "Q", layer, seq, step)
    return g.standard_normal((w.n_q_heads, w.head_dim), dtype=np.float32).astype(np.float16)


def seq_lens(w: Workload) -> np.ndarray:
    """int32 [n_seqs] context lengths (batched workload: uniform in len_range)."""
    if w.n_seqs == 1 or w.len_range == (0, 0):
        return np.full(w.n_seqs, w.ctx, np.int32)
    g = _gen(w, "lens")
    lo, hi = w.len_range
    return g.integers(lo, hi + 1, size=w.n_seqs).astype(np.int32)


def page_table(w: Workload, capacity_tokens: int) -> tuple[np.ndarray, int]:
    """int32 [n_seqs, max_pages] physical page ids (a seeded random permutation of all
    pages) and the pool size in pages.  Every sequence gets room for capacity_tokens."""
    pt = w.page_tokens
    max_pages = (capacity_tokens + pt - 1) // pt
    n_pages = w.n_seqs * max_pages
    perm = _gen(w, "pages").permutation(n_pages).astype(np.int32)
    return perm.reshape(w.n_seqs, max_pages), n_pages


def scaled(w: Workload, **changes) -> Workload:
    """A copy of a workload with some fields changed (smaller parity-test cases)."""
    return dataclasses.replace(w, **changes)
