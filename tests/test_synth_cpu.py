"""The seeded synthetic inputs follow their stated recipe.

The pages measure on real models (Qwen2.5-Coder-14B and a head_dim-256 9B model,
"llama.cpp に TurboQuant を実装", "Numbers on real models"); these draws stand in for them, so
the tests check the recipe the generator states: the five workload shapes; V and q ~ N(0, 1);
K with a lognormal(0, 0.5) gain per (layer, KV head, channel) and outlier_gain on n_outliers
channels per (layer, KV head); fp16 values; batched lengths uniform in [1024, 16384]; pages a
permutation of the pool; any token range regenerates to the same values.
"""
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from rotated_bit_kv_tq_gb300 import synth  # noqa: E402


def test_workload_shapes():
    t, l, q, h, b = synth.WORKLOADS
    assert (t.layers, t.n_kv_heads, t.n_q_heads, t.head_dim, t.ctx, t.types) == (1, 2, 8, 128, 256, (3,))
    assert (l.layers, l.n_kv_heads, l.n_q_heads, l.head_dim, l.ctx, l.types, l.decode_steps) == \
        (32, 8, 32, 128, 32768, (3,), 128)
    assert (q.layers, q.n_kv_heads, q.n_q_heads, q.head_dim, q.ctx, q.types) == (48, 8, 40, 128, 32768, (3, 2))
    assert (h.layers, h.n_kv_heads, h.n_q_heads, h.head_dim, h.ctx, h.types) == (32, 4, 16, 256, 131072, (2,))
    assert (h.n_outliers, h.outlier_gain) == (8, 20.0)
    assert (b.n_seqs, b.layers, b.n_kv_heads, b.n_q_heads, b.head_dim, b.page_tokens, b.len_range) == \
        (64, 32, 8, 32, 128, 256, (1024, 16384))
    assert all(w.n_outliers == 4 and w.outlier_gain == 10.0 for w in (t, l, q, b))


def test_v_and_q_standard_normal_fp16():
    w = synth.LLAMA3_8B_32K
    v = synth.kv_tokens(w, 3, "V", 0, 4096)
    assert v.dtype == np.float16 and v.shape == (4096, 8, 128)
    x = v.astype(np.float64)
    assert abs(x.mean()) < 0.005 and abs(x.std() - 1.0) < 0.005
    qs = np.stack([synth.query(w, 3, s) for s in range(64)]).astype(np.float64)
    assert qs.shape == (64, 32, 128)
    assert abs(qs.mean()) < 0.02 and abs(qs.std() - 1.0) < 0.02


@pytest.mark.parametrize("w", [synth.LLAMA3_8B_32K, synth.HD256_128K], ids=lambda w: w.name)
def test_k_channel_gains(w):
    layer = 2
    gain = synth.k_channel_gain(w, layer)
    assert gain.shape == (w.n_kv_heads, w.head_dim)
    k = synth.kv_tokens(w, layer, "K", 0, 8192).astype(np.float64)
    std = k.std(axis=0)                                  # per (head, channel)
    assert np.allclose(std, gain, rtol=0.05)             # K = N(0, 1) x gain
    # the same draws with the outlier factor set to 1 give the lognormal part alone: the
    # ratio is outlier_gain on exactly n_outliers channels of every head and 1 elsewhere
    base = synth.k_channel_gain(synth.scaled(w, outlier_gain=1.0), layer)
    ratio = gain / base
    assert np.all(np.isclose(ratio, 1.0) | np.isclose(ratio, w.outlier_gain))
    assert np.all(np.isclose(ratio, w.outlier_gain).sum(axis=1) == w.n_outliers)
    # and log(base) ~ N(0, 0.5^2)
    lb = np.log(base.astype(np.float64)).ravel()
    assert abs(lb.mean()) < 0.1 and 0.4 < lb.std() < 0.6


def test_any_token_range_regenerates():
    w = synth.QWEN25_14B_32K
    full = synth.kv_tokens(w, 5, "K", 0, 700, seq=0)
    assert np.array_equal(synth.kv_tokens(w, 5, "K", 123, 400), full[123:523])
    assert np.array_equal(synth.kv_tokens(w, 5, "K", 699, 1), full[699:])
    assert not np.array_equal(synth.kv_tokens(w, 6, "K", 0, 64), full[:64])   # layers differ
    assert not np.array_equal(synth.kv_tokens(w, 5, "V", 0, 64), full[:64])   # K and V differ


def test_batched_lengths_and_pages():
    w = synth.BATCHED_PAGED
    lens = synth.seq_lens(w)
    assert lens.shape == (64,) and lens.dtype == np.int32
    assert lens.min() >= 1024 and lens.max() <= 16384
    assert np.array_equal(lens, synth.seq_lens(w))
    assert len(np.unique(lens)) > 50
    pt, n_pages = synth.page_table(w, 16384)
    assert pt.shape == (64, 64) and n_pages == 64 * 64
    assert np.array_equal(np.sort(pt.ravel()), np.arange(n_pages))
    assert np.array_equal(synth.seq_lens(synth.LLAMA3_8B_32K), [32768])
