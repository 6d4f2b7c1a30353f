"""Pins of the prompt-chunk (prefill) attention oracle.

Query j of a chunk sits at position pos0 + j and attends to rows 0 .. pos0 + j: the
KV-cache rule of the TinyLLaMA article, section 7 (position N writes row N and attends to
the view of rows 0..N), applied at every position of the chunk.  The pins are
- a single query reduces to the decode-step oracle, itself pinned by closed forms in
  test_oracle_codec_attn.py;
- causality: rows after a query's position never change its output, while the rows up
  to it do;
- equal keys give the plain mean of the dequantised values of the query's prefix
  (an off-by-one in the prefix length changes that mean).
"""
import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _case(seed, n_rows, hkv, d, tk=3, tv=3):
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((n_rows, hkv * d)).astype(np.float16)
    v = rng.standard_normal((n_rows, hkv * d)).astype(np.float16)
    return oracle.encode_rows(tk, k, hkv, d), oracle.encode_rows(tv, v, hkv, d)


@pytest.mark.parametrize("pos0", [0, 5, 40])
def test_single_query_is_the_decode_step(pos0):
    hkv, hq, d = 2, 8, 128
    kr, vr = _case(1, pos0 + 1, hkv, d)
    q = np.random.default_rng(2).standard_normal((1, hq, d)).astype(np.float16)
    scale = 1 / np.sqrt(d)
    got = oracle.attn_prefill(3, 3, kr, vr, q, pos0, hkv, d, scale)
    ref = oracle.attn_decode(3, 3, kr, vr, q[0], pos0 + 1, hq, hkv, d, scale)
    assert np.array_equal(got[0], ref)


def test_every_query_is_the_decode_step_at_its_position():
    hkv, hq, d, pos0, nq = 2, 4, 256, 7, 6
    kr, vr = _case(3, pos0 + nq, hkv, d, tk=2, tv=3)
    q = np.random.default_rng(4).standard_normal((nq, hq, d)).astype(np.float16)
    got = oracle.attn_prefill(2, 3, kr, vr, q, pos0, hkv, d, 0.0625)
    for j in range(nq):
        ref = oracle.attn_decode(2, 3, kr, vr, q[j], pos0 + j + 1, hq, hkv, d, 0.0625)
        assert np.array_equal(got[j], ref)


def test_causality():
    hkv, hq, d, pos0, nq = 1, 2, 128, 3, 5
    kr, vr = _case(5, pos0 + nq, hkv, d)
    q = np.random.default_rng(6).standard_normal((nq, hq, d)).astype(np.float16)
    base = oracle.attn_prefill(3, 3, kr, vr, q, pos0, hkv, d, 0.1)
    # replace the rows of positions pos0 + 2 onwards with other data
    k2, v2 = _case(7, pos0 + nq, hkv, d)
    kr2, vr2 = kr.copy(), vr.copy()
    kr2[pos0 + 2:], vr2[pos0 + 2:] = k2[pos0 + 2:], v2[pos0 + 2:]
    other = oracle.attn_prefill(3, 3, kr2, vr2, q, pos0, hkv, d, 0.1)
    assert np.array_equal(base[:2], other[:2])            # queries at pos0, pos0 + 1
    for j in range(2, nq):                                 # the later ones see the change
        assert not np.allclose(base[j], other[j])


def test_equal_keys_average_the_prefix_values():
    hkv, hq, d, pos0, nq = 1, 3, 128, 4, 4
    rng = np.random.default_rng(8)
    krow = rng.standard_normal((1, hkv * d)).astype(np.float16)
    k = np.repeat(krow, pos0 + nq, axis=0)
    v = rng.standard_normal((pos0 + nq, hkv * d)).astype(np.float16)
    kr, vr = oracle.encode_rows(3, k, hkv, d), oracle.encode_rows(3, v, hkv, d)
    q = rng.standard_normal((nq, hq, d)).astype(np.float16)
    got = oracle.attn_prefill(3, 3, kr, vr, q, pos0, hkv, d, 0.2)
    vh = oracle.decode_rows(3, vr, hkv, d).reshape(pos0 + nq, d)
    for j in range(nq):
        mean = vh[: pos0 + j + 1].mean(axis=0)
        for h in range(hq):
            np.testing.assert_allclose(got[j, h], mean, rtol=1e-12, atol=1e-12)
