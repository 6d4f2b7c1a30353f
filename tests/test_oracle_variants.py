"""Pins of the oracle's quality variants (random-sign Hadamard W D, norm correction).

- Random signs: the rotation becomes W D, so encoding x with sign mask s is the plain
  encoding of D x, bit for bit, and decoding is D times the plain decode.  A constant
  block is the plain FWHT's worst case (W 1 is a single spike, which one 3-bit code cannot
  hold); D spreads it, which is the point of the random signs ("llama.cpp に TurboQuant を
  実装", "What TurboQuant does differently").
- Norm correction: the codes are unchanged and the decoded block has the input's norm up
  to the fp16 rounding of the stored value.
"""
import numpy as np
import pytest

import oracle


def _f16_block(rng, scale=1.0):
    return (rng.standard_normal(128) * scale).astype(np.float16)


def _mask(rng):
    return rng.integers(0, 2, 128)


@pytest.mark.parametrize("bits", [2, 3])
def test_signs_are_a_flip_of_the_input(bits):
    rng = np.random.default_rng(10 + bits)
    for _ in range(20):
        x = _f16_block(rng, 3.0)
        s = _mask(rng)
        var = oracle.variant(signs=s)
        got = oracle.encode_block(bits, x.view(np.uint16), var)
        flipped = np.where(s == 1, -x, x).astype(np.float16)
        assert np.array_equal(got, oracle.encode_block(bits, flipped.view(np.uint16)))
        dec = oracle.decode_block(bits, got, var)
        plain = oracle.decode_block(bits, got)
        assert np.array_equal(dec, np.where(s == 1, -plain, plain))


def test_zero_mask_is_the_plain_method():
    rng = np.random.default_rng(3)
    x = _f16_block(rng)
    var = oracle.variant(signs=np.zeros(128, int))
    assert np.array_equal(oracle.encode_block(3, x.view(np.uint16), var),
                          oracle.encode_block(3, x.view(np.uint16)))


def test_mask_bit_order():
    """Bit i of the mask (word i // 32, bit i % 32) belongs to coordinate i."""
    rng = np.random.default_rng(4)
    x = _f16_block(rng, 2.0)
    for i in (0, 1, 31, 32, 63, 64, 95, 96, 127):
        flipped = x.copy()
        flipped[i] = -flipped[i]
        got = oracle.encode_block(3, x.view(np.uint16), oracle.variant(signs=1 << i))
        assert np.array_equal(got, oracle.encode_block(3, flipped.view(np.uint16))), i


@pytest.mark.parametrize("bits", [2, 3])
def test_random_signs_rescue_a_constant_block(bits):
    x = np.full(128, 0.5, np.float16)
    plain = oracle.decode_block(bits, oracle.encode_block(bits, x.view(np.uint16)))
    err_plain = np.linalg.norm(plain - x) / np.linalg.norm(x)
    rng = np.random.default_rng(5)
    errs = []
    for _ in range(8):
        var = oracle.variant(signs=_mask(rng))
        dec = oracle.decode_block(bits, oracle.encode_block(bits, x.view(np.uint16), var), var)
        errs.append(np.linalg.norm(dec - x) / np.linalg.norm(x))
    # plain: W 1 = 128 e_0, the unit vector (1, 0, ..., 0) keeps only the top centroid
    assert err_plain > 0.75
    # signed: an ordinary spread block, near the quantiser's normalised RMS error
    assert max(errs) < (0.30 if bits == 3 else 0.45)


@pytest.mark.parametrize("bits", [2, 3])
def test_norm_correction_keeps_codes_and_restores_the_norm(bits):
    rng = np.random.default_rng(20 + bits)
    var = oracle.variant(norm_correction=True)
    for _ in range(30):
        x = _f16_block(rng, float(rng.uniform(0.1, 30)))
        blk = oracle.encode_block(bits, x.view(np.uint16), var)
        plain = oracle.encode_block(bits, x.view(np.uint16))
        c1, n1 = oracle.unpack_block(bits, blk)
        c0, n0 = oracle.unpack_block(bits, plain)
        assert np.array_equal(c1, c0)
        nx = np.linalg.norm(x.astype(np.float64))
        nd = np.linalg.norm(oracle.decode_block(bits, blk, var))
        assert abs(nd / nx - 1) < 2.0 ** -10          # fp16 rounding of the stored value


def test_variant_attention_uses_the_variant_decode():
    """Attention over a cache encoded with a variant equals dense attention over the rows
    dequantised with that variant."""
    rng = np.random.default_rng(7)
    hkv, hq, d, n = 1, 2, 128, 9
    k = rng.standard_normal((n, d)).astype(np.float16)
    v = rng.standard_normal((n, d)).astype(np.float16)
    vk, vv = oracle.variant(signs=_mask(rng)), oracle.variant(signs=_mask(rng), norm_correction=True)
    kr, vr = oracle.encode_rows(3, k, hkv, d, var=vk), oracle.encode_rows(2, v, hkv, d, var=vv)
    q = rng.standard_normal((hq, d)).astype(np.float16)
    got = oracle.attn_decode(3, 2, kr, vr, q, n, hq, hkv, d, 0.1, var_k=vk, var_v=vv)
    ref = oracle.dense_attention(q.astype(np.float64), oracle.decode_rows(3, kr, hkv, d, var=vk),
                                 oracle.decode_rows(2, vr, hkv, d, var=vv), hkv, 0.1)
    assert np.array_equal(got, ref)
