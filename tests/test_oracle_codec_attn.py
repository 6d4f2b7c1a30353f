"""Pins of the oracle's encoder, decoder and attention (CPU only).

Brute force with a dense Hadamard matrix and a nearest-centroid search, closed forms
of the decoder, the round trip of codeword vectors, and closed forms of softmax
attention ("llama.cpp に TurboQuant を実装", sections "What TurboQuant does
differently" and "How small does it get"; kenji.blog section 8 for attention and
the TinyLLaMA article section 4.3 for GQA).
"""
import numpy as np
import pytest
import scipy.linalg

import oracle

H128 = scipy.linalg.hadamard(128).astype(np.float64)


def _f16_bits(x):
    return np.asarray(x, np.float32).astype(np.float16).view(np.uint16)


def _nearest(y, c):
    return np.argmin(np.abs(y[:, None] - c[None, :].astype(np.float64)), axis=1)


@pytest.mark.parametrize("bits", [2, 3])
def test_encode_matches_dense_bruteforce(bits):
    """Codes = nearest centroid of H x / (sqrt(128) |x|), computed with a dense Hadamard
    matrix in binary64; compared wherever the value is not within 1e-5 of a cell edge."""
    c, t = oracle.type_codebook(bits)
    rng = np.random.default_rng(11 + bits)
    checked = 0
    for trial in range(300):
        gain = np.exp(rng.standard_normal(128) * 0.5)
        if trial % 3 == 0:
            gain[rng.choice(128, 4, replace=False)] *= 10.0
        x16 = (rng.standard_normal(128) * gain * 10.0 ** rng.uniform(-3, 2)).astype(np.float16)
        blk = oracle.encode_block(bits, x16.view(np.uint16))
        codes, norm = oracle.unpack_block(bits, blk)
        x = x16.astype(np.float64)
        n = np.linalg.norm(x)
        y = H128 @ x / (np.sqrt(128.0) * n)
        want = _nearest(y, c)
        margin = np.min(np.abs(y[:, None] - t[None, :].astype(np.float64)), axis=1)
        ok = margin > 1e-5
        assert np.array_equal(codes[ok], want[ok]), trial
        checked += int(ok.sum())
        # the stored norm is |x| rounded to binary16 (skip values next to a rounding edge)
        n16 = np.float16(n)
        lo, hi = np.nextafter(n16, np.float16(0)), np.nextafter(n16, np.float16(np.inf))
        if min(n - (float(lo) + float(n16)) / 2, (float(hi) + float(n16)) / 2 - n) > 1e-6 * n:
            assert norm == int(n16.view(np.uint16))
    assert checked > 0.99 * 300 * 128


@pytest.mark.parametrize("bits", [2, 3])
def test_decode_uniform_codes_closed_form(bits):
    """All 128 codes equal j: W (c_j 1) = 128 c_j e_0, so x_hat = norm c_j sqrt(128) e_0.
    The block is built by hand (every field equal, so no bit order is assumed)."""
    c, _ = oracle.type_codebook(bits)
    for j in range(1 << bits):
        for norm in (1.0, 3.5, 1000.0):
            blk = np.zeros(oracle.block_bytes(bits), np.uint8)
            nb = int(np.float16(norm).view(np.uint16))
            blk[0], blk[1] = nb & 0xFF, nb >> 8
            blk[2:34] = (j & 3) * 0x55
            if bits == 3:
                blk[34:50] = 0xFF if j & 4 else 0
            x = oracle.decode_block(bits, blk)
            expect = np.zeros(128)
            expect[0] = norm * float(c[j]) * np.sqrt(128.0)
            assert np.allclose(x, expect, rtol=1e-12, atol=1e-12)


def _layout_block(bits, codes, norm_bits):
    """The documented layout, written out: value i -> low-plane word i//16, bits
    4k+2r, 4k+2r+1 (j=i%16, r=j//8, k=j%8); high-plane word i//32, bit 4k+p
    (j=i%32, p=j//8, k=j%8)."""
    blk = np.zeros(oracle.block_bytes(bits), np.uint8)
    blk[0], blk[1] = norm_bits & 0xFF, norm_bits >> 8
    low = np.zeros(8, np.uint32)
    high = np.zeros(4, np.uint32)
    for i, code in enumerate(codes):
        j = i % 16
        low[i // 16] |= np.uint32((int(code) & 3) << (4 * (j % 8) + 2 * (j // 8)))
        j = i % 32
        high[i // 32] |= np.uint32(((int(code) >> 2) & 1) << (4 * (j % 8) + j // 8))
    blk[2:34] = low.astype("<u4").view(np.uint8)
    if bits == 3:
        blk[34:50] = high.astype("<u4").view(np.uint8)
    return blk


@pytest.mark.parametrize("bits", [2, 3])
def test_layout_and_decode_random_codes(bits):
    """Hand-packed random codes: unpack returns them, and decode equals the dense
    formula norm / sqrt(128) * H c."""
    c, _ = oracle.type_codebook(bits)
    rng = np.random.default_rng(5)
    for _ in range(20):
        codes = rng.integers(0, 1 << bits, 128)
        norm16 = np.float16(rng.uniform(0.1, 300.0))
        blk = _layout_block(bits, codes, int(norm16.view(np.uint16)))
        got_codes, got_norm = oracle.unpack_block(bits, blk)
        assert np.array_equal(got_codes, codes) and got_norm == int(norm16.view(np.uint16))
        x = oracle.decode_block(bits, blk)
        expect = float(norm16) / np.sqrt(128.0) * (H128 @ c[codes].astype(np.float64))
        assert np.allclose(x, expect, rtol=1e-12, atol=1e-12)
        # the encoder writes the same layout: re-encode a vector far from every edge
        assert np.array_equal(oracle.encode_block(bits, _f16_bits(x)).shape, blk.shape)


@pytest.mark.parametrize("bits", [2, 3])
def test_codeword_round_trip(bits):
    """Quantising a random unit vector gives codes q; the codeword vector c[q],
    rotated back and scaled, is re-encoded to the same codes wherever c[q]/|c[q]| sits
    clearly inside its cell (a codeword vector is not unit-norm, so cells can change)."""
    c, t = oracle.type_codebook(bits)
    c64 = c.astype(np.float64)
    rng = np.random.default_rng(17)
    exact = 0
    for _ in range(200):
        u = rng.standard_normal(128)
        u /= np.linalg.norm(u)
        q = _nearest(u, c)
        w = c64[q]
        x = H128 @ w / np.sqrt(128.0) * (40.0 / np.linalg.norm(w))
        x16 = x.astype(np.float16)
        codes, _ = oracle.unpack_block(bits, oracle.encode_block(bits, x16.view(np.uint16)))
        y = H128 @ x16.astype(np.float64) / (np.sqrt(128.0) * np.linalg.norm(x16.astype(np.float64)))
        want = _nearest(y, c)
        margin = np.min(np.abs(y[:, None] - t[None, :].astype(np.float64)), axis=1)
        ok = margin > 1e-4
        assert np.array_equal(codes[ok], want[ok])
        inside = np.min(np.abs((w / np.linalg.norm(w))[:, None] - t[None, :]), axis=1) > 2e-3
        assert np.array_equal(codes[inside], q[inside])
        exact += int(np.array_equal(codes, q))
    assert exact > 0


@pytest.mark.parametrize("bits,lo,hi", [(3, 0.025, 0.045), (2, 0.09, 0.14)])
def test_quantisation_error_level(bits, lo, hi):
    """decode(encode(x)) keeps |x - x_hat|^2 / |x|^2 near the Lloyd-Max distortion."""
    rng = np.random.default_rng(23)
    x16 = (rng.standard_normal((400, 128)) * np.exp(0.5 * rng.standard_normal(128))).astype(np.float16)
    rows = oracle.encode_rows(bits, x16, n_kv_heads=1, head_dim=128)
    xh = oracle.decode_rows(bits, rows, n_kv_heads=1, head_dim=128)[:, 0, :]
    x = x16.astype(np.float64)
    err = np.sum((x - xh) ** 2) / np.sum(x * x)
    assert lo < err < hi


def test_zero_and_spike_blocks():
    for bits in (2, 3):
        blk = oracle.encode_block(bits, np.zeros(128, np.uint16))
        codes, norm = oracle.unpack_block(bits, blk)
        assert norm == 0 and np.all(codes == (1 << bits) // 2)   # y = +0 -> first positive cell
        assert np.all(oracle.decode_block(bits, blk) == 0.0)
        # a spike: H e_i / sqrt(128) has every coordinate at +-1/sqrt(128) = +-0.0884
        for i in (0, 77):
            x = np.zeros(128, np.float32)
            x[i] = 3.0
            codes, norm = oracle.unpack_block(bits, oracle.encode_block(bits, _f16_bits(x)))
            assert norm == int(np.float16(3.0).view(np.uint16))
            s = H128[:, i]
            c, _ = oracle.type_codebook(bits)
            assert np.array_equal(codes, _nearest(s / np.sqrt(128.0), c))


def test_norm_saturates_to_fp16_max():
    x = np.full(128, 60000.0, np.float16)            # |x| = 678,823 > 65504
    _, norm = oracle.unpack_block(3, oracle.encode_block(3, x.view(np.uint16)))
    assert norm == int(np.float16(65504.0).view(np.uint16))


def test_encode_rows_stride_and_heads():
    rng = np.random.default_rng(2)
    src = rng.standard_normal((5, 3 * 256 + 64)).astype(np.float16)   # padded token stride
    rows = oracle.encode_rows(3, src, n_kv_heads=3, head_dim=256, src_stride=3 * 256 + 64)
    assert rows.shape == (5, 3 * 2 * 50)
    for tkn in range(5):
        for h in range(3):
            for b in range(2):
                blk = oracle.encode_block(3, src[tkn, h * 256 + b * 128: h * 256 + b * 128 + 128].view(np.uint16))
                off = (h * 2 + b) * 50
                assert np.array_equal(rows[tkn, off:off + 50], blk)


# ------------------------------------------------------------------ attention

def test_attention_single_token_returns_v():
    rng = np.random.default_rng(0)
    q, k, v = rng.standard_normal((4, 128)), rng.standard_normal((1, 2, 128)), rng.standard_normal((1, 2, 128))
    out = oracle.dense_attention(q, k, v, n_kv_heads=2, scale=1 / np.sqrt(128))
    assert np.allclose(out, np.repeat(v[0], 2, axis=0), rtol=0, atol=1e-14)


def test_attention_equal_keys_average_values():
    rng = np.random.default_rng(1)
    q = rng.standard_normal((2, 128))
    k = np.repeat(rng.standard_normal((1, 1, 128)), 37, axis=0)
    v = rng.standard_normal((37, 1, 128))
    out = oracle.dense_attention(q, k, v, n_kv_heads=1, scale=0.3)
    assert np.allclose(out, np.repeat(v.mean(axis=0), 2, axis=0), atol=1e-13)


def test_attention_two_tokens_closed_form():
    q = np.zeros((1, 128)); q[0, 0] = 2.0
    k = np.zeros((2, 1, 128)); k[0, 0, 0] = 1.0; k[1, 0, 0] = -0.5
    v = np.zeros((2, 1, 128)); v[0, 0, 3] = 1.0; v[1, 0, 3] = 5.0
    scale = 0.7
    s0, s1 = 2.0 * 1.0 * scale, 2.0 * -0.5 * scale
    w0 = np.exp(s0) / (np.exp(s0) + np.exp(s1))
    out = oracle.dense_attention(q, k, v, n_kv_heads=1, scale=scale)
    assert abs(out[0, 3] - (w0 * 1.0 + (1 - w0) * 5.0)) < 1e-14
    # huge scores do not overflow (the row maximum is subtracted)
    out = oracle.dense_attention(q * 1e4, k, v, n_kv_heads=1, scale=scale)
    assert abs(out[0, 3] - 1.0) < 1e-14


def test_attention_gqa_head_mapping():
    """Query head h reads KV head floor(h / G) (kenji.blog TinyLLaMA 4.3: K/V are
    broadcast to the query-head count)."""
    rng = np.random.default_rng(4)
    hq, hkv, T = 8, 2, 9
    q = rng.standard_normal((hq, 128))
    k = rng.standard_normal((T, hkv, 128))
    v = np.zeros((T, hkv, 128))
    v[:, 0, :] = 1.0
    v[:, 1, :] = -2.0
    out = oracle.dense_attention(q, k, v, n_kv_heads=hkv, scale=0.1)
    assert np.allclose(out[:4], 1.0) and np.allclose(out[4:], -2.0)


def test_attn_decode_rotated_domain_identity():
    """q . x_hat computed in the original domain equals (H q / sqrt(128)) . (norm * c),
    the rotated-domain form a fused kernel uses: H is symmetric and H H = 128 I."""
    rng = np.random.default_rng(9)
    for bits in (2, 3):
        c, _ = oracle.type_codebook(bits)
        x16 = rng.standard_normal(128).astype(np.float16)
        blk = oracle.encode_block(bits, x16.view(np.uint16))
        codes, nb = oracle.unpack_block(bits, blk)
        q = rng.standard_normal(128)
        lhs = q @ oracle.decode_block(bits, blk)
        rhs = (H128 @ q / np.sqrt(128.0)) @ (float(np.uint16(nb).view(np.float16)) * c[codes].astype(np.float64))
        assert abs(lhs - rhs) < 1e-12 * max(1.0, abs(lhs))


def test_attn_decode_single_token_is_decoded_v():
    rng = np.random.default_rng(12)
    k16 = rng.standard_normal((1, 2, 128)).astype(np.float16)
    v16 = rng.standard_normal((1, 2, 128)).astype(np.float16)
    q16 = rng.standard_normal((4, 128)).astype(np.float16)
    kr = oracle.encode_rows(3, k16.reshape(1, -1), 2, 128)
    vr = oracle.encode_rows(2, v16.reshape(1, -1), 2, 128)
    out = oracle.attn_decode(3, 2, kr, vr, q16, 1, 4, 2, 128, 1 / np.sqrt(128))
    vhat = oracle.decode_rows(2, vr, 2, 128)[0]
    assert np.allclose(out, np.repeat(vhat, 2, axis=0), atol=1e-14)
    # zero tokens: the output is zero by convention (nothing to attend to)
    out0 = oracle.attn_decode(3, 3, kr[:0], kr[:0], q16, 0, 4, 2, 128, 0.1)
    assert np.all(out0 == 0.0)
