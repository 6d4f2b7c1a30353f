"""Pins of the oracle against what the pages and mathematics fix (CPU only).

Each test checks one oracle function against something other than the oracle itself:
numbers printed on the pages, closed forms, textbook special cases, scipy quadrature,
dense matrices, or brute force on tiny inputs.  A plausible slip anywhere in the oracle
(a dropped term, a wrong sign or index, a transposed layout) fails at least one of them.
"""
import os

import numpy as np
import pytest
import scipy.integrate
import scipy.linalg

import oracle

INV_SQRT128_F32 = np.float32(1.0 / np.sqrt(128.0))


def _read_rows(path):
    rows = []
    for line in open(path):
        line = line.strip()
        if line and not line.startswith("#"):
            rows.append(line.split())
    return rows


# ------------------------------------------------------------------ sizes (pages)

def test_block_bytes_match_pages(golden_dir):
    """"How small does it get": 128 values + one FP16 norm = 0.39 / 0.27 B per value."""
    for name, bits, bpv, frac in _read_rows(os.path.join(golden_dir, "block_bytes.txt")):
        t = int(bits)
        nbytes = oracle.block_bytes(t)
        assert nbytes == 2 + 128 * t // 8
        assert round(nbytes / 128, 2) == float(bpv)
        assert int(2.0 / (nbytes / 128)) == int(frac)   # about 1/5, 1/7 of FP16 (5.12x, 7.53x)
    assert oracle.block_bytes(4) == 0


def test_kv_size_formula(golden_dir):
    """"Why the KV cache is so heavy": layers x heads x head_dim x ctx x 2 x bytes."""
    for row in _read_rows(os.path.join(golden_dir, "kv_size_14b.txt")):
        L, H, D, C, num, den, nbytes, mib = map(int, row)
        got = oracle.kv_bytes(L, H, D, C, num, den)
        assert got == nbytes
        assert got == mib * 2 ** 20


# ------------------------------------------------------------------ binary16

def test_f16_to_f32_exhaustive():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float32)
    got = np.array([oracle.f16_to_f32(int(b)) for b in bits], np.float32)
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin].view(np.uint32), ref[fin].view(np.uint32))
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(np.isinf(got), np.isinf(ref))


def test_f32_to_f16_rne_sweep():
    rng = np.random.default_rng(1)
    # random magnitudes across the whole binary16 range plus exact halfway cases
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(10.0) ** rng.integers(-9, 5, 20000),
        (np.arange(2048, dtype=np.float32) + np.float32(0.5)) * np.float32(2.0 ** -24),  # subnormal ties
        np.float32([0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e30, -1e30, 6.1e-5, 5.96e-8, 2.98e-8,
                    2.99e-8, 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11]),
    ]).astype(np.float32)
    ref = x.astype(np.float16).view(np.uint16)
    got = np.array([oracle.f32_to_f16(float(v)) for v in x], np.uint16)
    assert np.array_equal(got, ref)


# ------------------------------------------------------------------ FWHT

@pytest.mark.parametrize("n", [2, 4, 8, 16, 32, 64, 128])
def test_fwht_equals_dense_sylvester(n):
    """"What TurboQuant does differently": the FWHT is the Hadamard transform done with
    adds and subtracts only.  Integer inputs make both sides exact."""
    H = scipy.linalg.hadamard(n).astype(np.float64)   # Sylvester construction
    rng = np.random.default_rng(n)
    for _ in range(5):
        x = rng.integers(-1000, 1000, n).astype(np.float64)
        assert np.array_equal(oracle.fwht_f32(x.astype(np.float32)).astype(np.float64), H @ x)
        assert np.array_equal(oracle.fwht_f64(x), H @ x)


def test_fwht_self_inverse_and_spikes():
    rng = np.random.default_rng(7)
    x = rng.integers(-50, 50, 128).astype(np.float64)
    assert np.array_equal(oracle.fwht_f64(oracle.fwht_f64(x)), 128 * x)   # W W = 128 I
    for i in (0, 1, 37, 127):
        e = np.zeros(128)
        e[i] = 1.0
        y = oracle.fwht_f64(e)
        assert np.all(np.abs(y) == 1.0)                                   # +-1 row
        assert np.array_equal(y / np.sqrt(128), scipy.linalg.hadamard(128)[:, i] / np.sqrt(128))


# ------------------------------------------------------------------ codebook

def test_codebook_d3_is_uniform_quantiser():
    """For d = 3 one coordinate of a uniform unit vector is uniform on [-1, 1]
    (Archimedes), and the Lloyd-Max quantiser of a uniform law is the uniform one."""
    for L in (4, 8):
        c64, _, _, _ = oracle.codebook(3, L)
        expect = -1.0 + (2.0 * np.arange(L) + 1.0) / L
        assert np.max(np.abs(c64 - expect)) < 1e-11


@pytest.mark.parametrize("bits", [2, 3])
def test_codebook_symmetric(bits):
    c, t = oracle.type_codebook(bits)
    L = 1 << bits
    assert np.array_equal(c, -c[::-1])
    assert np.array_equal(t, -t[::-1])
    assert t[L // 2 - 1] == 0.0
    assert np.all(np.diff(c) > 0)
    # thresholds are binary32 midpoints of the binary32 centroids
    assert np.array_equal(t, ((c[:-1] + c[1:]) * np.float32(0.5)).astype(np.float32))


def _density(d):
    a = (d - 3) / 2.0
    return lambda y: (1.0 - y * y) ** a


@pytest.mark.parametrize("bits", [2, 3])
def test_codebook_lloyd_conditions_scipy(bits):
    """Centroid condition c_j = E[Y | Y in cell j] for the d = 128 coordinate law,
    re-integrated with scipy's adaptive quadrature (QUADPACK), and the midpoint
    condition for the cell boundaries."""
    d, L = 128, 1 << bits
    c64, _, _, _ = oracle.codebook(d, L)
    f = _density(d)
    edges = np.concatenate([[-1.0], 0.5 * (c64[:-1] + c64[1:]), [1.0]])
    for j in range(L):
        m0 = scipy.integrate.quad(f, edges[j], edges[j + 1], epsabs=0, epsrel=1e-13, limit=200)[0]
        m1 = scipy.integrate.quad(lambda y: y * f(y), edges[j], edges[j + 1], epsabs=0,
                                  epsrel=1e-13, limit=200)[0]
        assert abs(m1 / m0 - c64[j]) <= 1e-10 * abs(c64[j])


def test_codebook_gaussian_limit(golden_dir):
    """As d grows, sqrt(d) * Y tends to N(0, 1), so sqrt(d) * c tends to the Gaussian
    Lloyd-Max levels tabulated by Max (1960)."""
    for row in _read_rows(os.path.join(golden_dir, "max1960_gaussian_levels.txt")):
        L = int(row[0])
        pos = np.array(list(map(float, row[1:])))
        c64, _, _, _ = oracle.codebook(200003, L)
        got = np.sqrt(200003.0) * c64[L // 2:]
        assert np.max(np.abs(got - pos)) < 2e-3
        c128, _, _, _ = oracle.codebook(128, L)
        got = np.sqrt(128.0) * c128[L // 2:]
        assert np.max(np.abs(got - pos) / pos) < 0.03   # d = 128 is already close


@pytest.mark.parametrize("bits", [2, 3])
def test_codebook_mse_matches_monte_carlo(bits):
    """Uniform unit vectors (normalised Gaussians) quantised coordinate-wise with the
    codebook: the empirical MSE matches the analytic MSE of the d = 128 law."""
    d, L = 128, 1 << bits
    c64, c32, t32, _ = oracle.codebook(d, L)
    f = _density(d)
    z = scipy.integrate.quad(f, -1, 1, epsabs=0, epsrel=1e-13)[0]
    edges = np.concatenate([[-1.0], 0.5 * (c64[:-1] + c64[1:]), [1.0]])
    mse = sum(scipy.integrate.quad(lambda y, cj=c64[j]: (y - cj) ** 2 * f(y), edges[j], edges[j + 1],
                                   epsabs=0, epsrel=1e-12)[0] for j in range(L)) / z
    rng = np.random.default_rng(3)
    u = rng.standard_normal((20000, d))
    u /= np.linalg.norm(u, axis=1, keepdims=True)
    idx = np.searchsorted(t32.astype(np.float64), u.ravel(), side="left")
    emp = np.mean((u.ravel() - c32.astype(np.float64)[idx]) ** 2)
    assert abs(emp - mse) < 0.01 * mse
    # and the normalised distortion per 128-block sits where Lloyd-Max puts it
    assert 0.02 < d * mse < 0.05 if bits == 3 else 0.09 < d * mse < 0.14
