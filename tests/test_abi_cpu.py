"""The C-ABI library without a GPU: it builds, loads, exports every symbol that
include/tq.h declares, and its host-only entry points behave (no kernel launches)."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from rotated_bit_kv_tq_gb300 import build, _lib
    build.build()
    return _lib.load()


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "tq.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tq_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
    from rotated_bit_kv_tq_gb300._lib import SIGNATURES
    assert set(SIGNATURES) == set(names)


def test_sizes(lib):
    assert lib.tq_block_bytes(3) == 50 and lib.tq_block_bytes(2) == 34 and lib.tq_block_bytes(4) == 0
    assert lib.tq_row_bytes(3, 8, 128) == 400
    assert lib.tq_row_bytes(2, 4, 256) == 272
    assert lib.tq_row_bytes(3, 8, 100) == 0 and lib.tq_row_bytes(3, 0, 128) == 0


@pytest.mark.parametrize("bits", [2, 3])
def test_library_codebook_equals_oracle(lib, bits):
    """The library solves Lloyd-Max on its own (incomplete-beta masses, closed-form
    moments); its fp32 table must equal the oracle's quadrature solution bit for bit."""
    L = 1 << bits
    c = np.zeros(L, np.float32)
    t = np.zeros(L - 1, np.float32)
    assert lib.tq_codebook_get(bits, c.ctypes.data_as(ctypes.c_void_p), t.ctypes.data_as(ctypes.c_void_p)) == 0
    oc, ot = oracle.type_codebook(bits)
    assert np.array_equal(c.view(np.uint32), oc.view(np.uint32))
    assert np.array_equal(t.view(np.uint32), ot.view(np.uint32))


def test_host_validation_without_gpu(lib):
    from rotated_bit_kv_tq_gb300._lib import TqCache
    assert lib.tq_encode(None, None, 1, 256, None, None, 0, 0, None) == 1
    assert lib.tq_codebook_get(5, None, None) == 1
    bad = TqCache(3, 2, 100, 0, 16, 10, 1, 0, None, 0)   # head_dim not a multiple of 128
    assert lib.tq_encode(ctypes.byref(bad), None, 1, 256, None, None, 0, 0, None) == 2
    unaligned = TqCache(3, 2, 128, 0, 8, 10, 1, 0, None, 0)
    assert lib.tq_decode(ctypes.byref(unaligned), 0, 0, 1, None, None) == 1
    odd_pages = TqCache(3, 2, 128, 100, 16, 0, 1, 1, 16, 4)  # page_tokens % 32 != 0
    assert lib.tq_decode(ctypes.byref(odd_pages), 0, 0, 1, None, None) == 2
    assert lib.tq_status_str(4) == b"TQ_ERR_WORKSPACE_TOO_SMALL"
    assert lib.tq_status_str(99) == b"TQ_UNKNOWN_STATUS"
    assert lib.tq_device_status(None, None) == 1


def test_noalloc_scratch_size_matches_header():
    """The binding's NOALLOC_SCRATCH_BYTES is the header's TQ_NOALLOC_SCRATCH_BYTES."""
    from rotated_bit_kv_tq_gb300 import NOALLOC_SCRATCH_BYTES
    text = open(os.path.join(ROOT, "include", "tq.h")).read()
    m = re.search(r"#define\s+TQ_NOALLOC_SCRATCH_BYTES\s+\(\(size_t\)(\d+)\s*<<\s*(\d+)\)", text)
    assert m, "TQ_NOALLOC_SCRATCH_BYTES not found in tq.h"
    assert NOALLOC_SCRATCH_BYTES == int(m.group(1)) << int(m.group(2))


def test_inject_wait_timeout_arguments(lib):
    """Host-only: a negative count is refused; 0 cancels (no kernel is involved)."""
    assert lib.tq_inject_wait_timeout(-1) == 1
    assert lib.tq_inject_wait_timeout(0) == 0
