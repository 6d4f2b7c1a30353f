"""Attention tolerance of the GPU parity tests.

The bar is 2e-3 relative L2 against the oracle's fp64 attention over the same packed
cache, applied to every single (query token, query head) output vector of head_dim
values and, as well, to a whole output.  Every check records its largest per-head error
under a label; the session prints the records at the end (tests/conftest.py).
"""
import numpy as np

ATTN_TOL = 2e-3

RECORDS = []   # (label, largest per-head error, whole-output error)


def attn_rel_errors(got, ref):
    """Relative L2 errors of every output vector along the last axis, and of the whole."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    per = np.linalg.norm(got - ref, axis=-1) / np.linalg.norm(ref, axis=-1)
    whole = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    return per, whole


def assert_attn_close(got, ref, label="", tol=ATTN_TOL):
    """got / ref: [..., n_q_heads, head_dim] attention outputs; every head vector and the
    whole must be within tol.  Returns the largest per-head error."""
    per, whole = attn_rel_errors(got, ref)
    worst = float(per.max())
    RECORDS.append((label, worst, float(whole)))
    at = np.unravel_index(int(np.argmax(per)), per.shape)
    assert worst < tol and whole < tol, (
        f"{label}: per-head max {worst:.3e} at {tuple(int(i) for i in at)}, whole {whole:.3e}")
    return worst
