"""tq_attn_decode_noalloc: attention without a caller-provided workspace.

Some callers cannot allocate device memory when they run attention: their memory pools
are reserved up front, or cudaMalloc (which can synchronise the device) is banned on
their decode path, so they cannot pass a workspace.  This entry point keeps its scratch
in a fixed array inside the library (NOALLOC_SCRATCH_BYTES, the header's
TQ_NOALLOC_SCRATCH_BYTES).  The tests call it through the C ABI twice in a row, with
different shapes and data, and check each result against tq_attn_decode with a
workspace (the same kernels, so the same bits) and against the oracle within the
attention tolerance of the other parity tests, per (query, head) output vector.  A shape
whose partials come close to the limit must still work; one past it must be refused.
The file name makes pytest collect it last.
"""
import ctypes

import numpy as np
import pytest

import oracle
from rotated_bit_kv_tq_gb300 import NOALLOC_SCRATCH_BYTES, synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from attn_check import assert_attn_close  # noqa: E402


@pytest.fixture(scope="module")
def tq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import rotated_bit_kv_tq_gb300 as m
    from rotated_bit_kv_tq_gb300 import build
    build.build()
    torch.cuda.set_device(0)
    m.codebook_init(m.TQ_TURBO3, 0)
    m.codebook_init(m.TQ_TURBO2, 0)
    return m


def _setup(tq, w, tt, lens, layer):
    S, Hkv, D = len(lens), w.n_kv_heads, w.head_dim
    cap = max(lens)
    kc = tq.KVCache(tt, Hkv, D, n_seqs=S, capacity_tokens=cap)
    vc = tq.KVCache(tt, Hkv, D, n_seqs=S, capacity_tokens=cap)
    ks, vs = [], []
    for s, L in enumerate(lens):
        k = synth.kv_tokens(w, layer, "K", 0, L, s).reshape(L, -1)
        v = synth.kv_tokens(w, layer, "V", 0, L, s).reshape(L, -1)
        ks.append(k)
        vs.append(v)
        tq.encode(kc, torch.from_numpy(k).cuda(), seq_id=s)
        tq.encode(vc, torch.from_numpy(v).cuda(), seq_id=s)
    q16 = np.stack([synth.query(w, layer, 0, s) for s in range(S)])
    return kc, vc, ks, vs, q16


def _noalloc(tq, kc, vc, q, lens_t, max_len, out):
    lib = tq.load()
    return lib.tq_attn_decode_noalloc(ctypes.byref(kc.view), ctypes.byref(vc.view),
                                      ctypes.c_void_p(q.data_ptr()), q.shape[0], q.shape[1],
                                      ctypes.c_void_p(lens_t.data_ptr()), max_len, 0.0,
                                      ctypes.c_void_p(out.data_ptr()),
                                      ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _run_and_check(tq, w, tt, lens, layer, label):
    kc, vc, ks, vs, q16 = _setup(tq, w, tt, lens, layer)
    q = torch.from_numpy(q16).cuda()
    S, Hq, D = q.shape
    Hkv = w.n_kv_heads
    lens_t = torch.tensor(lens, dtype=torch.int32, device="cuda")
    max_len = max(lens)
    need = tq.attn_workspace_bytes(S, Hq, D, max_len)
    assert 0 < need <= NOALLOC_SCRATCH_BYTES
    ref = torch.empty(S, Hq, D, device="cuda")
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    tq.attn_decode(kc, vc, q, lens_t, max_len, ref, ws)
    got = torch.full((S, Hq, D), float("nan"), device="cuda")
    st = _noalloc(tq, kc, vc, q, lens_t, max_len, got)
    assert st == 0, tq.load().tq_status_str(st)
    torch.cuda.synchronize()
    assert tq.device_status() == 0
    # the same kernels with the same split plan: the same bits as the workspace path
    assert torch.equal(got, ref), label
    g = got.cpu().numpy().astype(np.float64)
    for s, L in enumerate(lens):
        kr = oracle.encode_rows(tt, ks[s], Hkv, D)
        vr = oracle.encode_rows(tt, vs[s], Hkv, D)
        o = oracle.attn_decode(tt, tt, kr, vr, q16[s], L, Hq, Hkv, D, 1.0 / np.sqrt(D))
        assert_attn_close(g[s], o, f"noalloc {label}#s{s}")
    return need


def test_noalloc_matches_workspace_path_and_oracle_twice(tq):
    """Two calls in a row with different shapes and data share the array."""
    _run_and_check(tq, synth.LLAMA3_8B_32K, 3, [3000], 2, "llama3-8b turbo3")
    _run_and_check(tq, synth.HD256_128K, 2, [777, 1500, 64], 5, "hd256 turbo2 batch 3")


def test_noalloc_shape_near_the_limit(tq):
    """A shape whose split partials fill more than 90 % of the array (found from this
    device's split plan through tq_attn_workspace_bytes)."""
    best = None
    for d in (128, 256):
        for g in range(1, 9):
            for n in range(1, 9):
                for L in (2500, 5000, 10000):
                    need = tq.attn_workspace_bytes(n, 8 * g, d, L)
                    if need <= NOALLOC_SCRATCH_BYTES and (best is None or need > best[0]):
                        best = (need, d, g, n, L)
    need, d, g, n, L = best
    assert need > 0.9 * NOALLOC_SCRATCH_BYTES, best
    w = synth.scaled(synth.TINY, n_kv_heads=8, n_q_heads=8 * g, head_dim=d)
    lens = [L - 7 * s for s in range(n)]
    got = _run_and_check(tq, w, 3, lens, 4, f"near limit D{d} G{g} S{n} L{L}")
    assert got == need


def test_noalloc_rejects_oversized_shape(tq):
    """A shape whose partials exceed the fixed array is refused, not truncated."""
    S, Hkv, Hq, D, big = 512, 8, 128, 256, 1 << 20
    need = tq.attn_workspace_bytes(S, Hq, D, big)
    assert need > NOALLOC_SCRATCH_BYTES
    kc = tq.KVCache(3, Hkv, D, n_seqs=S, capacity_tokens=16)
    q = torch.zeros(S, Hq, D, dtype=torch.float16, device="cuda")
    out = torch.zeros(S, Hq, D, device="cuda")
    lens_t = torch.full((S,), 16, dtype=torch.int32, device="cuda")
    lib = tq.load()
    st = lib.tq_attn_decode_noalloc(ctypes.byref(kc.view), ctypes.byref(kc.view),
                                    ctypes.c_void_p(q.data_ptr()), S, Hq,
                                    ctypes.c_void_p(lens_t.data_ptr()), big, 0.0,
                                    ctypes.c_void_p(out.data_ptr()), None)
    assert st == 4
    torch.cuda.synchronize()
    assert not out.any()
