"""tq_attn_decode_noalloc: attention without a caller-provided workspace.

Some callers cannot allocate device memory when they run attention (their pools are
reserved up front, or cudaMalloc is banned on their decode path), so they cannot pass
a workspace.  This entry point keeps its scratch in a fixed array inside the library.
The test calls it through the C ABI twice in a row, with different inputs, and checks
each result against tq_attn_decode with a workspace, within the attention tolerance of
the other parity tests.  The file name makes pytest collect it last.
"""
import ctypes

import numpy as np
import pytest

from rotated_bit_kv_tq_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ATTN_TOL = 2e-3


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
    for s, L in enumerate(lens):
        k = synth.kv_tokens(w, layer, "K", 0, L, s).reshape(L, -1)
        v = synth.kv_tokens(w, layer, "V", 0, L, s).reshape(L, -1)
        tq.encode(kc, torch.from_numpy(k).cuda(), seq_id=s)
        tq.encode(vc, torch.from_numpy(v).cuda(), seq_id=s)
    q = torch.from_numpy(np.stack([synth.query(w, layer, 0, s) for s in range(S)])).cuda()
    return kc, vc, q


def _noalloc(tq, kc, vc, q, lens_t, max_len, out):
    lib = tq.load()
    st = lib.tq_attn_decode_noalloc(ctypes.byref(kc.view), ctypes.byref(vc.view),
                                    ctypes.c_void_p(q.data_ptr()), q.shape[0], q.shape[1],
                                    ctypes.c_void_p(lens_t.data_ptr()), max_len, 0.0,
                                    ctypes.c_void_p(out.data_ptr()),
                                    ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, tq.load().tq_status_str(st)


def test_noalloc_matches_workspace_path_twice(tq):
    cases = [(synth.LLAMA3_8B_32K, 3, [3000], 2), (synth.HD256_128K, 2, [777, 1500, 64], 5)]
    for w, tt, lens, layer in cases:          # two calls in a row, different shapes/data
        kc, vc, q = _setup(tq, w, tt, lens, layer)
        S, Hq, D = q.shape
        lens_t = torch.tensor(lens, dtype=torch.int32, device="cuda")
        max_len = max(lens)
        ref = torch.empty(S, Hq, D, device="cuda")
        ws = torch.empty(tq.attn_workspace_bytes(S, Hq, D, max_len), dtype=torch.uint8, device="cuda")
        tq.attn_decode(kc, vc, q, lens_t, max_len, ref, ws)
        got = torch.full((S, Hq, D), float("nan"), device="cuda")
        _noalloc(tq, kc, vc, q, lens_t, max_len, got)
        torch.cuda.synchronize()
        assert tq.device_status() == 0
        r, g = ref.cpu().numpy().astype(np.float64), got.cpu().numpy().astype(np.float64)
        for s in range(S):
            err = np.linalg.norm(g[s] - r[s]) / np.linalg.norm(r[s])
            assert err < ATTN_TOL, (w.name, s, err)


def test_noalloc_rejects_oversized_shape(tq):
    """A shape whose partials exceed the fixed 8 MiB array is refused, not truncated."""
    S, Hkv, Hq, D, big = 512, 8, 128, 256, 1 << 20
    need = tq.attn_workspace_bytes(S, Hq, D, big)
    assert need > 8 << 20
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
