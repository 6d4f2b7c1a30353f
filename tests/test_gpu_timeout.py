"""Failure detection of the bounded device waits, without a GPU fault.

tq_inject_wait_timeout makes the next decode-attention launch request no tile copies and
gives every tile wait a limit of 64 polls.  No copy is in flight, so each wait simply runs
out: the kernel must record TQ_ERR_DEVICE_TIMEOUT (6), write empty partials (a zero
output) and return normally, leaving the context usable; the next call is clean and
matches the oracle.
"""
import numpy as np
import pytest

import oracle
from rotated_bit_kv_tq_gb300 import synth

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
    return m


@pytest.mark.parametrize("append", [False, True])
def test_injected_wait_timeout_is_reported_and_recovers(tq, append):
    w = synth.LLAMA3_8B_32K
    n, Hkv, Hq, D = 2000, w.n_kv_heads, w.n_q_heads, w.head_dim
    k = synth.kv_tokens(w, 6, "K", 0, n).reshape(n, -1)
    v = synth.kv_tokens(w, 6, "V", 0, n).reshape(n, -1)
    kc = tq.KVCache(3, Hkv, D, capacity_tokens=n)
    vc = tq.KVCache(3, Hkv, D, capacity_tokens=n)
    kd, vd = torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda()
    tq.encode_kv(kc, vc, kd[: n - 1], vd[: n - 1])
    q16 = synth.query(w, 6, 0)
    q = torch.from_numpy(q16).cuda().reshape(1, Hq, D)
    lens = torch.tensor([n], dtype=torch.int32, device="cuda")
    ws = torch.empty(tq.attn_workspace_bytes(1, Hq, D, n), dtype=torch.uint8, device="cuda")
    assert tq.device_status() == 0

    def call(out):
        if append:
            tq.attn_decode_append(kc, vc, kd[n - 1:].reshape(1, Hkv, D), vd[n - 1:].reshape(1, Hkv, D),
                                  q, lens, n, out, ws)
        else:
            tq.attn_decode(kc, vc, q, lens, n, out, ws)

    if not append:
        tq.encode_kv(kc, vc, kd[n - 1:], vd[n - 1:], pos0=n - 1)
    tq.inject_wait_timeout(1)
    out = torch.full((1, Hq, D), float("nan"), device="cuda")
    call(out)
    torch.cuda.synchronize()                   # the kernel returned: the context is usable
    assert tq.device_status() == 6             # TQ_ERR_DEVICE_TIMEOUT
    assert not out.isnan().any() and not out.any()   # empty partials: a zero output
    assert tq.device_status() == 0             # read and cleared

    out2 = torch.empty((1, Hq, D), device="cuda")
    call(out2)                                  # the next call is clean
    assert tq.device_status() == 0
    kr = oracle.encode_rows(3, k, Hkv, D)
    vr = oracle.encode_rows(3, v, Hkv, D)
    # the appended row was written by the timed-out call too (the append precedes the waits)
    assert np.array_equal(kc.buffer.cpu().numpy().reshape(n, -1), kr)
    ref = oracle.attn_decode(3, 3, kr, vr, q16, n, Hq, Hkv, D, 1.0 / np.sqrt(D))
    assert_attn_close(out2.cpu().numpy()[0], ref, f"after injected timeout append={append}")
