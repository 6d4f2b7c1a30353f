"""GPU parity of the quality variants (random-sign Hadamard W D, norm correction) against
the oracle: encode bit-exact (both encoders), decode within 1e-3, decode-step and
prompt-chunk attention within 2e-3 relative L2 of each query's output."""
import numpy as np
import pytest

import oracle
from rotated_bit_kv_tq_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DEV = "cuda"
from attn_check import assert_attn_close  # noqa: E402
MASK_K = int.from_bytes(np.random.default_rng(101).bytes(16), "little")
MASK_V = int.from_bytes(np.random.default_rng(202).bytes(16), "little")


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


def _rows(cache, n):
    return cache.buffer[: n * cache.row_bytes].cpu().numpy().reshape(n, cache.row_bytes)


VARIANTS = [(MASK_K, False), (0, True), (MASK_V, True)]


@pytest.mark.parametrize("tt", [2, 3])
@pytest.mark.parametrize("n", [40, 2100])      # warp-per-block encoder, one-thread-per-block
@pytest.mark.parametrize("signs,nc", VARIANTS)
def test_encode_variants_bit_exact(tq, tt, n, signs, nc):
    hkv, d = 2, 128
    w = synth.scaled(synth.TINY, n_kv_heads=hkv, n_q_heads=hkv, head_dim=d)
    x = synth.kv_tokens(w, 0, "K", 0, n).reshape(n, -1)
    x[0] = 0
    x[1, :128] = np.float16(0.5)                 # constant block: the signs' best case
    cache = tq.KVCache(tt, hkv, d, capacity_tokens=n, rotation_signs=signs, norm_correction=nc)
    tq.encode(cache, torch.from_numpy(x).to(DEV))
    assert tq.device_status() == 0
    ref = oracle.encode_rows(tt, x, hkv, d, var=oracle.variant(signs=signs, norm_correction=nc))
    assert np.array_equal(_rows(cache, n), ref)


@pytest.mark.parametrize("tt", [2, 3])
def test_decode_with_signs(tq, tt):
    hkv, d, n = 4, 256, 50
    w = synth.scaled(synth.TINY, n_kv_heads=hkv, n_q_heads=hkv, head_dim=d)
    x = synth.kv_tokens(w, 0, "V", 0, n).reshape(n, -1)
    var = oracle.variant(signs=MASK_V)
    cache = tq.KVCache(tt, hkv, d, capacity_tokens=n, rotation_signs=MASK_V)
    tq.encode(cache, torch.from_numpy(x).to(DEV))
    out = torch.empty((n, hkv, d), device=DEV)
    tq.decode(cache, 0, 0, n, out)
    ref = oracle.decode_rows(tt, oracle.encode_rows(tt, x, hkv, d, var=var), hkv, d, var=var)
    assert np.abs(out.cpu().numpy() - ref).max() < 1e-3


@pytest.mark.parametrize("hkv,hq", [(8, 32), (2, 8)])   # tensor-core kernel, fp32 kernel
def test_attention_decode_with_variants(tq, hkv, hq):
    d, n = 128, 700
    w = synth.scaled(synth.TINY, n_kv_heads=hkv, n_q_heads=hq, head_dim=d)
    k = synth.kv_tokens(w, 1, "K", 0, n).reshape(n, -1)
    v = synth.kv_tokens(w, 1, "V", 0, n).reshape(n, -1)
    kc = tq.KVCache(3, hkv, d, capacity_tokens=n, rotation_signs=MASK_K)
    vc = tq.KVCache(2, hkv, d, capacity_tokens=n, rotation_signs=MASK_V, norm_correction=True)
    tq.encode_kv(kc, vc, torch.from_numpy(k).to(DEV), torch.from_numpy(v).to(DEV))
    q = synth.query(w, 1, 0)
    out = torch.empty((1, hq, d), device=DEV)
    ws = torch.empty(tq.attn_workspace_bytes(1, hq, d, n), dtype=torch.uint8, device=DEV)
    tq.attn_decode(kc, vc, torch.from_numpy(q[None]).to(DEV), torch.tensor([n], dtype=torch.int32, device=DEV),
                   n, out, ws)
    assert tq.device_status() == 0
    vk, vv = oracle.variant(signs=MASK_K), oracle.variant(signs=MASK_V, norm_correction=True)
    ref = oracle.attn_decode(3, 2, _rows(kc, n), _rows(vc, n), q, n, hq, hkv, d, 1 / np.sqrt(d),
                             var_k=vk, var_v=vv)
    got = out.cpu().numpy()[0].astype(np.float64)
    assert_attn_close(got, ref, "decode variants turbo3/2")


@pytest.mark.parametrize("hkv,hq,d,pos0,n_q", [(8, 32, 128, 90, 40), (4, 16, 256, 150, 40)])
def test_prefill_with_variants(tq, hkv, hq, d, pos0, n_q):
    n = pos0 + n_q
    w = synth.scaled(synth.TINY, n_kv_heads=hkv, n_q_heads=hq, head_dim=d)
    k = synth.kv_tokens(w, 2, "K", 0, n).reshape(n, -1)
    v = synth.kv_tokens(w, 2, "V", 0, n).reshape(n, -1)
    kc = tq.KVCache(3, hkv, d, capacity_tokens=n, rotation_signs=MASK_K, norm_correction=True)
    vc = tq.KVCache(3, hkv, d, capacity_tokens=n, rotation_signs=MASK_V)
    tq.encode_kv(kc, vc, torch.from_numpy(k).to(DEV), torch.from_numpy(v).to(DEV))
    q = np.stack([synth.query(w, 2, pos0 + j) for j in range(n_q)])
    out = torch.empty((n_q, hq, d), device=DEV)
    tq.attn_prefill(kc, vc, torch.from_numpy(q).to(DEV), out, pos0=pos0)
    assert tq.device_status() == 0
    ref = oracle.attn_prefill(3, 3, _rows(kc, n), _rows(vc, n), q, pos0, hkv, d, 1 / np.sqrt(d),
                              var_k=oracle.variant(signs=MASK_K, norm_correction=True),
                              var_v=oracle.variant(signs=MASK_V))
    got = out.cpu().numpy().astype(np.float64)
    assert_attn_close(got, ref, f"prefill variants turbo3/3 D{d}")
    assert_attn_close(got.reshape(n_q, -1), ref.reshape(n_q, -1), f"prefill variants turbo3/3 D{d} (per token)")
