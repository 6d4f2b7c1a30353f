"""GPU parity of tq_attn_decode_append: one decode step that appends each sequence's new
token and attends over the positions that include it.

The decode step of the kenji.blog article (section 8) writes the token at position N into
row N, then attends to rows 0..N.  The fused call must give exactly what the two-call
form gives (tq_encode_kv of the new rows, then tq_attn_decode): the same cache bytes and
the same output bits, since both run the same attention kernel over the same rows.  The
output is also checked against the oracle (encode and attention), within the attention
tolerance of 2e-3 relative L2.
"""
import numpy as np
import pytest

import oracle
from rotated_bit_kv_tq_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from attn_check import assert_attn_close  # noqa: E402
DEV = "cuda"
MASK_K = 0x9E3779B97F4A7C15F39CC0605CEDC834
MASK_V = 0x2545F4914F6CDD1D94D049BB133111EB


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


def _kv(w, layer, kind, n, seq):
    return synth.kv_tokens(w, layer, kind, 0, n, seq).reshape(n, w.n_kv_heads * w.head_dim)


def _caches(tq, w, tk, tv, S, cap, paged, var):
    kw = dict(n_seqs=S)
    if paged:
        pt, n_pages = synth.page_table(synth.scaled(w, n_seqs=S), cap)
        kw.update(page_tokens=256, page_table=torch.from_numpy(pt).to(DEV), n_pages=n_pages)
    else:
        kw.update(capacity_tokens=cap)
    kc = tq.KVCache(tk, w.n_kv_heads, w.head_dim, rotation_signs=var.get("k_signs"), **kw)
    vc = tq.KVCache(tv, w.n_kv_heads, w.head_dim, rotation_signs=var.get("v_signs"),
                    norm_correction=var.get("v_nc", False), **kw)
    return kc, vc


def _append_case(tq, w, tk, tv, lens, *, layer=0, paged=False, cap=None, var=None,
                 oracle_seqs=None):
    """Rows 0 .. L-2 of each sequence are encoded first; row L-1 is the step's new token."""
    var = var or {}
    S, Hkv, Hq, D = len(lens), w.n_kv_heads, w.n_q_heads, w.head_dim
    max_len = int(max(lens))
    cap = cap or max(max_len, 1)
    fused = _caches(tq, w, tk, tv, S, cap, paged, var)
    split = _caches(tq, w, tk, tv, S, cap, paged, var)
    ks = [_kv(w, layer, "K", L, s) for s, L in enumerate(lens)]
    vs = [_kv(w, layer, "V", L, s) for s, L in enumerate(lens)]
    for kc, vc in (fused, split):
        for s, L in enumerate(lens):
            if L > 1:
                tq.encode_kv(kc, vc, torch.from_numpy(ks[s][: L - 1]).to(DEV),
                             torch.from_numpy(vs[s][: L - 1]).to(DEV), seq_id=s)
    zero = np.zeros(Hkv * D, np.float16)
    k_new = torch.from_numpy(np.stack([ks[s][L - 1] if L else zero for s, L in enumerate(lens)])).to(DEV)
    v_new = torch.from_numpy(np.stack([vs[s][L - 1] if L else zero for s, L in enumerate(lens)])).to(DEV)
    q16 = np.stack([synth.query(w, layer, 0, s) for s in range(S)])
    q = torch.from_numpy(q16).to(DEV)
    lens_t = torch.tensor(lens, dtype=torch.int32, device=DEV)
    ws = torch.empty(max(16, tq.attn_workspace_bytes(S, Hq, D, max_len)), dtype=torch.uint8, device=DEV)
    out_f = torch.empty(S, Hq, D, dtype=torch.float32, device=DEV)
    out_s = torch.empty_like(out_f)
    tq.attn_decode_append(fused[0], fused[1], k_new.view(S, Hkv, D), v_new.view(S, Hkv, D), q,
                          lens_t, max_len, out_f, ws)
    assert tq.device_status() == 0
    live = [s for s, L in enumerate(lens) if L > 0]
    if live:
        idx = torch.tensor(live, dtype=torch.int32, device=DEV)
        tq.encode_kv(split[0], split[1], k_new[idx.long()], v_new[idx.long()], seq_ids=idx,
                     positions=lens_t[idx.long()] - 1)
    tq.attn_decode(split[0], split[1], q, lens_t, max_len, out_s, ws)
    assert tq.device_status() == 0
    # the two forms: same cache bytes, same output bits
    assert torch.equal(fused[0].buffer, split[0].buffer)
    assert torch.equal(fused[1].buffer, split[1].buffer)
    assert torch.equal(out_f, out_s)
    # against the oracle
    o = out_f.cpu().numpy().astype(np.float64)
    kvar = oracle.variant(signs=var.get("k_signs"))
    vvar = oracle.variant(signs=var.get("v_signs"), norm_correction=var.get("v_nc", False))
    for s in (oracle_seqs if oracle_seqs is not None else range(S)):
        L = lens[s]
        if L == 0:
            assert np.all(o[s] == 0.0)
            continue
        kr = oracle.encode_rows(tk, ks[s], Hkv, D, var=kvar)
        vr = oracle.encode_rows(tv, vs[s], Hkv, D, var=vvar)
        ref = oracle.attn_decode(tk, tv, kr, vr, q16[s], L, Hq, Hkv, D, 1.0 / np.sqrt(D),
                                 var_k=kvar, var_v=vvar)
        assert_attn_close(o[s], ref, f"append {w.name} turbo{tk}/{tv}#s{s} L{L}")


@pytest.mark.parametrize("tk,tv", [(3, 3), (2, 2), (3, 2), (2, 3)])
def test_append_llama_shape(tq, tk, tv):
    _append_case(tq, synth.LLAMA3_8B_32K, tk, tv, [1500])


def test_append_tiny_workload(tq):
    _append_case(tq, synth.TINY, 3, 3, [synth.TINY.ctx])


def test_append_gqa5_qwen_shape(tq):
    _append_case(tq, synth.QWEN25_14B_32K, 3, 3, [1234])


def test_append_head_dim_256(tq):
    _append_case(tq, synth.HD256_128K, 2, 2, [2100])


def test_append_batched_paged_with_empty_and_single(tq):
    """Several sequences, one of them empty (nothing appended, zero output) and one whose
    only row is the new token; split boundaries at 256-token pages."""
    _append_case(tq, synth.BATCHED_PAGED, 3, 3, [1, 37, 256, 257, 600, 999, 0, 1024],
                 paged=True, cap=1024)


def test_append_variants(tq):
    _append_case(tq, synth.LLAMA3_8B_32K, 3, 2, [700],
                 var={"k_signs": MASK_K, "v_signs": MASK_V, "v_nc": True})


def test_append_fallback_shape(tq):
    """Three KV heads (150-byte rows): the fp32 kernel, which appends in a launch of its own."""
    w = synth.scaled(synth.TINY, n_kv_heads=3, n_q_heads=6)
    _append_case(tq, w, 3, 3, [1, 90, 333])


def test_append_rejects_unaligned_rows(tq):
    w = synth.TINY
    kc = tq.KVCache(3, w.n_kv_heads, w.head_dim, capacity_tokens=16)
    q = torch.zeros(1, w.n_q_heads, w.head_dim, dtype=torch.float16, device=DEV)
    new = torch.zeros(2 * w.n_kv_heads * w.head_dim + 8, dtype=torch.float16, device=DEV)
    out = torch.zeros(1, w.n_q_heads, w.head_dim, device=DEV)
    ws = torch.empty(tq.attn_workspace_bytes(1, w.n_q_heads, w.head_dim, 16), dtype=torch.uint8, device=DEV)
    lens = torch.tensor([4], dtype=torch.int32, device=DEV)
    with pytest.raises(tq.TQError):
        tq.attn_decode_append(kc, kc, new[1:], new[1:], q, lens, 16, out, ws)


def test_full_llama_layer_32k_append(tq):
    """The benchmark's decode step at full size: one layer of the Llama-3-8B-shaped
    workload, the token at position 32,768 appended and attended over 32,769 rows."""
    _append_case(tq, synth.LLAMA3_8B_32K, 3, 3, [32769], layer=3)


def test_append_row_reaches_its_tile_through_a_refill(tq):
    """A context of 152 x 224 tokens fills every split of the Llama shape (224 tokens: tiles of
    64, 128 and 32), so the new row sits in a third tile that reuses a stage; the row then
    reaches shared memory through the cache and the refill copy instead of being written
    into the stage directly."""
    _append_case(tq, synth.LLAMA3_8B_32K, 3, 3, [152 * 224], layer=2)
