"""GPU parity of prompt-chunk (prefill) attention, through the C ABI, against the oracle.

Query j of a chunk sits at position pos0 + j and attends to rows 0 .. pos0 + j.  Small
cases (several query blocks and key tiles, ragged tails, every GQA group shape the
kernel takes, mixed cache types, a paged cache) compare every query element-wise; the
full-size case compares sampled queries with the oracle's decode step at their
positions.  Tolerance: the attention bar, 2e-3 relative L2 of each query token's output,
as the decode-step tests measure each sequence's output.
"""
import numpy as np
import pytest

import oracle
from rotated_bit_kv_tq_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from attn_check import assert_attn_close  # noqa: E402
DEV = "cuda"


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


def _queries(w, layer, pos0, n_q, seq=0):
    return np.stack([synth.query(w, layer, pos0 + j, seq) for j in range(n_q)])


def _check(got, ref, label):
    """Every (query token, head) output vector within the tolerance, and every query
    token's whole output [Hq][D] as well."""
    assert_attn_close(got, ref, label)
    n = ref.shape[0]
    assert_attn_close(got.reshape(n, -1), ref.reshape(n, -1), label + " (per token)")


PREFILL_CASES = [
    # (tk, tv, n_kv_heads, n_q_heads, pos0, n_q)
    (3, 3, 8, 32, 100, 70),    # G 4: 32 queries per CTA, ragged last block, 3 key tiles
    (3, 3, 2, 10, 0, 60),      # G 5 (rows 125..127 unused); first query sees one key
    (3, 3, 4, 4, 37, 200),     # G 1: 128 queries per CTA
    (2, 2, 1, 8, 500, 33),     # G 8, turbo2, long prefix
    (2, 3, 2, 8, 64, 64),      # mixed types, tile-aligned
    (3, 2, 2, 16, 5, 17),
    # eight KV heads: the blocks of heads 0..7 start at every even offset mod 16 of a row
    # (50 g and 34 g bytes), so the producers' 64-byte staging windows see every alignment
    (2, 2, 8, 16, 129, 40),    # turbo2, G 2
    (3, 2, 8, 8, 256, 31),     # mixed types, G 1, two full key tiles before the chunk
]


@pytest.mark.parametrize("tk,tv,hkv,hq,pos0,n_q", PREFILL_CASES)
def test_prefill_matches_oracle(tq, tk, tv, hkv, hq, pos0, n_q):
    w = synth.scaled(synth.TINY, n_kv_heads=hkv, n_q_heads=hq, head_dim=128)
    n_rows = pos0 + n_q
    k = synth.kv_tokens(w, 0, "K", 0, n_rows).reshape(n_rows, -1)
    v = synth.kv_tokens(w, 0, "V", 0, n_rows).reshape(n_rows, -1)
    kc = tq.KVCache(tk, hkv, 128, capacity_tokens=n_rows + 5)
    vc = tq.KVCache(tv, hkv, 128, capacity_tokens=n_rows + 5)
    tq.encode(kc, torch.from_numpy(k).to(DEV))
    tq.encode(vc, torch.from_numpy(v).to(DEV))
    q = _queries(w, 0, pos0, n_q)
    out = torch.full((n_q, hq, 128), float("nan"), device=DEV)
    tq.attn_prefill(kc, vc, torch.from_numpy(q).to(DEV), out, pos0=pos0)
    assert tq.device_status() == 0
    kr = kc.buffer[: n_rows * kc.row_bytes].cpu().numpy().reshape(n_rows, -1)
    vr = vc.buffer[: n_rows * vc.row_bytes].cpu().numpy().reshape(n_rows, -1)
    ref = oracle.attn_prefill(tk, tv, kr, vr, q, pos0, hkv, 128, 1 / np.sqrt(128))
    got = out.cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all()
    _check(got, ref, f"prefill turbo{tk}/{tv} Hkv{hkv} Hq{hq}#{pos0}+{n_q}")


def test_prefill_paged_cache_other_sequence(tq):
    """Sequence 1 of a paged cache (256-token pages in a seeded random order in the pool);
    its 390 rows span two pages."""
    w = synth.scaled(synth.BATCHED_PAGED, n_seqs=3, n_kv_heads=2, n_q_heads=8)
    pos0, n_q = 300, 90
    n_rows = pos0 + n_q
    pt, n_pages = synth.page_table(w, 512)
    k = synth.kv_tokens(w, 0, "K", 0, n_rows, 1).reshape(n_rows, -1)
    v = synth.kv_tokens(w, 0, "V", 0, n_rows, 1).reshape(n_rows, -1)
    ptd = torch.from_numpy(pt).to(DEV)
    kc = tq.KVCache(3, 2, 128, n_seqs=3, page_tokens=256, page_table=ptd, n_pages=n_pages)
    vc = tq.KVCache(3, 2, 128, n_seqs=3, page_tokens=256, page_table=ptd, n_pages=n_pages)
    tq.encode(kc, torch.from_numpy(k).to(DEV), seq_id=1)
    tq.encode(vc, torch.from_numpy(v).to(DEV), seq_id=1)
    q = _queries(w, 0, pos0, n_q, seq=1)
    out = torch.empty((n_q, 8, 128), device=DEV)
    tq.attn_prefill(kc, vc, torch.from_numpy(q).to(DEV), out, pos0=pos0, seq_id=1)
    assert tq.device_status() == 0
    ref = oracle.attn_prefill(3, 3, oracle.encode_rows(3, k, 2, 128), oracle.encode_rows(3, v, 2, 128),
                              q, pos0, 2, 128, 1 / np.sqrt(128))
    _check(out.cpu().numpy().astype(np.float64), ref, "prefill paged seq 1")


def test_prefill_head_dim_256_paged_cache_other_sequence(tq):
    """head_dim 256 on sequence 1 of a paged cache (256-token pages in a seeded random order),
    turbo2 K and turbo3 V, 2 KV heads (136- and 200-byte rows: the 2-byte staging path);
    its 420 rows span two pages and seven 64-key tiles."""
    w = synth.scaled(synth.BATCHED_PAGED, n_seqs=3, n_kv_heads=2, n_q_heads=8, head_dim=256)
    pos0, n_q = 333, 87
    n_rows = pos0 + n_q
    pt, n_pages = synth.page_table(w, 512)
    k = synth.kv_tokens(w, 0, "K", 0, n_rows, 1).reshape(n_rows, -1)
    v = synth.kv_tokens(w, 0, "V", 0, n_rows, 1).reshape(n_rows, -1)
    ptd = torch.from_numpy(pt).to(DEV)
    kc = tq.KVCache(2, 2, 256, n_seqs=3, page_tokens=256, page_table=ptd, n_pages=n_pages)
    vc = tq.KVCache(3, 2, 256, n_seqs=3, page_tokens=256, page_table=ptd, n_pages=n_pages)
    tq.encode(kc, torch.from_numpy(k).to(DEV), seq_id=1)
    tq.encode(vc, torch.from_numpy(v).to(DEV), seq_id=1)
    q = _queries(w, 0, pos0, n_q, seq=1)
    out = torch.full((n_q, 8, 256), float("nan"), device=DEV)
    tq.attn_prefill(kc, vc, torch.from_numpy(q).to(DEV), out, pos0=pos0, seq_id=1)
    assert tq.device_status() == 0
    ref = oracle.attn_prefill(2, 3, oracle.encode_rows(2, k, 2, 256), oracle.encode_rows(3, v, 2, 256),
                              q, pos0, 2, 256, 1 / np.sqrt(256))
    got = out.cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all()
    _check(got, ref, "prefill hd256 paged seq 1")


def test_prefill_zero_queries_and_unsupported_shapes(tq):
    kc = tq.KVCache(3, 2, 128, capacity_tokens=8)
    out = torch.empty((0, 4, 128), device=DEV)
    tq.attn_prefill(kc, kc, torch.zeros((0, 4, 128), dtype=torch.float16, device=DEV), out, pos0=3)
    k384 = tq.KVCache(3, 2, 384, capacity_tokens=8)   # three blocks per head: not taken
    with pytest.raises(tq.TQError) as e:
        tq.attn_prefill(k384, k384, torch.zeros((2, 4, 384), dtype=torch.float16, device=DEV),
                        torch.empty((2, 4, 384), device=DEV), pos0=0)
    assert e.value.status == 2
    with pytest.raises(tq.TQError) as e:   # a sequence the cache does not have
        tq.attn_prefill(kc, kc, torch.zeros((2, 4, 128), dtype=torch.float16, device=DEV),
                        torch.empty((2, 4, 128), device=DEV), pos0=0, seq_id=1)
    assert e.value.status == 1


@pytest.mark.slow
def test_prefill_full_size_llama_chunk_sampled(tq):
    """The last 512-token chunk of the Llama-3-8B-shape 32K prompt: every query runs, and
    four sampled queries match the oracle's decode step at their positions."""
    w = synth.LLAMA3_8B_32K
    T, n_q = w.ctx, 512
    pos0 = T - n_q
    k = synth.kv_tokens(w, 3, "K", 0, T).reshape(T, -1)
    v = synth.kv_tokens(w, 3, "V", 0, T).reshape(T, -1)
    kc = tq.KVCache(3, 8, 128, capacity_tokens=T)
    vc = tq.KVCache(3, 8, 128, capacity_tokens=T)
    tq.encode_kv(kc, vc, torch.from_numpy(k).to(DEV), torch.from_numpy(v).to(DEV))
    q = _queries(w, 3, pos0, n_q)
    out = torch.empty((n_q, 32, 128), device=DEV)
    tq.attn_prefill(kc, vc, torch.from_numpy(q).to(DEV), out, pos0=pos0)
    assert tq.device_status() == 0
    got = out.cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all()
    kr = kc.buffer.cpu().numpy().reshape(T, -1)
    vr = vc.buffer.cpu().numpy().reshape(T, -1)
    for j in (0, 1, 257, n_q - 1):
        ref = oracle.attn_decode(3, 3, kr, vr, q[j], pos0 + j + 1, 32, 8, 128, 1 / np.sqrt(128))
        _check(got[j][None], ref[None], f"prefill llama3-8b 32K last chunk#{j}")


PREFILL256_CASES = [
    # (tk, tv, n_kv_heads, n_q_heads, pos0, n_q) at head_dim 256 (two 128-value blocks per
    # head; the K blocks of a key have different norms)
    (2, 2, 4, 16, 100, 70),    # the head_dim-256 workload's heads (G 4), ragged last block
    (3, 3, 2, 10, 0, 60),      # G 5; the first query sees one key
    (3, 2, 1, 8, 300, 33),     # G 8, mixed types, 3 key tiles
    (2, 3, 2, 2, 37, 150),     # G 1: 128 queries per CTA
]


@pytest.mark.parametrize("tk,tv,hkv,hq,pos0,n_q", PREFILL256_CASES)
def test_prefill_head_dim_256_matches_oracle(tq, tk, tv, hkv, hq, pos0, n_q):
    w = synth.scaled(synth.HD256_128K, n_kv_heads=hkv, n_q_heads=hq, ctx=pos0 + n_q)
    n_rows = pos0 + n_q
    k = synth.kv_tokens(w, 0, "K", 0, n_rows).reshape(n_rows, -1)
    v = synth.kv_tokens(w, 0, "V", 0, n_rows).reshape(n_rows, -1)
    kc = tq.KVCache(tk, hkv, 256, capacity_tokens=n_rows + 3)
    vc = tq.KVCache(tv, hkv, 256, capacity_tokens=n_rows + 3)
    tq.encode(kc, torch.from_numpy(k).to(DEV))
    tq.encode(vc, torch.from_numpy(v).to(DEV))
    q = _queries(w, 0, pos0, n_q)
    out = torch.full((n_q, hq, 256), float("nan"), device=DEV)
    tq.attn_prefill(kc, vc, torch.from_numpy(q).to(DEV), out, pos0=pos0)
    assert tq.device_status() == 0
    kr = kc.buffer[: n_rows * kc.row_bytes].cpu().numpy().reshape(n_rows, -1)
    vr = vc.buffer[: n_rows * vc.row_bytes].cpu().numpy().reshape(n_rows, -1)
    ref = oracle.attn_prefill(tk, tv, kr, vr, q, pos0, hkv, 256, 1 / np.sqrt(256))
    got = out.cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all()
    _check(got, ref, f"prefill hd256 turbo{tk}/{tv} Hkv{hkv} Hq{hq}#{pos0}+{n_q}")


@pytest.mark.slow
def test_prefill_full_size_head_dim_256_chunk_sampled(tq):
    """The last 512-token chunk of the head_dim-256 workload's 131,072-token prompt (turbo2,
    4 KV heads, 16 query heads): every query runs, and three sampled queries match the
    oracle's decode step at their positions."""
    w = synth.HD256_128K
    T, n_q = w.ctx, 512
    pos0 = T - n_q
    k = synth.kv_tokens(w, 2, "K", 0, T).reshape(T, -1)
    v = synth.kv_tokens(w, 2, "V", 0, T).reshape(T, -1)
    kc = tq.KVCache(2, 4, 256, capacity_tokens=T)
    vc = tq.KVCache(2, 4, 256, capacity_tokens=T)
    tq.encode_kv(kc, vc, torch.from_numpy(k).to(DEV), torch.from_numpy(v).to(DEV))
    q = _queries(w, 2, pos0, n_q)
    out = torch.empty((n_q, 16, 256), device=DEV)
    tq.attn_prefill(kc, vc, torch.from_numpy(q).to(DEV), out, pos0=pos0)
    assert tq.device_status() == 0
    got = out.cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all()
    kr = kc.buffer.cpu().numpy().reshape(T, -1)
    vr = vc.buffer.cpu().numpy().reshape(T, -1)
    for j in (0, 300, n_q - 1):
        ref = oracle.attn_decode(2, 2, kr, vr, q[j], pos0 + j + 1, 16, 4, 256, 1 / np.sqrt(256))
        _check(got[j][None], ref[None], f"prefill hd256 131K last chunk#{j}")


SPLIT_CASES = [
    # (tk, tv, n_kv_heads, n_q_heads, pos0, n_q): shapes whose one-CTA-per-query-block grid
    # fills the last wave of 152 SMs poorly, so the key tiles of each query block are split
    # over a cluster of two CTAs (merged by log-sum-exp)
    (3, 3, 8, 32, 400, 250),   # 64 CTAs -> 128; 6 key tiles per block, 3 per CTA
    (3, 2, 2, 8, 0, 600),      # 38 CTAs -> 76; block 0 sees one key tile (its second CTA none)
    (2, 2, 4, 20, 517, 130),   # G 5 (25 queries per block), odd tile counts (5 / 6)
]


@pytest.mark.parametrize("tk,tv,hkv,hq,pos0,n_q", SPLIT_CASES)
def test_prefill_split_key_range_matches_oracle(tq, tk, tv, hkv, hq, pos0, n_q):
    w = synth.scaled(synth.TINY, n_kv_heads=hkv, n_q_heads=hq, head_dim=128)
    n_rows = pos0 + n_q
    k = synth.kv_tokens(w, 1, "K", 0, n_rows).reshape(n_rows, -1)
    v = synth.kv_tokens(w, 1, "V", 0, n_rows).reshape(n_rows, -1)
    kc = tq.KVCache(tk, hkv, 128, capacity_tokens=n_rows)
    vc = tq.KVCache(tv, hkv, 128, capacity_tokens=n_rows)
    tq.encode(kc, torch.from_numpy(k).to(DEV))
    tq.encode(vc, torch.from_numpy(v).to(DEV))
    q = _queries(w, 1, pos0, n_q)
    out = torch.full((n_q, hq, 128), float("nan"), device=DEV)
    tq.attn_prefill(kc, vc, torch.from_numpy(q).to(DEV), out, pos0=pos0)
    assert tq.device_status() == 0
    kr = kc.buffer.cpu().numpy().reshape(n_rows, -1)
    vr = vc.buffer.cpu().numpy().reshape(n_rows, -1)
    ref = oracle.attn_prefill(tk, tv, kr, vr, q, pos0, hkv, 128, 1 / np.sqrt(128))
    got = out.cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all()
    _check(got, ref, f"prefill split turbo{tk}/{tv} Hkv{hkv} Hq{hq}#{pos0}+{n_q}")
