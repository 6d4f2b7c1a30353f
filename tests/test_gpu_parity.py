"""GPU parity: the CUDA path (through the C ABI) against the oracle.

Encode: codes and norms bit-exact.  Decode: within 1e-3 absolute.  Attention: within
2e-3 relative L2 of the oracle's attention over the same packed cache.  Inputs are the
seeded synthetic workloads of rotated_bit_kv_tq_gb300.synth, at sizes the oracle
finishes in seconds (several tiles and a ragged tail) and, for the full-size workloads,
on sampled rows and sequences.
"""
import numpy as np
import pytest

import oracle
from rotated_bit_kv_tq_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from attn_check import ATTN_TOL, assert_attn_close  # noqa: E402

DECODE_TOL = 1e-3


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


DEV = "cuda"


def _rows_from(cache, n_rows):
    return cache.buffer[: n_rows * cache.row_bytes].cpu().numpy().reshape(n_rows, cache.row_bytes)


def _kv(w, layer, kind, n, t0=0, seq=0):
    return synth.kv_tokens(w, layer, kind, t0, n, seq).reshape(n, w.n_kv_heads * w.head_dim)


# ------------------------------------------------------------------ encode

ENCODE_CASES = [
    # (type, n_kv_heads, head_dim, tokens)
    (3, 2, 128, 256),     # tiny workload
    (3, 8, 128, 1000),    # 16 rows per tile, ragged tail
    (2, 8, 128, 515),
    (2, 4, 256, 777),     # head_dim 256 = two blocks per head
    (3, 1, 128, 333),     # 50-byte rows: 2-byte store path
    (2, 3, 128, 100),     # 102-byte rows
    (3, 5, 256, 64),      # 10 blocks per row, 12 rows per tile
]


@pytest.mark.parametrize("tt,hkv,d,n", ENCODE_CASES)
def test_encode_bit_exact(tq, tt, hkv, d, n):
    w = synth.scaled(synth.TINY, n_kv_heads=hkv, n_q_heads=hkv, head_dim=d)
    src = _kv(w, 0, "K", n)
    cache = tq.KVCache(tt, hkv, d, capacity_tokens=n + 3)
    tq.encode(cache, torch.from_numpy(src).to(DEV))
    assert tq.device_status() == 0
    got = _rows_from(cache, n)
    ref = oracle.encode_rows(tt, src, hkv, d)
    assert np.array_equal(got, ref)
    # rows past the written range stay untouched
    assert not cache.buffer[n * cache.row_bytes:].any()


@pytest.mark.parametrize("n", [40, 2100])
def test_encode_edge_values(tq, n):
    """Zero blocks, single spikes, fp16 extremes, subnormals, norm saturation.  40 tokens
    (80 blocks) take the warp-per-block encoder of small appends, 2100 tokens (4200
    blocks) the one-thread-per-block encoder."""
    rng = np.random.default_rng(0)
    hkv, d = 2, 128
    x = rng.standard_normal((n, hkv * d)).astype(np.float16)
    x[0] = 0
    x[1] = 0; x[1, 5] = 3.0
    x[2] = np.float16(65504.0)
    x[3] = np.float16(-65504.0); x[3, ::2] = np.float16(65504.0)
    x[4] = np.float16(6e-8)
    x[5] = (rng.standard_normal(hkv * d) * 1e-6).astype(np.float16)
    x[6, :128] = np.float16(1.0)            # constant block: W x is a single spike
    x[7] = -0.0
    for tt in (2, 3):
        cache = tq.KVCache(tt, hkv, d, capacity_tokens=n)
        tq.encode(cache, torch.from_numpy(x).to(DEV))
        assert np.array_equal(_rows_from(cache, n), oracle.encode_rows(tt, x, hkv, d))


def test_encode_strided_source_and_offset(tq):
    """Rows taken from a wider buffer (stride > row) and written at pos0 > 0."""
    rng = np.random.default_rng(1)
    n, hkv, d = 70, 2, 256
    wide = rng.standard_normal((n, hkv * d + 3 * 8)).astype(np.float16)
    t = torch.from_numpy(wide).to(DEV)[:, : hkv * d]
    assert t.stride(0) == hkv * d + 24
    cache = tq.KVCache(2, hkv, d, capacity_tokens=200)
    tq.encode(cache, t, pos0=50)
    rows = cache.buffer.cpu().numpy().reshape(200, -1)
    ref = oracle.encode_rows(2, np.ascontiguousarray(wide[:, : hkv * d]), hkv, d)
    assert np.array_equal(rows[50:120], ref)
    assert not rows[:50].any() and not rows[120:].any()


def test_encode_paged_scattered(tq):
    """One token per sequence at arbitrary positions of a paged cache (the batched
    append of the batched-decode workload)."""
    w = synth.scaled(synth.BATCHED_PAGED, n_seqs=9)
    cap = 1024
    pt, n_pages = synth.page_table(w, cap)
    rng = np.random.default_rng(3)
    pos = rng.integers(0, cap, w.n_seqs).astype(np.int32)
    seqs = np.arange(w.n_seqs, dtype=np.int32)[::-1].copy()
    src = np.concatenate([_kv(w, 0, "V", 1, t0=int(p), seq=int(s)) for s, p in zip(seqs, pos)])
    cache = tq.KVCache(3, w.n_kv_heads, w.head_dim, n_seqs=w.n_seqs, page_tokens=256,
                       page_table=torch.from_numpy(pt).to(DEV), n_pages=n_pages)
    tq.encode(cache, torch.from_numpy(src).to(DEV), seq_ids=torch.from_numpy(seqs).to(DEV),
              positions=torch.from_numpy(pos).to(DEV))
    assert tq.device_status() == 0
    pool = cache.buffer.cpu().numpy().reshape(n_pages * 256, -1)
    ref = oracle.encode_rows(3, src, w.n_kv_heads, w.head_dim)
    for i, (s, p) in enumerate(zip(seqs, pos)):
        row = pt[s, p // 256] * 256 + p % 256
        assert np.array_equal(pool[row], ref[i])


LARGE_ENCODE_CASES = [
    # (type, n_kv_heads, head_dim, tokens, extra source stride, pos0): more than 4,096
    # blocks, so the one-thread-per-block encoder runs
    (3, 8, 128, 1100, 0, 0),      # dense source, one byte run per tile
    (2, 2, 256, 1500, 24, 37),    # strided source, offset rows, 2-byte stores
    (3, 5, 256, 500, 0, 3),       # 10 blocks per row, 12 rows per tile
    (2, 3, 128, 1500, 8, 0),      # 3 blocks per row, strided, 2-byte stores
]


@pytest.mark.parametrize("tt,hkv,d,n,extra,pos0", LARGE_ENCODE_CASES)
def test_encode_large_bit_exact(tq, tt, hkv, d, n, extra, pos0):
    w = synth.scaled(synth.TINY, n_kv_heads=hkv, n_q_heads=hkv, head_dim=d)
    src = _kv(w, 0, "V", n)
    wide = np.zeros((n, hkv * d + extra), dtype=np.float16)
    wide[:, : hkv * d] = src
    t = torch.from_numpy(wide).to(DEV)[:, : hkv * d]
    cap = pos0 + n + 5
    cache = tq.KVCache(tt, hkv, d, capacity_tokens=cap)
    tq.encode(cache, t, pos0=pos0)
    assert tq.device_status() == 0
    rows = cache.buffer.cpu().numpy().reshape(cap, -1)
    assert np.array_equal(rows[pos0:pos0 + n], oracle.encode_rows(tt, src, hkv, d))
    assert not rows[:pos0].any() and not rows[pos0 + n:].any()


@pytest.mark.parametrize("hkv", [8, 5])
def test_encode_large_paged_and_out_of_range(tq, hkv):
    """A prompt written into a paged cache whose pages are scattered, starting inside a
    page (tiles straddle page boundaries), and one that runs past the last page: its rows
    beyond are reported and never written, the rest are exact."""
    w = synth.scaled(synth.BATCHED_PAGED, n_seqs=2, n_kv_heads=hkv, n_q_heads=hkv)
    cap = 1024
    pt, n_pages = synth.page_table(w, cap)
    n = 900
    src = _kv(w, 0, "K", n)
    ref = oracle.encode_rows(3, src, hkv, w.head_dim)
    cache = tq.KVCache(3, hkv, w.head_dim, n_seqs=w.n_seqs, page_tokens=256,
                       page_table=torch.from_numpy(pt).to(DEV), n_pages=n_pages)
    all_rows = np.arange(n_pages * 256)
    for pos0, status in ((101, 0), (203, 7)):   # 203 + 900 > 1024: the last 79 rows are out
        cache.buffer.zero_()
        tq.encode(cache, torch.from_numpy(src).to(DEV), seq_id=1, pos0=pos0)
        assert tq.device_status() == status
        pool = cache.buffer.cpu().numpy().reshape(n_pages * 256, -1)
        end = min(pos0 + n, cap)
        phys = np.array([pt[1, p // 256] * 256 + p % 256 for p in range(pos0, end)])
        assert np.array_equal(pool[phys], ref[: end - pos0])
        assert not pool[np.setdiff1d(all_rows, phys)].any()


def test_encode_out_of_range_is_reported(tq):
    """A position past the capacity is skipped and reported, never written."""
    cache = tq.KVCache(3, 2, 128, capacity_tokens=4)
    src = torch.zeros(2, 256, dtype=torch.float16, device=DEV)
    tq.encode(cache, src, pos0=3)               # rows 3 (ok) and 4 (out of range)
    assert tq.device_status() == 7
    assert tq.device_status() == 0              # read clears it


def test_encode_zero_tokens_is_noop(tq):
    cache = tq.KVCache(3, 2, 128, capacity_tokens=4)
    tq.encode(cache, torch.zeros(0, 256, dtype=torch.float16, device=DEV))
    assert not cache.buffer.any()


# ------------------------------------------------------------------ decode

@pytest.mark.parametrize("tt,hkv,d,n", [(3, 2, 128, 256), (2, 4, 256, 300), (3, 8, 128, 77)])
def test_decode_within_tolerance(tq, tt, hkv, d, n):
    w = synth.scaled(synth.TINY, n_kv_heads=hkv, n_q_heads=hkv, head_dim=d)
    src = _kv(w, 0, "K", n)
    cache = tq.KVCache(tt, hkv, d, capacity_tokens=n)
    tq.encode(cache, torch.from_numpy(src).to(DEV))
    out = torch.empty(n - 5, hkv, d, dtype=torch.float32, device=DEV)
    tq.decode(cache, 0, 5, n - 5, out)
    ref = oracle.decode_rows(tt, oracle.encode_rows(tt, src, hkv, d)[5:], hkv, d)
    assert np.max(np.abs(out.cpu().numpy() - ref)) < DECODE_TOL


# ------------------------------------------------------------------ attention

def _attn_case(tq, w, tk, tv, lens, layer=0, paged=False, cap=None):
    """Encode K/V of every sequence, run attention, compare each sequence to the oracle."""
    S, Hkv, Hq, D = len(lens), w.n_kv_heads, w.n_q_heads, w.head_dim
    max_len = int(max(lens))
    cap = cap or max(max_len, 1)
    kw = dict(n_seqs=S)
    if paged:
        pt, n_pages = synth.page_table(synth.scaled(w, n_seqs=S), cap)
        kw.update(page_tokens=256, page_table=torch.from_numpy(pt).to(DEV), n_pages=n_pages)
    else:
        kw.update(capacity_tokens=cap)
    kc = tq.KVCache(tk, Hkv, D, **kw)
    vc = tq.KVCache(tv, Hkv, D, **kw)
    ks, vs = [], []
    for s, L in enumerate(lens):
        k16, v16 = _kv(w, layer, "K", L, seq=s), _kv(w, layer, "V", L, seq=s)
        ks.append(k16)
        vs.append(v16)
        if L:
            tq.encode(kc, torch.from_numpy(k16).to(DEV), seq_id=s)
            tq.encode(vc, torch.from_numpy(v16).to(DEV), seq_id=s)
    q16 = np.stack([synth.query(w, layer, 0, s) for s in range(S)])
    out = torch.empty(S, Hq, D, dtype=torch.float32, device=DEV)
    ws = torch.empty(max(16, tq.attn_workspace_bytes(S, Hq, D, max_len)), dtype=torch.uint8, device=DEV)
    tq.attn_decode(kc, vc, torch.from_numpy(q16).to(DEV), torch.tensor(lens, dtype=torch.int32, device=DEV),
                   max_len, out, ws)
    assert tq.device_status() == 0
    o = out.cpu().numpy().astype(np.float64)
    errs = []
    for s, L in enumerate(lens):
        kr = oracle.encode_rows(tk, ks[s], Hkv, D) if L else np.zeros((0, kc.row_bytes), np.uint8)
        vr = oracle.encode_rows(tv, vs[s], Hkv, D) if L else np.zeros((0, vc.row_bytes), np.uint8)
        ref = oracle.attn_decode(tk, tv, kr, vr, q16[s], L, Hq, Hkv, D, 1.0 / np.sqrt(D))
        if L == 0:
            assert np.all(o[s] == 0.0)
            continue
        errs.append(assert_attn_close(o[s], ref, f"decode {w.name} turbo{tk}/{tv}#s{s} L{L}"))
    return errs


def test_attn_tiny_workload(tq):
    _attn_case(tq, synth.TINY, 3, 3, [synth.TINY.ctx])


@pytest.mark.parametrize("tk,tv", [(3, 3), (2, 2), (3, 2), (2, 3)])
def test_attn_llama_shape_small_ctx(tq, tk, tv):
    w = synth.LLAMA3_8B_32K
    _attn_case(tq, w, tk, tv, [1500])


def test_attn_gqa5_qwen_shape(tq):
    _attn_case(tq, synth.QWEN25_14B_32K, 3, 3, [1234])
    _attn_case(tq, synth.QWEN25_14B_32K, 2, 2, [611])


def test_attn_head_dim_256(tq):
    _attn_case(tq, synth.HD256_128K, 2, 2, [2100])


def test_attn_batched_paged(tq):
    w = synth.BATCHED_PAGED
    lens = [1, 37, 256, 257, 600, 999, 0, 1024]
    _attn_case(tq, w, 3, 3, lens, paged=True, cap=1024)


def test_attn_single_token_and_ragged(tq):
    w = synth.TINY
    _attn_case(tq, w, 3, 3, [1, 2, 31, 33, 65])


def test_attn_equal_keys_give_mean(tq):
    """All keys equal -> uniform weights -> output = mean of the decoded values."""
    n, hkv, hq, d = 300, 2, 4, 128
    k = np.tile(np.random.default_rng(1).standard_normal((1, hkv * d)), (n, 1)).astype(np.float16)
    v = np.random.default_rng(2).standard_normal((n, hkv * d)).astype(np.float16)
    kc = tq.KVCache(3, hkv, d, capacity_tokens=n)
    vc = tq.KVCache(3, hkv, d, capacity_tokens=n)
    tq.encode(kc, torch.from_numpy(k).to(DEV))
    tq.encode(vc, torch.from_numpy(v).to(DEV))
    q = torch.randn(1, hq, d, device=DEV).half()
    out = torch.empty(1, hq, d, device=DEV)
    ws = torch.empty(tq.attn_workspace_bytes(1, hq, d, n), dtype=torch.uint8, device=DEV)
    tq.attn_decode(kc, vc, q, torch.tensor([n], dtype=torch.int32, device=DEV), n, out, ws)
    vh = oracle.decode_rows(3, oracle.encode_rows(3, v, hkv, d), hkv, d).mean(axis=0)
    ref = np.repeat(vh, hq // hkv, axis=0)
    got = out.cpu().numpy()[0]
    assert_attn_close(got, ref, "decode equal keys")


def test_grid_merge_epochs_on_a_reused_workspace(tq):
    """Decode calls that merge their own partials after a grid barrier (one wave of CTAs),
    all on one workspace whose barrier area starts as random bytes.  The calls alternate
    between grids of different sizes, a batch that takes the merge kernel instead, and a
    repeat of the first shape.  Each call gets a new query, so a barrier passed on an
    earlier call's flags would merge stale partials.  Every output must equal, bit for
    bit, that of the same call on a fresh zeroed workspace, and each matches the oracle."""
    w = synth.LLAMA3_8B_32K
    Hkv, Hq, D = w.n_kv_heads, w.n_q_heads, w.head_dim
    S = 3
    cap = 5100   # 3 sequences of 5,100 tokens: 3 x 51 splits, more CTAs than one wave
    kc = tq.KVCache(3, Hkv, D, n_seqs=S, capacity_tokens=cap)
    vc = tq.KVCache(3, Hkv, D, n_seqs=S, capacity_tokens=cap)
    ks = [_kv(w, 2, "K", cap, seq=s) for s in range(S)]
    vs = [_kv(w, 2, "V", cap, seq=s) for s in range(S)]
    for s in range(S):
        tq.encode(kc, torch.from_numpy(ks[s]).to(DEV), seq_id=s)
        tq.encode(vc, torch.from_numpy(vs[s]).to(DEV), seq_id=s)
    calls = [(1, 1500), (1, 333), (S, cap), (1, 1500), (1, 40), (1, cap)]
    ws_bytes = max(tq.attn_workspace_bytes(n, Hq, D, L) for n, L in calls)
    shared = torch.randint(0, 256, (ws_bytes,), dtype=torch.uint8,
                           generator=torch.Generator().manual_seed(11)).to(DEV)
    for i, (n, L) in enumerate(calls):
        q16 = np.stack([synth.query(w, 2, 10 + i, s) for s in range(n)])
        q = torch.from_numpy(q16).to(DEV)
        lens = torch.full((n,), L, dtype=torch.int32, device=DEV)
        fresh = torch.zeros(ws_bytes, dtype=torch.uint8, device=DEV)
        want = torch.empty(n, Hq, D, device=DEV)
        got = torch.empty(n, Hq, D, device=DEV)
        tq.attn_decode(kc, vc, q, lens, L, want, fresh)
        tq.attn_decode(kc, vc, q, lens, L, got, shared)
        torch.cuda.synchronize()
        assert tq.device_status() == 0
        assert torch.equal(got, want), f"call {i} ({n} x {L}) differs on the reused workspace"
        o = got.cpu().numpy().astype(np.float64)
        for s in range(n):
            kr = oracle.encode_rows(3, ks[s][:L], Hkv, D)
            vr = oracle.encode_rows(3, vs[s][:L], Hkv, D)
            ref = oracle.attn_decode(3, 3, kr, vr, q16[s], L, Hq, Hkv, D, 1.0 / np.sqrt(D))
            assert_attn_close(o[s], ref, f"grid merge call {i} s{s} L{L}")


def test_attn_workspace_too_small_is_rejected(tq):
    kc = tq.KVCache(3, 2, 128, capacity_tokens=64)
    q = torch.zeros(1, 4, 128, dtype=torch.float16, device=DEV)
    out = torch.empty(1, 4, 128, device=DEV)
    ws = torch.empty(16, dtype=torch.uint8, device=DEV)
    with pytest.raises(tq.TQError) as e:
        tq.attn_decode(kc, kc, q, torch.tensor([64], dtype=torch.int32, device=DEV), 64, out, ws)
    assert e.value.status == 4


def test_attn_len_beyond_max_is_reported(tq):
    kc = tq.KVCache(3, 2, 128, capacity_tokens=64)
    q = torch.zeros(1, 4, 128, dtype=torch.float16, device=DEV)
    out = torch.empty(1, 4, 128, device=DEV)
    ws = torch.empty(tq.attn_workspace_bytes(1, 4, 128, 32), dtype=torch.uint8, device=DEV)
    tq.attn_decode(kc, kc, q, torch.tensor([64], dtype=torch.int32, device=DEV), 32, out, ws)
    assert tq.device_status() == 7


# ------------------------------------------------------------------ full-size workloads

def test_full_llama_layer_32k_sampled(tq):
    """One layer of the Llama-3-8B-shaped workload at its full 32,768-token context, in
    the configuration the benchmark times: full-size attention vs the oracle, and
    sampled rows of the packed cache."""
    _attn_case(tq, synth.LLAMA3_8B_32K, 3, 3, [32768], layer=5)


def test_full_llama_layer_32k_prefill_encode_bit_exact(tq):
    """The benchmark's prefill call: tq_encode_kv of one Llama-3-8B-shaped layer's K and V
    over the full 32,768-token context; every packed row equals the oracle's."""
    w = synth.LLAMA3_8B_32K
    T = w.ctx
    k16, v16 = _kv(w, 9, "K", T), _kv(w, 9, "V", T)
    kc = tq.KVCache(3, w.n_kv_heads, w.head_dim, capacity_tokens=T + 128)
    vc = tq.KVCache(3, w.n_kv_heads, w.head_dim, capacity_tokens=T + 128)
    tq.encode_kv(kc, vc, torch.from_numpy(k16).to(DEV), torch.from_numpy(v16).to(DEV))
    assert tq.device_status() == 0
    assert np.array_equal(_rows_from(kc, T), oracle.encode_rows(3, k16, w.n_kv_heads, w.head_dim))
    assert np.array_equal(_rows_from(vc, T), oracle.encode_rows(3, v16, w.n_kv_heads, w.head_dim))


def test_full_hd256_layer_128k(tq):
    """One layer of the head_dim-256 workload at its full 131,072-token context."""
    _attn_case(tq, synth.HD256_128K, 2, 2, [131072], layer=1)


def test_full_batched_sampled_sequences(tq):
    """The batched paged workload's real lengths (U[1024, 16384]) for 6 of its sequences."""
    w = synth.BATCHED_PAGED
    lens = [int(x) for x in synth.seq_lens(w)[:6]]
    _attn_case(tq, w, 3, 3, lens, paged=True, cap=16384)


def test_full_qwen14b_layer_32k_both_types(tq):
    """The Qwen2.5-14B-shaped workload (8 KV heads, 40 query heads: G = 5) at its full
    32,768-token context, run once with turbo3 and once with turbo2 on identical data."""
    w = synth.QWEN25_14B_32K
    _attn_case(tq, w, 3, 3, [32768], layer=7)
    _attn_case(tq, w, 2, 2, [32768], layer=7)


def test_qwen14b_bytes_freed_and_mse(tq):
    """Bytes freed against FP16 ('Why the KV cache is so heavy' size formula) and the
    quantisation error per type, K and V separately, on one full-context layer."""
    w = synth.QWEN25_14B_32K
    T = w.ctx
    fp16 = oracle.kv_bytes(w.layers, w.n_kv_heads, w.head_dim, T, 2, 1)
    for tt, mse_lo, mse_hi in ((3, 0.025, 0.045), (2, 0.09, 0.14)):
        cache = tq.KVCache(tt, w.n_kv_heads, w.head_dim, capacity_tokens=T)
        # allocated bytes of all layers' K and V equal the formula at 50/128 or 34/128 B/value
        allocated = 2 * w.layers * cache.nbytes
        assert allocated == oracle.kv_bytes(w.layers, w.n_kv_heads, w.head_dim, T,
                                            oracle.block_bytes(tt), 128)
        assert fp16 - allocated == {3: 4944, 2: 5328}[tt] * 2 ** 20
        for kind in ("K", "V"):
            x = torch.from_numpy(_kv(w, 3, kind, T)).to(DEV)
            tq.encode(cache, x)
            xh = torch.empty(T, w.n_kv_heads, w.head_dim, device=DEV)
            tq.decode(cache, 0, 0, T, xh)
            xf = x.float().reshape(T, w.n_kv_heads, w.head_dim)
            nmse = float(((xf - xh) ** 2).sum() / (xf ** 2).sum())
            assert mse_lo < nmse < mse_hi, (tt, kind, nmse)


@pytest.mark.parametrize("tk,tv", [(3, 3), (2, 2), (3, 2)])
def test_encode_kv_one_launch_bit_exact(tq, tk, tv):
    """tq_encode_kv writes K and V rows exactly as two tq_encode calls (and the oracle) do,
    for whole prefills and for one-token appends at device positions."""
    w = synth.LLAMA3_8B_32K
    n = 300
    k = _kv(w, 1, "K", n)
    v = _kv(w, 1, "V", n)
    kc = tq.KVCache(tk, w.n_kv_heads, w.head_dim, capacity_tokens=n + 1)
    vc = tq.KVCache(tv, w.n_kv_heads, w.head_dim, capacity_tokens=n + 1)
    tq.encode_kv(kc, vc, torch.from_numpy(k).to(DEV), torch.from_numpy(v).to(DEV))
    kn, vn = _kv(w, 1, "K", 1, t0=n), _kv(w, 1, "V", 1, t0=n)
    pos = torch.tensor([n], dtype=torch.int32, device=DEV)
    tq.encode_kv(kc, vc, torch.from_numpy(kn).to(DEV), torch.from_numpy(vn).to(DEV), positions=pos)
    assert tq.device_status() == 0
    assert np.array_equal(_rows_from(kc, n + 1), oracle.encode_rows(tk, np.concatenate([k, kn]), w.n_kv_heads, w.head_dim))
    assert np.array_equal(_rows_from(vc, n + 1), oracle.encode_rows(tv, np.concatenate([v, vn]), w.n_kv_heads, w.head_dim))
