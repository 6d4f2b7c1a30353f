#!/usr/bin/env python3
"""Benchmark of the rotated, bit-packed KV-cache hot path on GB300.

One step is the whole hot path over one batch of synthetic input of a workload:
  1. prefill: tq_encode_kv of the K and V of every prompt token in every layer;
  2. 128 decode iterations; in every layer each one calls tq_attn_decode_append, which
     encodes each sequence's new token's K and V into the caches (in the attention launch
     itself) and attends over the grown context.
Metric: decode-attention tokens/s (value) and encode GB/s (encode.gbs), with the fraction
of the measured HBM peak of the dominant kernel (roofline).

Workloads (--workload; the default is the headline, the Llama-3-8B-shaped 32K cache):
  llama3-8b-kv-32k     32 layers, 8 KV / 32 query heads, head_dim 128, 32,768 tokens, turbo3
  qwen2.5-14b-kv-32k   48 layers, 8 KV / 40 query heads, 32,768 tokens, turbo3 and turbo2 on
                       the same data (one line per type, with bytes freed against FP16 and
                       the quantisation MSE of K and V)
  hd256-kv-128k        32 layers, 4 KV / 16 query heads, head_dim 256, 131,072 tokens, turbo2
  batched-paged-64seq  64 sequences of 1,024 .. 16,384 tokens in 256-token pages, turbo3;
                       every iteration appends and attends for all 64 sequences in one call
  --all runs these four, one JSON line each (two for the Qwen shape).
Outside the timed step, the single-sequence workloads also time prompt-chunk attention
(tq_attn_prefill) on the last 2,048-token chunk of the prompt in every layer.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME | --all]

--impl reference times the CPU oracle (oracle/) on a bounded sample of the same workload.
Under torchrun every rank runs an independent replica (the path has no data exchange);
value is the sum over ranks, time the max over ranks.
"""
from __future__ import annotations

import argparse
import concurrent.futures
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from rotated_bit_kv_tq_gb300 import synth  # noqa: E402

DECODE_STEPS = 128
METRIC = "turbo3 decode-attn tokens/s & encode GB/s at 32K ctx; % of HBM peak"
BENCH_WORKLOADS = [synth.LLAMA3_8B_32K, synth.QWEN25_14B_32K, synth.HD256_128K,
                   synth.BATCHED_PAGED]

# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) per launch measured by ncu on the
# benchmark's own shapes; see the profile summaries.  A workload without a capture of the
# current kernels reports null.
TRAFFIC = {
    # (workload, type): {"attn_per_token": DRAM bytes of one tq_attn_decode_append launch per
    # context token (the launch reads every packed row once, so traffic grows with the
    # context), "encode": DRAM bytes of one tq_encode_kv launch of one layer's prefill}
    # Llama-3-8B shape, turbo3: `--kernel-probe 32768` captures of the decode-step and encode
    # kernels under ncu; the encode capture is the benchmark's own launch size.
    ("llama3-8b-kv-32k", 3): {"attn_per_token": 26492416 / 32768, "encode": 134294528 + 10227968},
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=synth.LLAMA3_8B_32K.name,
                    choices=[w.name for w in synth.WORKLOADS])
    ap.add_argument("--all", action="store_true",
                    help="run every benchmark workload, one JSON line per workload and type")
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="skip the oracle timing (kernel studies only)")
    ap.add_argument("--kernel-probe", type=int, default=0, metavar="CTX",
                    help="time one layer's encode and attention at context CTX (the small "
                         "case the ncu captures use) instead of the full benchmark")
    ap.add_argument("--probe-kv-heads", type=int, default=0, metavar="N",
                    help="kernel probe on N KV heads (same query heads per KV head), e.g. 3 for "
                         "150-byte rows, a shape only the fp32 CUDA-core kernel takes")
    ap.add_argument("--prefill-chunk", type=int, default=0, metavar="N",
                    help="prefill probe: the last N queries of the CTX-token prompt as one chunk "
                         "(default: the whole prompt)")
    ap.add_argument("--phase-trace", type=int, default=0, metavar="CTX",
                    help="per-phase globaltimer trace of the decode step (traced library, "
                         "32 layers of the workload's shape at context CTX, graph replay)")
    ap.add_argument("--prefill-probe", type=int, default=0, metavar="CTX",
                    help="time one layer's prompt attention over a whole CTX-token prompt "
                         "(one chunk from position 0; the small case of the prefill capture)")
    return ap.parse_args()


def workload(name):
    return {w.name: w for w in synth.WORKLOADS}[name]


# ------------------------------------------------------------------ accounting

def row_bytes(w, tq_type):
    return w.n_kv_heads * (w.head_dim // 128) * (2 + 128 * tq_type // 8)


def encode_bytes_per_token(w, tq_type=3):
    """Algorithmic bytes of encoding one token of one layer (K and V): fp16 in + packed out."""
    vals = w.n_kv_heads * w.head_dim
    return 2 * (2 * vals + row_bytes(w, tq_type))


def attn_bytes(w, ctx, tq_type=3):
    """Algorithmic bytes of one decode-attention launch (one layer, one sequence)."""
    return ctx * 2 * row_bytes(w, tq_type) + w.n_q_heads * w.head_dim * (2 + 4)


def attn_bytes_batch(w, lens, tq_type=3):
    """Algorithmic bytes of one decode-attention launch over a batch of sequences whose
    contexts are `lens` (one layer)."""
    return sum(attn_bytes(w, int(L), tq_type) for L in lens)


def append_bytes(w, tq_type=3):
    """Algorithmic bytes of the decode-step append (one layer, one sequence): the new
    token's fp16 K and V read, one packed row of each written."""
    return 2 * (w.n_kv_heads * w.head_dim * 2 + row_bytes(w, tq_type))


def fp16_kv_bytes(w, tokens):
    """FP16 K and V bytes of `tokens` rows of every layer (the size formula of 'Why the KV
    cache is so heavy': layers x heads x head_dim x ctx x 2 x bytes)."""
    return w.layers * w.n_kv_heads * w.head_dim * tokens * 2 * 2


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples during the timed region (SM clock, throttle reasons)."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def measured_peak_hbm():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def measured_peak_tensor():
    """Dense fp16/bf16 tensor peak in TFLOP/s: the measured cuBLAS bf16 burst figure (fp16
    has the same nominal rate), else the fallback."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return float(json.load(f)["bf16_tflops"]), "measured (bf16 burst; fp16 same nominal rate)"
    return 1900.0, "fallback"


PREFILL_CHUNK = 2048   # prompt-chunk attention sample: the last chunk of the prompt


def prefill_flops(n_q_heads, head_dim, pos0, n_q):
    """Algorithmic FLOPs of causal chunk attention: 2 (QK) + 2 (PV) multiply-adds per
    (query head, coordinate, visible key); query j sees pos0 + j + 1 keys."""
    pairs = n_q * pos0 + n_q * (n_q + 1) // 2
    return 4.0 * n_q_heads * head_dim * pairs


# ------------------------------------------------------------------ multi-rank timing

def reduce_max(values, dist, device):
    """Max over ranks of per-rank timings (the slowest replica sets the job's time)."""
    import torch
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_throughput(world, units_per_rank, max_ms):
    """Whole-job throughput: the units all ranks processed over the slowest rank's time."""
    return world * units_per_rank / (max_ms / 1e3)


# ------------------------------------------------------------------ inputs

class Inputs:
    """Host (pinned) fp16 inputs of one workload.

    prompt_k / prompt_v: the prompt rows.  Single sequence: [L][T][row] (every layer drawn
    separately).  Batched: [n_tok][row], the prompts of all sequences back to back, drawn
    for layer 0 and encoded into every layer (the attention time does not depend on the
    values); seq_ids / positions give each row's place.
    new: [S][L][2][n_seqs][row] the appended tokens; q: [S][L][n_seqs][Hq][D] the queries."""

    def __init__(self, w, torch, pin):
        L, row, S, n = w.layers, w.n_kv_heads * w.head_dim, DECODE_STEPS, w.n_seqs
        self.lens = synth.seq_lens(w)
        self.batched = n > 1
        f16 = torch.float16
        if self.batched:
            n_tok = int(self.lens.sum())
            self.prompt_k = torch.empty((n_tok, row), dtype=f16, pin_memory=pin)
            self.prompt_v = torch.empty((n_tok, row), dtype=f16, pin_memory=pin)
            seq_ids = np.repeat(np.arange(n, dtype=np.int32), self.lens)
            starts = np.concatenate([[0], np.cumsum(self.lens)[:-1]])
            positions = (np.arange(n_tok) - np.repeat(starts, self.lens)).astype(np.int32)
            self.seq_ids = torch.from_numpy(seq_ids)
            self.positions = torch.from_numpy(positions)
            o = 0
            for s, Ls in enumerate(self.lens):
                Ls = int(Ls)
                self.prompt_k[o:o + Ls].copy_(torch.from_numpy(synth.kv_tokens(w, 0, "K", 0, Ls, s).reshape(Ls, row)))
                self.prompt_v[o:o + Ls].copy_(torch.from_numpy(synth.kv_tokens(w, 0, "V", 0, Ls, s).reshape(Ls, row)))
                o += Ls
        else:
            T = w.ctx
            self.prompt_k = torch.empty((L, T, row), dtype=f16, pin_memory=pin)
            self.prompt_v = torch.empty((L, T, row), dtype=f16, pin_memory=pin)
            for l in range(L):
                self.prompt_k[l].copy_(torch.from_numpy(synth.kv_tokens(w, l, "K", 0, T).reshape(T, row)))
                self.prompt_v[l].copy_(torch.from_numpy(synth.kv_tokens(w, l, "V", 0, T).reshape(T, row)))
        self.new = torch.empty((S, L, 2, n, row), dtype=f16, pin_memory=pin)
        self.q = torch.empty((S, L, n, w.n_q_heads, w.head_dim), dtype=f16, pin_memory=pin)
        for l in range(L):
            for s in range(n):
                L0 = int(self.lens[s])
                for j, kind in enumerate("KV"):
                    self.new[:, l, j, s].copy_(torch.from_numpy(
                        synth.kv_tokens(w, l, kind, L0, S, s).reshape(S, row)))
                for i in range(S):
                    self.q[i, l, s].copy_(torch.from_numpy(synth.query(w, l, i, s)))

    def h2d_prefill_bytes(self):
        return (self.prompt_k.numel() + self.prompt_v.numel()) * 2

    def h2d_iter_bytes(self):
        return (self.new[0].numel() + self.q[0].numel()) * 2


# ------------------------------------------------------------------ our CUDA path

def run_ours(args, w, tt, rank, world, local_rank, dist, cpu_baseline_on):
    import torch
    import rotated_bit_kv_tq_gb300 as tq
    dev = torch.device("cuda", local_rank)
    tq.codebook_init(tt, local_rank)
    L, Hkv, Hq, D, S, n = w.layers, w.n_kv_heads, w.n_q_heads, w.head_dim, DECODE_STEPS, w.n_seqs
    row = Hkv * D

    t_gen = time.time()
    inp = Inputs(w, torch, pin=True)
    t_gen = time.time() - t_gen
    lens0 = inp.lens.astype(np.int64)
    max_len = int(lens0.max()) + S
    pk_dev = inp.prompt_k.to(dev)
    pv_dev = inp.prompt_v.to(dev)
    new_dev = inp.new.to(dev)
    q_dev = inp.q.to(dev)
    if inp.batched:
        seq_ids_dev = inp.seq_ids.to(dev)
        pos_dev = inp.positions.to(dev)
        pt, n_pages = synth.page_table(w, max_len)
        pt_dev = torch.from_numpy(pt).to(dev)
        mk = lambda: tq.KVCache(tt, Hkv, D, n_seqs=n, page_tokens=w.page_tokens,  # noqa: E731
                                page_table=pt_dev, n_pages=n_pages, device=dev)
    else:
        mk = lambda: tq.KVCache(tt, Hkv, D, capacity_tokens=max_len, device=dev)  # noqa: E731
    kc = [mk() for _ in range(L)]
    vc = [mk() for _ in range(L)]
    out_dev = torch.zeros((L, n, Hq, D), dtype=torch.float32, device=dev)
    ws = torch.empty(max(16, tq.attn_workspace_bytes(n, Hq, D, max_len)), dtype=torch.uint8, device=dev)
    lens_start = torch.from_numpy((lens0 + 1).astype(np.int32)).to(dev)   # the first new row counted
    lens_dev = lens_start.clone()
    step_dev = torch.zeros(1, dtype=torch.int64, device=dev)
    new_buf = torch.empty((1, L, 2, n, row), dtype=torch.float16, device=dev)
    q_buf = torch.empty((1, L, n, Hq, D), dtype=torch.float16, device=dev)

    def encode_layer(l):
        if inp.batched:   # every sequence's prompt rows at their (sequence, position)
            tq.encode_kv(kc[l], vc[l], pk_dev, pv_dev, seq_ids=seq_ids_dev, positions=pos_dev)
        else:
            tq.encode_kv(kc[l], vc[l], pk_dev[l], pv_dev[l])

    def prefill():
        for l in range(L):
            encode_layer(l)
        lens_dev.copy_(lens_start)
        step_dev.zero_()

    # every layer's argument views into the iteration buffers, made once: a caller keeps its
    # per-layer tensors, and slicing them anew per call would time PyTorch, not this library
    layer_args = [(kc[l], vc[l], new_buf[0, l, 0].view(n, Hkv, D), new_buf[0, l, 1].view(n, Hkv, D),
                   q_buf[0, l], out_dev[l]) for l in range(L)]

    def attend_layer(l):
        k_c, v_c, k_new, v_new, q_l, out_l = layer_args[l]
        tq.attn_decode_append(k_c, v_c, k_new, v_new, q_l, lens_dev, max_len, out_l, ws)

    def decode_iter():
        torch.index_select(new_dev, 0, step_dev, out=new_buf)
        torch.index_select(q_dev, 0, step_dev, out=q_buf)
        for l in range(L):
            attend_layer(l)
        lens_dev.add_(1)
        step_dev.add_(1)

    # eager once (also sets kernel attributes), then capture both phases as CUDA graphs
    prefill()
    decode_iter()
    torch.cuda.synchronize()
    assert tq.device_status() == 0
    cap = torch.cuda.Stream()
    g_pre, g_dec = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_pre, stream=cap, capture_error_mode="thread_local"):
        prefill()
    with torch.cuda.graph(g_dec, stream=cap, capture_error_mode="thread_local"):
        decode_iter()

    def step():
        g_pre.replay()
        for _ in range(S):
            g_dec.replay()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clocks = ClockSampler(local_rank)
    clocks.start()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    for k in range(args.steps):
        evs[k][0].record()
        g_pre.replay()
        evs[k][1].record()
        for _ in range(S):
            g_dec.replay()
        evs[k][2].record()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clk = clocks.stop()
    pre_ms = sum(e[0].elapsed_time(e[1]) for e in evs)
    dec_ms = sum(e[1].elapsed_time(e[2]) for e in evs)
    status = tq.device_status()

    # per-launch durations of the decode-step and encode calls, right after the timed region
    # and in the same state: each call is replayed from a CUDA graph of the L layers' calls
    # (as in the timed step), bracketed by CUDA events on the replay stream.  The decode
    # step re-appends the last iteration's token at the last position (the same bytes).
    lens_dev.copy_(lens_start + (S - 1))
    g_att, g_enc = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_att, stream=cap, capture_error_mode="thread_local"):
        for l in range(L):
            attend_layer(l)
    with torch.cuda.graph(g_enc, stream=cap, capture_error_mode="thread_local"):
        for l in range(L):   # the prefill's own call: K and V of one layer in one launch
            encode_layer(l)

    def graph_ms(g, reps=3):
        g.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / (reps * L)

    attn_launch_ms = graph_ms(g_att)
    enc_launch_ms = graph_ms(g_enc)
    final_ctx = lens0 + S                    # contexts of the timed launch (new row included)

    # prompt-chunk attention (tensor-bound, timed alone): the last PREFILL_CHUNK queries of
    # the prompt over every layer's cache (single-sequence workloads)
    prefill_line = None
    if not inp.batched:
        T = w.ctx
        pf_pos0 = T - PREFILL_CHUNK
        gen = torch.Generator(device=dev)
        gen.manual_seed(11)
        q_pf = torch.randn((PREFILL_CHUNK, Hq, D), generator=gen, device=dev).half()
        out_pf = torch.empty((PREFILL_CHUNK, Hq, D), dtype=torch.float32, device=dev)

        def prefill_layers():
            for l in range(L):
                tq.attn_prefill(kc[l], vc[l], q_pf, out_pf, pos0=pf_pos0)

        prefill_layers()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        pf_reps = 2
        e0.record()
        for _ in range(pf_reps):
            prefill_layers()
        e1.record()
        torch.cuda.synchronize()
        pf_ms = e0.elapsed_time(e1) / pf_reps        # all layers
        assert torch.isfinite(out_pf).all() and tq.device_status() == 0
        tpeak, tpeak_kind = measured_peak_tensor()
        pf_flops = prefill_flops(Hq, D, pf_pos0, PREFILL_CHUNK)
        pf_tflops = pf_flops * L / (pf_ms / 1e3) / 1e12
        prefill_line = {
            "metric": f"prompt-chunk attention tokens/s ({PREFILL_CHUNK}-token chunk at position "
                      f"{pf_pos0}, {L} layers)",
            "value": PREFILL_CHUNK / (pf_ms / 1e3), "unit": "tokens/s", "ms": pf_ms,
            "roofline": {"kernel": "tq_attn_prefill", "bound": "tensor",
                         "achieved": pf_tflops, "peak": tpeak, "unit": "TFLOP/s",
                         "frac": pf_tflops / tpeak, "peak_source": tpeak_kind, "traffic": None,
                         "flops_per_launch": pf_flops, "launch_ms": pf_ms / L}}

    # end to end through the public API with host buffers, no CUDA graph: every step copies
    # its fp16 prompt rows and every iteration its new tokens and queries from pinned host
    # memory, calls tq_encode_kv / tq_attn_decode_append once per layer from Python, and
    # reads the iteration's outputs back to pinned host memory
    out_host = torch.empty((S, L, n, Hq, D), dtype=torch.float32, pin_memory=True)
    stream = torch.cuda.current_stream()
    e2e_evs = []
    n_e2e = max(1, min(args.steps, 3))
    for k in range(n_e2e):
        ea, eb, ec = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        ea.record(stream)
        pk_dev.copy_(inp.prompt_k, non_blocking=True)
        pv_dev.copy_(inp.prompt_v, non_blocking=True)
        for l in range(L):
            encode_layer(l)
        lens_dev.copy_(lens_start)
        eb.record(stream)
        for i in range(S):
            new_buf.copy_(inp.new[i:i + 1], non_blocking=True)
            q_buf.copy_(inp.q[i:i + 1], non_blocking=True)
            for l in range(L):
                attend_layer(l)
            lens_dev.add_(1)
            out_host[i].copy_(out_dev, non_blocking=True)
        ec.record(stream)
        e2e_evs.append((ea, eb, ec))
    torch.cuda.synchronize()
    e2e_pre_ms = sum(a.elapsed_time(b) for a, b, _ in e2e_evs)
    e2e_dec_ms = sum(b.elapsed_time(c) for _, b, c in e2e_evs)
    assert np.isfinite(out_host.numpy()).all() and tq.device_status() == 0

    # the graph-replay form of the same end-to-end step (the launches captured once)
    g_evs = []
    for k in range(n_e2e):
        ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g_pre.replay()
        ea.record(stream)
        for i in range(S):
            new_dev[i].copy_(inp.new[i], non_blocking=True)
            q_dev[i].copy_(inp.q[i], non_blocking=True)
            g_dec.replay()
            out_host[i].copy_(out_dev, non_blocking=True)
        eb.record(stream)
        g_evs.append((ea, eb))
    torch.cuda.synchronize()
    e2e_graph_ms = sum(a.elapsed_time(b) for a, b in g_evs)

    # quantisation report of the Qwen-shaped workload: bytes freed against FP16 and the MSE
    # of K and V on one full-context layer (decoded by tq_decode)
    quality = None
    if w.name == synth.QWEN25_14B_32K.name:
        T = w.ctx
        fp16_b = fp16_kv_bytes(w, T)
        packed_b = 2 * L * T * kc[0].row_bytes
        quality = {"fp16_kv_mib": fp16_b / 2 ** 20, "packed_kv_mib": packed_b / 2 ** 20,
                   "bytes_freed_mib": (fp16_b - packed_b) / 2 ** 20,
                   "layer": 0, "tokens": T}
        xh = torch.empty((T, Hkv, D), dtype=torch.float32, device=dev)
        for kind, cache, src in (("K", kc[0], pk_dev[0]), ("V", vc[0], pv_dev[0])):
            tq.decode(cache, 0, 0, T, xh)
            xf = src.float().reshape(T, Hkv, D)
            err = ((xf - xh) ** 2).sum(dim=-1)            # per 128-value block (head_dim 128)
            nrm = (xf ** 2).sum(dim=-1)
            quality[f"{kind}_nmse"] = float(err.sum() / nrm.sum())
            quality[f"{kind}_nmse_block_mean"] = float((err / nrm.clamp_min(1e-30)).mean())
            quality[f"{kind}_mse"] = float(err.sum() / (T * Hkv * D))
        torch.cuda.synchronize()

    if dist:
        pre_ms, dec_ms, e2e_pre_ms, e2e_dec_ms, e2e_graph_ms = reduce_max(
            [pre_ms, dec_ms, e2e_pre_ms, e2e_dec_ms, e2e_graph_ms], dist, dev)
    if rank != 0:
        return None

    K = args.steps
    prompt_tokens = int(lens0.sum())
    enc_bytes = encode_bytes_per_token(w, tt) * prompt_tokens * L
    value = job_throughput(world, K * S * n, dec_ms)
    enc_gbs = world * K * enc_bytes / (pre_ms / 1e3) / 1e9
    peak, peak_kind = measured_peak_hbm()
    a_bytes = attn_bytes_batch(w, final_ctx, tt) + n * append_bytes(w, tt)
    a_gbs = a_bytes / (attn_launch_ms / 1e3) / 1e9
    e_bytes = encode_bytes_per_token(w, tt) * prompt_tokens      # K and V of one layer
    e_gbs = e_bytes / (enc_launch_ms / 1e3) / 1e9
    traffic = TRAFFIC.get((w.name, tt), {})
    attn_traffic = (traffic["attn_per_token"] * float(final_ctx.sum())
                    if "attn_per_token" in traffic else None)
    decode_gb = attn_bytes_batch(w, lens0 + S // 2, tt) * L / 1e9
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": (pre_ms + dec_ms) / K,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": f"f32 (fp16 in, {tt}-bit codes)",
        "data": "synthetic (seeded; K with lognormal channel scales and x%g outlier channels)"
                % w.outlier_gain + ("; prompt rows of every layer from layer 0's draws" if inp.batched else ""),
        "config": {"workload": w.name, "layers": L, "n_kv_heads": Hkv, "n_q_heads": Hq,
                   "head_dim": D, "ctx": w.ctx if not inp.batched else int(lens0.max()),
                   "prompt_tokens": prompt_tokens, "decode_steps": S, "cache_type": f"turbo{tt}",
                   "batch": n, "page_tokens": w.page_tokens,
                   "parallelism": f"replicas x{world}",
                   "l2": f"inputs larger than L2: {decode_gb:.2f} GB packed cache read per decode "
                         f"iteration, {enc_bytes / 1e9:.1f} GB moved per prefill"},
        "encode": {"gbs": enc_gbs, "tokens_per_s": world * K * prompt_tokens * L / (pre_ms / 1e3),
                   "ms_per_step": pre_ms / K},
        "decode_ms_per_step": dec_ms / K,
        "roofline": {"kernel": "tq_attn_decode_append (append + split-K partial + merge)",
                     "bound": "hbm",
                     "achieved": a_gbs, "peak": peak, "unit": "GB/s", "frac": a_gbs / peak,
                     "peak_source": peak_kind,
                     "traffic": attn_traffic,
                     "bytes_per_launch": a_bytes, "launch_ms": attn_launch_ms},
        "encode_roofline": {"kernel": "tq_encode_kv (prefill, one layer, K and V)", "bound": "hbm",
                            "achieved": e_gbs, "peak": peak, "unit": "GB/s", "frac": e_gbs / peak,
                            "peak_source": peak_kind, "bytes_per_launch": e_bytes,
                            "traffic": traffic.get("encode"), "launch_ms": enc_launch_ms},
        "e2e": {"value": world * n_e2e * S * n / (e2e_dec_ms / 1e3), "unit": "tokens/s",
                "h2d_bytes_per_step": inp.h2d_prefill_bytes() + S * inp.h2d_iter_bytes(),
                "d2h_bytes_per_step": S * L * n * Hq * D * 4,
                "how": "per-layer Python calls of tq_attn_decode_append (no CUDA graph), pinned "
                       "host copies of every iteration's new tokens and queries in, outputs out",
                "graph_replay_value": world * n_e2e * S * n / (e2e_graph_ms / 1e3),
                "encode_gbs": world * n_e2e * enc_bytes / (e2e_pre_ms / 1e3) / 1e9,
                "encode_note": "includes the host-to-device copy of the fp16 prompt rows"},
        # one tq_encode_kv launch per layer; one launch per decode call for a single sequence
        # (its splits fit one wave and merge inside the launch), two for a batch (attention,
        # then the merge kernel)
        "gpu_launches": K * (L + S * L * (1 if n == 1 else 2)),
        "clocks": clk,
        "device_status": status,
        "input_gen_s": t_gen,
    }
    if prefill_line:
        line["prefill"] = prefill_line
    if quality:
        line["quality"] = quality
    if world == 1 and cpu_baseline_on:
        line["cpu_baseline"] = cpu_baseline(w, tt)
    print(json.dumps(line), flush=True)
    # release this workload's device and pinned memory before the next one
    del inp, pk_dev, pv_dev, new_dev, q_dev, kc, vc, out_dev, ws, g_pre, g_dec, g_att, g_enc
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return line


# ------------------------------------------------------------------ the oracle on the host

def _oracle_layer_sample(w, tt, layer, n_seqs):
    """One layer of the workload through the oracle: the prefill encode of K and V of the
    first n_seqs sequences (full context) and one decode-attention step per sequence over
    its whole context.  Returns (encode seconds, attention seconds, encode bytes, tokens)."""
    import oracle
    Hkv, Hq, D = w.n_kv_heads, w.n_q_heads, w.head_dim
    row = Hkv * D
    lens = synth.seq_lens(w)[:n_seqs]
    data = []
    for s, Ls in enumerate(lens):
        Ls = int(Ls) + 1
        data.append((synth.kv_tokens(w, layer, "K", 0, Ls, s).reshape(Ls, row),
                     synth.kv_tokens(w, layer, "V", 0, Ls, s).reshape(Ls, row),
                     synth.query(w, layer, 0, s), Ls))
    t_enc = t_att = 0.0
    enc_b = 0
    for k16, v16, q16, Ls in data:
        t0 = time.perf_counter()
        kr = oracle.encode_rows(tt, k16, Hkv, D)
        vr = oracle.encode_rows(tt, v16, Hkv, D)
        t1 = time.perf_counter()
        oracle.attn_decode(tt, tt, kr, vr, q16, Ls, Hq, Hkv, D, 1.0 / np.sqrt(D))
        t2 = time.perf_counter()
        t_enc += t1 - t0
        t_att += t2 - t1
        enc_b += encode_bytes_per_token(w, tt) * Ls
    return t_enc, t_att, enc_b, len(data)


def cpu_baseline(w, tt, multi_thread=True):
    """The oracle (single-threaded C, as it stands) on a bounded sample of the workload,
    plus (multi_thread) a second, reported-only figure with one oracle call per host thread
    on different layers (ctypes releases the GIL, so the calls run in parallel)."""
    import oracle
    oracle.build()
    n_sample = 1 if w.n_seqs == 1 else 2           # sequences per layer sample
    t_enc, t_att, enc_b, ns = _oracle_layer_sample(w, tt, 0, n_sample)
    # decode tokens/s: the sample's sequences, one step each, scaled to all layers
    value = ns / (t_att * w.layers)
    host_cores = os.cpu_count() or 1
    mt = None
    if multi_thread:
        nt = min(host_cores, w.layers)
        t0 = time.perf_counter()
        with concurrent.futures.ThreadPoolExecutor(max_workers=nt) as ex:
            res = list(ex.map(lambda l: _oracle_layer_sample(w, tt, l, n_sample), range(nt)))
        wall = time.perf_counter() - t0
        mt = {"value": sum(r[3] for r in res) / wall / w.layers, "threads": nt,
              "encode_gbs": sum(r[2] for r in res) / wall / 1e9,
              "sample": f"{nt} layers in parallel, one per thread, each as the single-thread "
                        "sample (inputs drawn inside the timed threads)"}
    lens = synth.seq_lens(w)[:n_sample]
    out = {"value": value, "unit": "tokens/s", "cores": 1, "host_cores": host_cores,
            "kind": "oracle",
            "sample": f"layer 0 of {w.name}, turbo{tt}: encode of K and V of {ns} sequence(s) "
                      f"of {', '.join(str(int(x) + 1) for x in lens)} tokens, then one "
                      f"decode-attention step each over its whole context; tokens/s = "
                      f"sequences / (attention time x {w.layers} layers)",
            "encode_gbs": enc_b / t_enc / 1e9, "seconds": t_enc + t_att}
    if mt:
        out["multi_thread"] = mt
    return out


def run_reference(args, rank, world):
    """The reference arm: the oracle, as it stands, on the host cores."""
    if rank != 0:
        return
    w = workload(args.workload)
    tt = w.types[0]
    vals, secs = [], 0.0
    base = None
    for _ in range(max(1, args.steps)):
        base = cpu_baseline(w, tt, multi_thread=False)
        vals.append(base["value"])
        secs += base["seconds"]
        if secs > 150:
            break
    value = statistics.mean(vals)
    base["value"] = value
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": value, "unit": "tokens/s", "n_gpus": world, "steps": len(vals),
        "warmup": args.warmup, "ms_per_step": 1e3 * secs / len(vals), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)", "data": "synthetic",
        "config": {"workload": w.name, "layers": w.layers, "n_kv_heads": w.n_kv_heads,
                   "n_q_heads": w.n_q_heads, "head_dim": w.head_dim, "ctx": w.ctx,
                   "cache_type": f"turbo{tt}", "batch": w.n_seqs},
        "cpu_baseline": base,
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def kernel_probe(args):
    """One layer of the workload's shape at context args.kernel_probe: encode of K and V,
    then repeated decode attention and decode steps (append + attention, the benchmark's
    call); per-call times from CUDA events (not a bench line)."""
    import torch
    import rotated_bit_kv_tq_gb300 as tq
    from rotated_bit_kv_tq_gb300 import build
    build.build()
    w = workload(args.workload)
    if args.probe_kv_heads:
        w = synth.scaled(w, n_kv_heads=args.probe_kv_heads, n_q_heads=w.group * args.probe_kv_heads)
    tt = w.types[0]
    tq.codebook_init(tt, 0)
    ctx, Hkv, Hq, D = args.kernel_probe, w.n_kv_heads, w.n_q_heads, w.head_dim
    k16 = torch.from_numpy(synth.kv_tokens(w, 0, "K", 0, ctx).reshape(ctx, -1)).cuda()
    v16 = torch.from_numpy(synth.kv_tokens(w, 0, "V", 0, ctx).reshape(ctx, -1)).cuda()
    kc = tq.KVCache(tt, Hkv, D, capacity_tokens=ctx)
    vc = tq.KVCache(tt, Hkv, D, capacity_tokens=ctx)
    q = torch.from_numpy(synth.query(w, 0, 0)).cuda().reshape(1, Hq, D)
    out = torch.empty(1, Hq, D, device="cuda")
    lens = torch.tensor([ctx], dtype=torch.int32, device="cuda")
    ws = torch.empty(max(16, tq.attn_workspace_bytes(1, Hq, D, ctx)), dtype=torch.uint8, device="cuda")
    kn, vn = k16[ctx - 1:].reshape(1, Hkv, D), v16[ctx - 1:].reshape(1, Hkv, D)

    def timed(fn, n):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(n):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n

    def step():
        tq.attn_decode_append(kc, vc, kn, vn, q, lens, ctx, out, ws)

    for _ in range(3):
        tq.encode_kv(kc, vc, k16, v16)
        tq.attn_decode(kc, vc, q, lens, ctx, out, ws)
        step()
    torch.cuda.synchronize()
    enc_ms = timed(lambda: tq.encode_kv(kc, vc, k16, v16), 10)
    att_ms = timed(lambda: tq.attn_decode(kc, vc, q, lens, ctx, out, ws), 20)
    stp_ms = timed(step, 20)
    enc_b = ctx * encode_bytes_per_token(w, tt)
    att_b = attn_bytes(w, ctx, tt)
    print(json.dumps({"probe": w.name, "ctx": ctx, "encode_kv_us": enc_ms * 1e3,
                      "encode_gbs": enc_b / enc_ms / 1e6, "attn_us": att_ms * 1e3,
                      "attn_gbs": att_b / att_ms / 1e6, "step_us": stp_ms * 1e3,
                      "step_gbs": (att_b + append_bytes(w, tt)) / stp_ms / 1e6,
                      "status": tq.device_status()}))


TRACE_PHASES = {
    "attention": ["entry", "dependency wait returned",
                  "sequence length loaded (a full first tile requested)",
                  "set-up done (any other first tile requested)", "query rotated (CTA barrier)",
                  "first tile landed",
                  "loop end (slowest warp)",
                  "epilogue done (cluster barrier; grid merge: partial rows stored)",
                  "cluster merge done (grid merge: grid barrier passed)",
                  "grid merge: rows loaded", "grid merge: output stored",
                  "warps of each KV head combined"],
    "merge": ["entry", "dependency wait returned", "partial rows loaded", "output stored"],
}


def phase_trace(args):
    """Decode step of every layer of the workload's shape at context CTX, replayed from a
    CUDA graph through the traced library (rotated_bit_kv_tq_gb300.build(trace=True)); prints
    the per-layer call time and, for the last layer's call, each phase's time across CTAs
    (min / median / max, us after the first CTA's dependency wait returned)."""
    import ctypes
    import torch
    from rotated_bit_kv_tq_gb300 import _lib, build
    lib = _lib.load(build.build(trace=True))     # the traced library, before any other load
    import rotated_bit_kv_tq_gb300 as tq
    lib.tq_phase_trace_read.argtypes = [ctypes.c_void_p, ctypes.c_size_t]
    w = workload(args.workload)
    tt = w.types[0]
    tq.codebook_init(tt, 0)
    L, Hkv, Hq, D, n = w.layers, w.n_kv_heads, w.n_q_heads, w.head_dim, w.n_seqs
    row = Hkv * D
    if n == 1:   # one sequence of CTX tokens plus the appended one
        lens0 = np.array([args.phase_trace], np.int64)
    else:        # the batched workload's drawn lengths (CTX is ignored)
        lens0 = synth.seq_lens(w).astype(np.int64)
    max_len = int(lens0.max()) + 1
    # prompt rows of every layer from layer 0's draws (timing only), then the new token
    ks = [synth.kv_tokens(w, 0, "K", 0, int(L0) + 1, s).reshape(int(L0) + 1, row) for s, L0 in enumerate(lens0)]
    vs = [synth.kv_tokens(w, 0, "V", 0, int(L0) + 1, s).reshape(int(L0) + 1, row) for s, L0 in enumerate(lens0)]
    if n == 1:
        mk = lambda: tq.KVCache(tt, Hkv, D, capacity_tokens=max_len)  # noqa: E731
    else:
        pt, n_pages = synth.page_table(w, max_len)
        ptd = torch.from_numpy(pt).cuda()
        mk = lambda: tq.KVCache(tt, Hkv, D, n_seqs=n, page_tokens=w.page_tokens, page_table=ptd,  # noqa: E731
                                n_pages=n_pages)
    kc = [mk() for _ in range(L)]
    vc = [mk() for _ in range(L)]
    for s in range(n):
        kd = torch.from_numpy(ks[s][:-1]).cuda()
        vd = torch.from_numpy(vs[s][:-1]).cuda()
        for l in range(L):
            tq.encode_kv(kc[l], vc[l], kd, vd, seq_id=s)
    q = torch.from_numpy(np.stack([np.stack([synth.query(w, l, 0, s) for s in range(n)])
                                   for l in range(L)])).cuda()
    kn = torch.from_numpy(np.stack([k[-1] for k in ks])).cuda().reshape(n, Hkv, D)
    vn = torch.from_numpy(np.stack([v[-1] for v in vs])).cuda().reshape(n, Hkv, D)
    out = torch.empty(L, n, Hq, D, device="cuda")
    ws = torch.empty(tq.attn_workspace_bytes(n, Hq, D, max_len), dtype=torch.uint8, device="cuda")
    lens = torch.from_numpy((lens0 + 1).astype(np.int32)).cuda()

    def iteration():
        for l in range(L):
            tq.attn_decode_append(kc[l], vc[l], kn, vn, q[l], lens, max_len, out[l], ws)

    iteration()
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s, capture_error_mode="thread_local"):
        iteration()
    for _ in range(5):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(10):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    call_us = e0.elapsed_time(e1) / (10 * L) * 1e3
    assert lib.tq_phase_trace_clear() == 0
    g.replay()
    torch.cuda.synchronize()
    n_slots, n_points = 4096, 12
    tr = np.zeros((n_slots, n_points), np.uint64)
    assert lib.tq_phase_trace_read(tr.ctypes.data, tr.nbytes) == 0
    att, mrg = tr[:2048].astype(np.int64), tr[2048:].astype(np.int64)
    att, mrg = att[att[:, 1] > 0], mrg[mrg[:, 1] > 0]
    t0 = att[:, 1].min()
    busy = (att[:, 8] - att[:, 1]) / 1e3     # dependency wait to cluster merge done, per CTA
    res = {"probe": f"{w.name} decode-step phases", "ctx": max_len, "layers": L, "n_seqs": n,
           "cta_busy_us": {"sum_over_ctas": round(float(busy.sum()), 1),
                           "sum_with_tiles": round(float(busy[att[:, 5] > 0].sum()), 1),
                           "ctas_with_tiles": int((att[:, 5] > 0).sum())},
           "call_us": call_us, "attention_ctas": int(len(att)), "merge_ctas": int(len(mrg)),
           "phases_us": {}}
    for kind, arr in (("attention", att), ("merge", mrg)):
        for i, name in enumerate(TRACE_PHASES[kind]):
            col = (arr[:, i][arr[:, i] > 0] - t0) / 1e3
            if len(col):
                res["phases_us"][f"{kind}: {name}"] = [round(float(col.min()), 2),
                                                       round(float(np.median(col)), 2),
                                                       round(float(col.max()), 2)]
    print(json.dumps(res, indent=1))


def prefill_probe(args):
    """One layer of the workload's shape: encode a CTX-token prompt's K and V, then run the
    whole prompt (or its last --prefill-chunk queries) as one causal chunk; per-call times from
    CUDA events (not a bench line)."""
    import torch
    import rotated_bit_kv_tq_gb300 as tq
    from rotated_bit_kv_tq_gb300 import build
    build.build()
    w = workload(args.workload)
    tt = w.types[0]
    tq.codebook_init(tt, 0)
    ctx, Hkv, Hq, D = args.prefill_probe, w.n_kv_heads, w.n_q_heads, w.head_dim
    k16 = torch.from_numpy(synth.kv_tokens(w, 0, "K", 0, ctx).reshape(ctx, -1)).cuda()
    v16 = torch.from_numpy(synth.kv_tokens(w, 0, "V", 0, ctx).reshape(ctx, -1)).cuda()
    kc = tq.KVCache(tt, Hkv, D, capacity_tokens=ctx)
    vc = tq.KVCache(tt, Hkv, D, capacity_tokens=ctx)
    tq.encode_kv(kc, vc, k16, v16)
    n_q = args.prefill_chunk or ctx
    pos0 = ctx - n_q
    q = torch.randn(n_q, Hq, D, generator=torch.Generator().manual_seed(5)).half().cuda()
    out = torch.empty(n_q, Hq, D, device="cuda")
    for _ in range(3):
        tq.attn_prefill(kc, vc, q, out, pos0=pos0)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(5):
        tq.attn_prefill(kc, vc, q, out, pos0=pos0)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / 5
    print(json.dumps({"probe": w.name, "prompt": ctx, "chunk": n_q, "pos0": pos0,
                      "prefill_us": ms * 1e3, "tflops": prefill_flops(Hq, D, pos0, n_q) / ms / 1e9,
                      "status": tq.device_status()}))


def main():
    args = parse()
    if args.kernel_probe:
        kernel_probe(args)
        return
    if args.prefill_probe:
        prefill_probe(args)
        return
    if args.phase_trace:
        phase_trace(args)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    import torch
    from rotated_bit_kv_tq_gb300 import build
    build.build()
    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as tdist
        tdist.init_process_group("nccl")
        dist = tdist
    try:
        runs = BENCH_WORKLOADS if args.all else [workload(args.workload)]
        for w in runs:
            for tt in w.types:
                run_ours(args, w, tt, rank, world, local_rank, dist, not args.no_cpu_baseline)
    finally:
        if dist:
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
