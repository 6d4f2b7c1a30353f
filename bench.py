#!/usr/bin/env python3
"""Benchmark of the rotated, bit-packed KV-cache hot path on GB300.

Workload (default): the Llama-3-8B-shaped KV cache -- 32 layers, 8 KV heads, 32 query
heads, head_dim 128, one sequence, 32,768-token context, turbo3.  One step is the whole
hot path over one batch of synthetic input:
  1. prefill: tq_encode of the K and V of all 32,768 tokens in all 32 layers;
  2. 128 decode iterations; in every layer each one calls tq_attn_decode_append, which
     encodes the new token's K and V into the caches (in the attention launch itself) and
     attends over the grown context.
Metric: decode-attention tokens/s (value) and encode GB/s (encode.gbs), with the
fraction of the measured HBM peak of the dominant kernel (roofline).  Outside the timed
step, "prefill" times prompt-chunk attention (tq_attn_prefill) on the last 2,048-token
chunk of the prompt in every layer, with its tensor roofline.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (oracle/) on a bounded sample of the same workload.
Under torchrun every rank runs an independent replica (the path has no data exchange);
value is the sum over ranks, time the max over ranks.
"""
from __future__ import annotations

import argparse
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

# DRAM bytes per token measured by ncu (dram__bytes_read.sum + dram__bytes_write.sum) on the
# 262,144-token probe of the same kernels (profiles/*_262k.md), scaled to a launch by its
# token count: attention reads every packed row once, encode reads fp16 and writes packed rows,
# so traffic grows in proportion to tokens.  None once a kernel changes after its capture.
TRAFFIC_PER_TOKEN = {"attn": 212.85e6 / 262144, "encode": 627.06e6 / 262144}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=synth.LLAMA3_8B_32K.name,
                    choices=[w.name for w in synth.WORKLOADS])
    ap.add_argument("--kernel-probe", type=int, default=0, metavar="CTX",
                    help="time one layer's encode and attention at context CTX (the small "
                         "case the ncu captures use) instead of the full benchmark")
    ap.add_argument("--prefill-probe", type=int, default=0, metavar="CTX",
                    help="time one layer's prompt attention over a whole CTX-token prompt "
                         "(one chunk from position 0; the small case of the prefill capture)")
    return ap.parse_args()


def workload(name):
    return {w.name: w for w in synth.WORKLOADS}[name]


# ------------------------------------------------------------------ accounting

def encode_bytes_per_token(w, tq_type=3):
    """Algorithmic bytes of encoding one token of one layer (K and V): fp16 in + packed out."""
    vals = w.n_kv_heads * w.head_dim
    packed = w.n_kv_heads * (w.head_dim // 128) * (2 + 128 * tq_type // 8)
    return 2 * (2 * vals + packed)


def attn_bytes(w, ctx, tq_type=3):
    """Algorithmic bytes of one decode-attention launch (one layer, one sequence)."""
    row = w.n_kv_heads * (w.head_dim // 128) * (2 + 128 * tq_type // 8)
    return ctx * 2 * row + w.n_q_heads * w.head_dim * (2 + 4)


def append_bytes(w, tq_type=3):
    """Algorithmic bytes of the decode-step append (one layer, one sequence): the new
    token's fp16 K and V read, one packed row of each written."""
    row = w.n_kv_heads * (w.head_dim // 128) * (2 + 128 * tq_type // 8)
    return 2 * (w.n_kv_heads * w.head_dim * 2 + row)


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

def make_inputs(w, torch, pin):
    """Host fp16 inputs: prefill K/V [L][2][T][row], appended tokens [S][L][2][row],
    queries [S][L][Hq][D]."""
    L, T, row = w.layers, w.ctx, w.n_kv_heads * w.head_dim
    kv = torch.empty((L, 2, T, row), dtype=torch.float16, pin_memory=pin)
    new = torch.empty((DECODE_STEPS, L, 2, row), dtype=torch.float16, pin_memory=pin)
    q = torch.empty((DECODE_STEPS, L, w.n_q_heads, w.head_dim), dtype=torch.float16, pin_memory=pin)
    for l in range(L):
        for j, kind in enumerate("KV"):
            kv[l, j].copy_(torch.from_numpy(synth.kv_tokens(w, l, kind, 0, T).reshape(T, row)))
            new[:, l, j].copy_(torch.from_numpy(synth.kv_tokens(w, l, kind, T, DECODE_STEPS)
                                                .reshape(DECODE_STEPS, row)))
        for s in range(DECODE_STEPS):
            q[s, l].copy_(torch.from_numpy(synth.query(w, l, s)))
    return kv, new, q


# ------------------------------------------------------------------ our CUDA path

def run_ours(args, rank, world, local_rank, dist):
    import torch
    import rotated_bit_kv_tq_gb300 as tq
    from rotated_bit_kv_tq_gb300 import build
    build.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    w = workload(args.workload)
    if w.n_seqs != 1:
        raise SystemExit("bench.py times the single-sequence workloads")
    tt = w.types[0]
    tq.codebook_init(tt, local_rank)
    L, T, Hkv, Hq, D, S = w.layers, w.ctx, w.n_kv_heads, w.n_q_heads, w.head_dim, DECODE_STEPS
    row = Hkv * D
    max_len = T + S

    t_gen = time.time()
    kv_host, new_host, q_host = make_inputs(w, torch, pin=True)
    t_gen = time.time() - t_gen
    kv_dev = kv_host.to(dev)
    new_dev = new_host.to(dev)
    q_dev = q_host.to(dev)
    kc = [tq.KVCache(tt, Hkv, D, capacity_tokens=max_len, device=dev) for _ in range(L)]
    vc = [tq.KVCache(tt, Hkv, D, capacity_tokens=max_len, device=dev) for _ in range(L)]
    out_dev = torch.zeros((L, Hq, D), dtype=torch.float32, device=dev)
    ws = torch.empty(max(16, tq.attn_workspace_bytes(1, Hq, D, max_len)), dtype=torch.uint8, device=dev)
    lens_dev = torch.zeros(1, dtype=torch.int32, device=dev)
    step_dev = torch.zeros(1, dtype=torch.int64, device=dev)
    new_buf = torch.empty((1, L, 2, row), dtype=torch.float16, device=dev)
    q_buf = torch.empty((1, L, Hq, D), dtype=torch.float16, device=dev)

    def prefill():
        for l in range(L):
            tq.encode_kv(kc[l], vc[l], kv_dev[l, 0], kv_dev[l, 1])
        lens_dev.fill_(T + 1)
        step_dev.zero_()

    def decode_iter():
        torch.index_select(new_dev, 0, step_dev, out=new_buf)
        torch.index_select(q_dev, 0, step_dev, out=q_buf)
        for l in range(L):
            tq.attn_decode_append(kc[l], vc[l], new_buf[0, l, 0:1], new_buf[0, l, 1:2],
                                  q_buf[0, l:l + 1], lens_dev, max_len, out_dev[l:l + 1], ws)
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
    # and in the same state: each call is replayed from a CUDA graph of the 32 layers' calls
    # (as in the timed step), bracketed by CUDA events on the replay stream.  The decode
    # step re-appends the last iteration's token at the last position (the same bytes).
    lens_dev.fill_(max_len)
    g_att, g_enc = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_att, stream=cap, capture_error_mode="thread_local"):
        for l in range(L):
            tq.attn_decode_append(kc[l], vc[l], new_buf[0, l, 0:1], new_buf[0, l, 1:2],
                                  q_buf[0, l:l + 1], lens_dev, max_len, out_dev[l:l + 1], ws)
    with torch.cuda.graph(g_enc, stream=cap, capture_error_mode="thread_local"):
        for l in range(L):   # the prefill's own call: K and V of one layer in one launch
            tq.encode_kv(kc[l], vc[l], kv_dev[l, 0], kv_dev[l, 1])

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
    # (the encode graph rewrites the prefill rows with identical codes; rows >= T keep the
    #  decoded tokens)

    # prompt-chunk attention (tensor-bound, timed alone): the last PREFILL_CHUNK queries of
    # the prompt, positions T - PREFILL_CHUNK .. T - 1, over every layer's cache
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

    # end to end through the public API with host buffers: pinned host -> device copies of
    # every step's inputs and device -> host reads of every decode iteration's output
    out_host = torch.empty((S, L, Hq, D), dtype=torch.float32, pin_memory=True)
    e2e_evs = []
    for k in range(max(1, args.steps)):
        ea, eb, ec = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        ea.record()
        kv_dev.copy_(kv_host, non_blocking=True)
        g_pre.replay()
        eb.record()
        for i in range(S):
            new_dev[i].copy_(new_host[i], non_blocking=True)
            q_dev[i].copy_(q_host[i], non_blocking=True)
            g_dec.replay()
            out_host[i].copy_(out_dev, non_blocking=True)
        ec.record()
        e2e_evs.append((ea, eb, ec))
    torch.cuda.synchronize()
    e2e_pre_ms = sum(a.elapsed_time(b) for a, b, _ in e2e_evs)
    e2e_dec_ms = sum(b.elapsed_time(c) for _, b, c in e2e_evs)
    n_e2e = len(e2e_evs)
    assert np.isfinite(out_host.numpy()).all()

    if dist:
        pre_ms, dec_ms, e2e_pre_ms, e2e_dec_ms = reduce_max(
            [pre_ms, dec_ms, e2e_pre_ms, e2e_dec_ms], dist, dev)
    if rank != 0:
        return

    K = args.steps
    enc_bytes = encode_bytes_per_token(w, tt) * T * L
    value = job_throughput(world, K * S, dec_ms)
    enc_gbs = world * K * enc_bytes / (pre_ms / 1e3) / 1e9
    peak, peak_kind = measured_peak_hbm()
    a_bytes = attn_bytes(w, max_len, tt) + append_bytes(w, tt)
    a_gbs = a_bytes / (attn_launch_ms / 1e3) / 1e9
    e_bytes = encode_bytes_per_token(w, tt) * T          # K and V of one layer
    e_gbs = e_bytes / (enc_launch_ms / 1e3) / 1e9
    h2d = kv_host.numel() * 2 + S * (new_host[0].numel() + q_host[0].numel()) * 2
    tpeak, tpeak_kind = measured_peak_tensor()
    pf_tflops = prefill_flops(Hq, D, pf_pos0, PREFILL_CHUNK) * L / (pf_ms / 1e3) / 1e12
    d2h = S * L * Hq * D * 4
    line = {
        "metric": "turbo3 decode-attn tokens/s & encode GB/s at 32K ctx; % of HBM peak",
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": (pre_ms + dec_ms) / K,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32 (fp16 in, 3-bit codes)",
        "data": "synthetic (seeded; K with lognormal channel scales and x10 outlier channels)",
        "config": {"workload": w.name, "layers": L, "n_kv_heads": Hkv, "n_q_heads": Hq,
                   "head_dim": D, "ctx": T, "decode_steps": S, "cache_type": f"turbo{tt}",
                   "batch": 1, "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2: 0.84 GB packed cache read per decode iteration, "
                         "4.3 GB fp16 read per prefill"},
        "encode": {"gbs": enc_gbs, "tokens_per_s": world * K * T * L / (pre_ms / 1e3),
                   "ms_per_step": pre_ms / K},
        "decode_ms_per_step": dec_ms / K,
        "roofline": {"kernel": "tq_attn_decode_append (append + split-K partial + merge)",
                     "bound": "hbm",
                     "achieved": a_gbs, "peak": peak, "unit": "GB/s", "frac": a_gbs / peak,
                     "peak_source": peak_kind,
                     "traffic": TRAFFIC_PER_TOKEN["attn"] * max_len if TRAFFIC_PER_TOKEN["attn"] else None,
                     "bytes_per_launch": a_bytes, "launch_ms": attn_launch_ms},
        "encode_roofline": {"kernel": "tq_encode_kv (prefill, one layer, K and V)", "bound": "hbm",
                            "achieved": e_gbs, "peak": peak, "unit": "GB/s", "frac": e_gbs / peak,
                            "peak_source": peak_kind, "bytes_per_launch": e_bytes,
                            "traffic": 2 * TRAFFIC_PER_TOKEN["encode"] * T if TRAFFIC_PER_TOKEN["encode"] else None,
                            "launch_ms": enc_launch_ms},
        "e2e": {"value": world * n_e2e * S / (e2e_dec_ms / 1e3), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "encode_gbs": world * n_e2e * enc_bytes / (e2e_pre_ms / 1e3) / 1e9},
        "prefill": {
            "metric": f"prompt-chunk attention tokens/s ({PREFILL_CHUNK}-token chunk at position "
                      f"{pf_pos0}, {L} layers)",
            "value": PREFILL_CHUNK / (pf_ms / 1e3), "unit": "tokens/s", "ms": pf_ms,
            "roofline": {"kernel": "tq_attn_prefill", "bound": "tensor",
                         "achieved": pf_tflops, "peak": tpeak, "unit": "TFLOP/s",
                         "frac": pf_tflops / tpeak, "peak_source": tpeak_kind, "traffic": None,
                         "flops_per_launch": prefill_flops(Hq, D, pf_pos0, PREFILL_CHUNK),
                         "launch_ms": pf_ms / L}},
        "gpu_launches": K * (L + S * L * 2),
        "clocks": clk,
        "device_status": status,
        "input_gen_s": t_gen,
    }
    if world == 1:
        line["cpu_baseline"] = cpu_baseline(w, tt)
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ the oracle on the host

def cpu_baseline(w, tt, layers_sample=1):
    """The oracle (single-threaded C) on a bounded sample of the workload: the prefill
    encode of one layer's K and V (full context) and one decode-attention step of that
    layer over the full context; tokens/s scales the per-layer time by the layer count."""
    import oracle
    oracle.build()
    T, Hkv, Hq, D = w.ctx, w.n_kv_heads, w.n_q_heads, w.head_dim
    row = Hkv * D
    k16 = synth.kv_tokens(w, 0, "K", 0, T + 1).reshape(T + 1, row)
    v16 = synth.kv_tokens(w, 0, "V", 0, T + 1).reshape(T + 1, row)
    q16 = synth.query(w, 0, 0)
    t0 = time.perf_counter()
    kr = oracle.encode_rows(tt, k16, Hkv, D)
    vr = oracle.encode_rows(tt, v16, Hkv, D)
    t_enc = time.perf_counter() - t0
    t0 = time.perf_counter()
    for _ in range(layers_sample):
        oracle.attn_decode(tt, tt, kr, vr, q16, T + 1, Hq, Hkv, D, 1.0 / np.sqrt(D))
    t_attn = (time.perf_counter() - t0) / layers_sample
    enc_bytes = encode_bytes_per_token(w, tt) * (T + 1)
    return {"value": 1.0 / (t_attn * w.layers), "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"1 layer of {w.name}: encode of K and V over {T + 1} tokens, then "
                      f"{layers_sample} decode-attention step(s) over {T + 1} tokens; tokens/s = "
                      f"1 / (per-layer time x {w.layers} layers)",
            "encode_gbs": enc_bytes / t_enc / 1e9, "seconds": t_enc + t_attn * layers_sample}


def run_reference(args, rank, world):
    """The reference arm: the oracle, as it stands, on the host cores."""
    if rank != 0:
        return
    w = workload(args.workload)
    tt = w.types[0]
    for _ in range(args.warmup and 1):
        pass
    vals, secs = [], 0.0
    base = None
    for _ in range(max(1, args.steps)):
        base = cpu_baseline(w, tt)
        vals.append(base["value"])
        secs += base["seconds"]
        if secs > 150:
            break
    value = statistics.mean(vals)
    base["value"] = value
    line = {
        "impl": "reference",
        "metric": "turbo3 decode-attn tokens/s & encode GB/s at 32K ctx; % of HBM peak",
        "value": value, "unit": "tokens/s", "n_gpus": world, "steps": len(vals),
        "warmup": args.warmup, "ms_per_step": 1e3 * secs / len(vals), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)", "data": "synthetic",
        "config": {"workload": w.name, "layers": w.layers, "n_kv_heads": w.n_kv_heads,
                   "n_q_heads": w.n_q_heads, "head_dim": w.head_dim, "ctx": w.ctx,
                   "cache_type": f"turbo{tt}", "batch": 1},
        "cpu_baseline": base,
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def kernel_probe(args):
    """One layer of the workload's shape at context args.kernel_probe: encode of K and V,
    then repeated decode attention; per-call times from CUDA events (not a bench line)."""
    import torch
    import rotated_bit_kv_tq_gb300 as tq
    from rotated_bit_kv_tq_gb300 import build
    build.build()
    w = workload(args.workload)
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

    def timed(fn, n):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(n):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n

    for _ in range(3):
        tq.encode(kc, k16)
        tq.encode(vc, v16)
        tq.attn_decode(kc, vc, q, lens, ctx, out, ws)
    torch.cuda.synchronize()
    enc_ms = timed(lambda: tq.encode(kc, k16), 10)
    att_ms = timed(lambda: tq.attn_decode(kc, vc, q, lens, ctx, out, ws), 20)
    enc_b = ctx * (Hkv * D * 2 + kc.row_bytes)
    att_b = attn_bytes(w, ctx, tt)
    print(json.dumps({"probe": w.name, "ctx": ctx, "encode_us": enc_ms * 1e3,
                      "encode_gbs": enc_b / enc_ms / 1e6, "attn_us": att_ms * 1e3,
                      "attn_gbs": att_b / att_ms / 1e6, "status": tq.device_status()}))


def prefill_probe(args):
    """One layer of the workload's shape: encode a CTX-token prompt's K and V, then run the
    whole prompt as one causal chunk; per-call times from CUDA events (not a bench line)."""
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
    q = torch.randn(ctx, Hq, D, generator=torch.Generator().manual_seed(5)).half().cuda()
    out = torch.empty(ctx, Hq, D, device="cuda")
    for _ in range(3):
        tq.attn_prefill(kc, vc, q, out, pos0=0)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(5):
        tq.attn_prefill(kc, vc, q, out, pos0=0)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / 5
    print(json.dumps({"probe": w.name, "prompt": ctx, "prefill_us": ms * 1e3,
                      "tflops": prefill_flops(Hq, D, 0, ctx) / ms / 1e9,
                      "status": tq.device_status()}))


def main():
    args = parse()
    if args.kernel_probe:
        kernel_probe(args)
        return
    if args.prefill_probe:
        prefill_probe(args)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    dist = None
    if world > 1:
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(local_rank)
        tdist.init_process_group("nccl")
        dist = tdist
    try:
        run_ours(args, rank, world, local_rank, dist)
    finally:
        if dist:
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
