"""The benchmark's algorithmic byte and FLOP counts, pinned to closed forms.

The roofline fractions bench.py reports divide these counts by measured times, so each is
checked here against a value computed another way: bytes per value from the block sizes
("How small does it get": 50 B and 34 B per 128 values, fp16 in), totals for the Llama-3-8B
KV shape (32 layers, 8 KV heads, head_dim 128, 32,768 tokens), and the causal pair count by
brute force.
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from rotated_bit_kv_tq_gb300 import synth  # noqa: E402


@pytest.mark.parametrize("tq_type,per_value", [(3, 2.390625), (2, 2.265625)])
def test_encode_bytes_per_value(tq_type, per_value):
    w = synth.LLAMA3_8B_32K
    values = 2 * w.n_kv_heads * w.head_dim          # K and V of one token of one layer
    assert bench.encode_bytes_per_token(w, tq_type) == values * per_value


def test_llama_prefill_encode_total():
    w = synth.LLAMA3_8B_32K
    total = w.layers * w.ctx * bench.encode_bytes_per_token(w, 3)
    # 32 layers x 32,768 tokens x 2,048 values x (2 + 50/128) B
    assert total == 32 * 32768 * 2048 * 2 + 32 * 32768 * 16 * 50
    assert abs(total / 1e9 - 5.13) < 0.01


def test_decode_attention_bytes():
    w = synth.LLAMA3_8B_32K
    ctx = 32768
    b = bench.attn_bytes(w, ctx, 3)
    # K and V rows of 8 blocks x 50 B, the fp16 query and the fp32 output of 32 heads
    assert b == ctx * 2 * 8 * 50 + 32 * 128 * 2 + 32 * 128 * 4
    assert abs(w.layers * b / 1e6 - 839) < 1.0       # all layers of one decode step
    # head_dim 256 splits each head vector into two blocks
    w256 = synth.HD256_128K
    assert bench.attn_bytes(w256, 1, 2) == 2 * 4 * 2 * 34 + 16 * 256 * 6


def test_append_bytes():
    w = synth.LLAMA3_8B_32K
    assert bench.append_bytes(w, 3) == 2 * (8 * 128 * 2 + 8 * 50)


@pytest.mark.parametrize("pos0,n_q", [(0, 1), (0, 7), (5, 3), (30720, 16)])
def test_prefill_flops_brute_force(pos0, n_q):
    hq, d = 4, 128
    pairs = sum(pos0 + j + 1 for j in range(n_q))    # query j sees rows 0 .. pos0 + j
    assert bench.prefill_flops(hq, d, pos0, n_q) == 4.0 * hq * d * pairs


def test_job_throughput_sums_ranks_over_slowest():
    assert bench.job_throughput(4, 100, 250.0) == 4 * 100 / 0.25
