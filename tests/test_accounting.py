"""The benchmark's algorithmic byte counts reproduce the figures the FlexGen pages
print (tests/golden/flexgen_closed_forms.json, each entry cited there)."""
import json
import os

import pytest

from bit_compressed_throughput_gb300 import accounting as A

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                   "flexgen_closed_forms.json")))


def test_fp16_layer_weight_formula():
    # the cost model's 8*h1^2 + 4*h1*h2
    assert A.fp16_layer_weight_bytes(3, 5) == 8 * 9 + 4 * 15
    d = GOLD["opt175b_dims"]
    w = A.fp16_layer_weight_bytes(d["h1"], d["h2"]) * d["layers"]
    assert abs(w / 2 ** 30 / GOLD["weights_175b_fp16"]["printed_GB"] - 1) < 0.01   # "approximately"


def test_kv_cache_175b():
    d, g = GOLD["opt175b_dims"], GOLD["kv_cache_175b"]
    kv = A.kv_cache_bytes(d["layers"], g["batch"], g["prompt"] + g["gen"], d["h1"])
    assert round(kv / 2 ** 40, 1) == g["printed_TB"]
    w = A.fp16_layer_weight_bytes(d["h1"], d["h2"]) * d["layers"]
    assert round(kv / w, 1) == g["printed_ratio_to_weights"]


def test_int4_weights_175b():
    d = GOLD["opt175b_dims"]
    codes_only = A.layer_weight_elems(d["h1"], d["h2"]) * d["layers"] * 0.5
    assert abs(codes_only / 1e9 - GOLD["weights_175b_int4"]["printed_GB"]) < 1.0
    # with the (a, b) fp16 pair per group of 64: 0.5625 bytes per element
    assert A.q4_bytes(64) == 36.0


def test_block_reuse_example():
    g = GOLD["block_reuse_example"]
    assert A.weight_traffic(g["layers"], g["layer_GB"], g["gpu_batches"], False) == g["row_by_row_GB"]
    assert A.weight_traffic(g["layers"], g["layer_GB"], g["gpu_batches"], True) == g["block_GB"]


def test_delegation_ratio():
    g = GOLD["delegation_ratio"]
    assert A.delegation_io_ratio(g["b"], g["s"], g["h1"]) == g["ratio"]


def test_average_kv_over_decoding():
    # 4*bls*(s+n/2)*h1 equals the mean of the exact per-step sizes to first order
    bls, s, n, h1 = 8, 512, 32, 64
    exact = sum(4.0 * bls * (s + t) * h1 for t in range(n + 1)) / (n + 1)
    assert abs(A.kv_cache_bytes_avg_decode(bls, s, n, h1) - exact) / exact < 1e-12


def test_topk_attention_bytes():
    # keeping every position reads what dense attention reads, plus the score keys; keeping
    # a tenth saves 90% of the V bytes (the KV-dominated workload: 512 x 56 heads x 1056)
    B, H, d, T = 512, 56, 128, 1056
    h = H * d
    dense = A.decode_attn_bytes(B, T, h)
    assert A.decode_attn_topk_bytes(B, H, T, T, h) == pytest.approx(dense + 8.0 * B * H * T)
    v = A.q4_bytes(B * T * h)
    saved = dense + 8.0 * B * H * T - A.decode_attn_topk_bytes(B, H, T, 106, h)
    assert saved == pytest.approx(v * (1 - 106 / T))
