"""The analytical cost model as a predictor (host logic, no GPU).

Pins: the pages' block formula T = T_pre*l + T_gen*(n-1)*l and its max-over-paths phase
latency [FlexGen paper explainer, "Analytical Cost Model"], checked through the predictor's
outputs rather than by retyping them; the invariants that relate the two granularities; and
the per-kernel work it sums, checked against independent closed forms of the layer's shapes.
"""
import dataclasses
import math

import pytest

import fg_synth
from bit_compressed_throughput_gb300 import cost_model as C

HW = C.Hardware(hbm_bytes_per_s=6.69e12, tensor_flops=1.915e15)


def test_single_token_generation_is_prefill_only():
    # n = 1: the block is prefill alone, T = T_pre * l (no decoding steps)
    wl = fg_synth.WORKLOADS["opt-6.7b"].with_(n=1)
    p = C.predict(wl, HW)
    assert p["T_block_s"] == pytest.approx(p["T_pre_s"] * wl.L, rel=1e-12)


def test_decoding_steps_add_linearly():
    # each further generated token adds one decoding step per layer, at the average cache
    # length: T(n) - T_pre*l is (n-1) * T_gen(n) * l
    wl = fg_synth.WORKLOADS["opt-6.7b"]
    for n in (2, 9, 33):
        p = C.predict(wl.with_(n=n), HW)
        assert p["T_block_s"] - p["T_pre_s"] * wl.L == pytest.approx((n - 1) * p["T_gen_s"] * wl.L,
                                                                     rel=1e-12)


def test_phase_latency_is_the_slowest_path():
    ops = [C.Op("a", bytes=6.69e9, flops=0.0), C.Op("b", bytes=0.0, flops=3.83e12)]
    # layer form: max(6.69e9 B / 6.69e12 B/s, 3.83e12 / 1.915e15) = max(1 ms, 2 ms)
    assert C.phase_time(ops, HW, "layer") == pytest.approx(2e-3)
    # kernel form: each kernel bounded by its own path, then summed: 1 ms + 2 ms
    assert C.phase_time(ops, HW, "kernel") == pytest.approx(3e-3)


@pytest.mark.parametrize("name", ["tiny", "opt-6.7b", "opt-30b", "opt-175b", "kv-decode"])
def test_overlap_bound_is_faster(name):
    # max of sums <= sum of maxes: assuming perfect overlap across a layer can only predict
    # more throughput than kernel-by-kernel execution
    wl = fg_synth.WORKLOADS[name]
    assert C.predict(wl, HW, "layer")["tokens_per_s"] >= C.predict(wl, HW, "kernel")["tokens_per_s"]
    # the auxiliary kernels (LayerNorm, KV append) only add time
    assert (C.predict(wl, HW, include_aux=False)["tokens_per_s"]
            >= C.predict(wl, HW, include_aux=True)["tokens_per_s"])


def test_layer_work_matches_the_shapes():
    # flops of one prefill layer of the 6.7B shape, from the layer's matrix shapes:
    # QKV (3h x h), O (h x h), FC1 (f x h), FC2 (h x f) over B*s rows, plus causal attention
    wl = fg_synth.WORKLOADS["opt-6.7b"]
    B, s, h, f = wl.B, wl.s, wl.h, wl.f
    ops = C.layer_ops(h, f, wl.H, B * s, B, s, "prefill", include_aux=False)
    gemm = 2.0 * B * s * (3 * h * h + h * h + 2 * h * f)
    attn = 4.0 * B * h * sum(t + 1 for t in range(s))          # QK^T and PV, row t sees t+1
    assert sum(o.flops for o in ops) == pytest.approx(gemm + attn, rel=1e-12)
    # decoding-step bytes: 4-bit weights of the layer, the 4-bit K and V of kv_len positions,
    # fp16 activations in and out of each kernel
    L = 528.0
    ops = C.layer_ops(h, f, wl.H, B, B, L, "decode", include_aux=False)
    w4 = (4 * h * h + 2 * h * f) * (0.5 + 4 / 64)
    kv4 = 2 * B * L * h * (0.5 + 4 / 64)
    act = 2 * B * (h + 3 * h) + 4 * B * h + 2 * B * (h + h + h) + 2 * B * (h + f) + 2 * B * (f + h + h)
    assert sum(o.bytes for o in ops) == pytest.approx(w4 + kv4 + act, rel=1e-12)


def test_decode_is_hbm_bound_and_prefill_gemms_tensor_bound_at_the_6p7b_shape():
    # the 6.7B decode GEMMs (M = 64, 228 flop per weight byte) sit left of the ridge
    # (1.915 PF / 6.69 TB/s ~ 286 flop/B); the prefill GEMMs (M = 8192) far right of it
    bn = C.bottlenecks(fg_synth.WORKLOADS["opt-6.7b"], HW)
    assert dict((k, b) for k, b, _ in bn["decode"])["fc1"] == "hbm"
    assert dict((k, b) for k, b, _ in bn["decode"])["attention"] == "hbm"
    assert dict((k, b) for k, b, _ in bn["prefill"])["fc1"] == "tensor"


def test_layer_scale_multiplies_the_block():
    wl = fg_synth.WORKLOADS["opt-175b"]
    p = C.predict(wl, HW)
    q = C.predict(dataclasses.replace(wl, layer_scale=1.0), HW)
    assert p["T_block_s"] == pytest.approx(q["T_block_s"] * 12.0)
    assert math.isfinite(p["tokens_per_s"]) and p["tokens_per_s"] > 0
