"""Kernel microbenchmarks at the workloads' shapes, through the C ABI.

Each case is captured once in a CUDA graph and replayed between CUDA events, with a 256 MB
buffer written before every replay so that the inputs come from HBM (L2 is 129 MB); the
median of the replays is reported.  Inputs are seeded random device tensors (the parity
tests check the results; this only times them).

    python -m bit_compressed_throughput_gb300.microbench gemm      # GEMMs, fused K/V append
    python -m bit_compressed_throughput_gb300.microbench attn      # dense and Top-K decode
    python -m bit_compressed_throughput_gb300.microbench prefill   # causal prefill attention
"""
from __future__ import annotations

import argparse
import math
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

REPS = 15


def time_graph(fn, reps: int = REPS) -> float:
    """Median microseconds of one graph replay of `fn`, L2 flushed before each replay."""
    import torch
    flush = time_graph.flush
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        for _ in range(3):
            fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        fn()
    ts = []
    for _ in range(reps):
        flush.zero_()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    ts.sort()
    return ts[len(ts) // 2] * 1e3


def gemm_cases(fg, torch):
    """opt-6.7b projections: plain GEMMs, the QKV projection with the K/V append in its
    epilogue, and the QKV projection followed by the append kernel."""
    h = 4096
    g = torch.Generator(device="cuda")
    g.manual_seed(5)
    for name, M, K, N, mode in (("qkv prefill", 8192, h, 3 * h, "plain"),
                                ("qkv prefill + kv epilogue", 8192, h, 3 * h, "fused"),
                                ("qkv prefill, then append", 8192, h, 3 * h, "separate"),
                                ("fc1 prefill", 8192, h, 4 * h, "plain"),
                                ("qkv decode", 64, h, 3 * h, "plain"),
                                ("qkv decode + kv epilogue", 64, h, 3 * h, "fused"),
                                ("qkv decode, then append", 64, h, 3 * h, "separate"),
                                ("fc1 decode", 64, h, 4 * h, "plain"),
                                ("o decode (split K + reduce)", 64, h, h, "plain")):
        X = torch.randn((M, K), generator=g, device="cuda").half()
        W = fg.Q4Weight.from_fp16((torch.randn((K, N), generator=g, device="cuda") * 0.02).half())
        bias = torch.zeros(N, dtype=torch.float16, device="cuda")
        Y = torch.empty((M, N), dtype=torch.float16, device="cuda")
        wsb = fg.fg_gemm_workspace_bytes(M, K, N)
        ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device="cuda") if wsb else None
        B, T = (16, 512) if M == 8192 else (64, 1)
        pos = 0 if T > 1 else 520
        cache = fg.KVCacheQ4(B, 1024 if T > 1 else 544, h, 32) if mode != "plain" else None

        if mode == "plain":
            def fn():
                fg.fg_dequant_gemm_q4(X, W, bias, 0, None, Y, ws)
        elif mode == "fused":
            def fn():
                fg.fg_dequant_gemm_q4_kv(X, W, bias, Y, cache, T, pos, ws)
        else:
            def fn():
                fg.fg_dequant_gemm_q4(X, W, bias, 0, None, Y, ws)
                fg.fg_kv_append_q4(Y[:, h:], Y[:, 2 * h:], 3 * h, T, pos, cache)
        us = time_graph(fn)
        fg.fg_check_device_error()
        rate = (f"{2.0 * M * N * K / us / 1e6:7.1f} TFLOP/s" if M > 128 else
                f"{0.5625 * K * N / us / 1e3:7.1f} GB/s of 4-bit weights")
        print(f"gemm  {name:30s} {us:9.1f} us  {rate}", flush=True)


def attn_cases(fg, torch):
    """Dense and Top-K (top 10%) decode attention over a seeded 4-bit cache."""
    import fg_synth
    for B, H, d, length in ((64, 32, 128, 543), (512, 56, 128, 1056)):
        cap = (length + 15) // 16 * 16
        k = max(1, math.ceil(0.1 * length - 1e-9))
        kc, vc, ka, va = fg_synth.random_q4_cache_torch(B, H, cap, d, seed=3)
        cache = fg.KVCacheQ4.__new__(fg.KVCacheQ4)
        cache.B, cache.cap, cache.h, cache.H, cache.d = B, cap, H * d, H, d
        cache.k_codes, cache.v_codes, cache.k_ab, cache.v_ab = kc, vc, ka, va
        q = torch.randn((B, H * d), device="cuda").half()
        out = torch.empty_like(q)
        wsd = fg.fg_decode_attn_workspace_bytes(cache, length)
        wsd_t = torch.empty(max(wsd, 1), dtype=torch.uint8, device="cuda") if wsd else None
        wst = torch.empty(fg.fg_decode_attn_topk_workspace_bytes(cache, length),
                          dtype=torch.uint8, device="cuda")
        scale = 1.0 / math.sqrt(d)
        dense_bytes = 2.0 * B * length * H * d * 0.5625 + 4.0 * B * H * d
        topk_bytes = (B * length * H * d * 0.5625 + B * k * H * d * 0.5625 + 8.0 * B * H * length
                      + 4.0 * B * H * d)
        for name, fn, byts in (
                ("dense", lambda: fg.fg_decode_attn_q4kv(q, H * d, cache, length, scale, out,
                                                         wsd_t), dense_bytes),
                (f"top-{k}", lambda: fg.fg_decode_attn_q4kv_topk(q, H * d, cache, length, k,
                                                                 scale, out, wst), topk_bytes)):
            us = time_graph(fn)
            fg.fg_check_device_error()
            print(f"attn  {B}x{H}x{length:<5d} {name:8s} {us:9.1f} us  "
                  f"{byts / us / 1e3:7.1f} GB/s (algorithmic)", flush=True)


def prefill_cases(fg, torch):
    """Causal prefill attention over fp16 Q/K/V read from a [rows][3h] buffer."""
    for nseq, s, H, d in ((16, 512, 32, 128), (48, 512, 56, 128), (4, 2048, 32, 128)):
        qkv = torch.randn((nseq * s, 3 * H * d), device="cuda").half()
        out = torch.empty((nseq * s, H * d), device="cuda").half()
        us = time_graph(lambda: fg.fg_prefill_attn(qkv, nseq, s, H, d, 1.0 / math.sqrt(d), out))
        fg.fg_check_device_error()
        fl = 2.0 * nseq * H * d * s * (s + 1)
        print(f"prefill {nseq}x{H}x{s:<5d} {us:9.1f} us  {fl / us / 1e6:7.1f} TFLOP/s", flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("cases", nargs="*", help="gemm, attn, prefill (default: all)")
    a = ap.parse_args()
    cases = a.cases or ["gemm", "attn", "prefill"]
    for c in cases:
        if c not in ("gemm", "attn", "prefill"):
            ap.error(f"unknown case {c!r}")
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from bit_compressed_throughput_gb300 import fg
    time_graph.flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    for c in cases:
        {"gemm": gemm_cases, "attn": attn_cases, "prefill": prefill_cases}[c](fg, torch)


if __name__ == "__main__":
    main()
