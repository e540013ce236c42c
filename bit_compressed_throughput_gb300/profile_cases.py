"""Single-kernel cases for profiler captures: one warm-up launch, then `--reps` launches of
one hot-path kernel at a workload's shape, inputs larger than L2 and a few GB at most.

    python -m bit_compressed_throughput_gb300.profile_cases gemm-fc1-opt67b
    python -m bit_compressed_throughput_gb300.profile_cases decode-attn-opt67b
    python -m bit_compressed_throughput_gb300.profile_cases decode-attn-kv
    python -m bit_compressed_throughput_gb300.profile_cases prefill-attn-opt67b
    python -m bit_compressed_throughput_gb300.profile_cases gemm-prefill-opt175b --reps 0
    python -m bit_compressed_throughput_gb300.profile_cases layer-prefill-opt175b --reps 0

Inputs are seeded random device tensors (no parity check here; the tests do that).
"""
from __future__ import annotations

import argparse
import math
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def gemm_case(M, K, N, epi, reps):
    import torch
    from bit_compressed_throughput_gb300 import fg
    g = torch.Generator(device="cuda")
    g.manual_seed(5)
    X = torch.randn((M, K), generator=g, device="cuda").half()
    W = fg.Q4Weight.from_fp16((torch.randn((K, N), generator=g, device="cuda") * 0.02).half())
    bias = torch.zeros(N, dtype=torch.float16, device="cuda")
    Y = torch.empty((M, N), dtype=torch.float16, device="cuda")
    wsb = fg.fg_gemm_workspace_bytes(M, K, N)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda") if wsb else None
    for _ in range(1 + reps):
        fg.fg_dequant_gemm_q4(X, W, bias, epi, None, Y, ws)
    fg.fg_check_device_error()


def gemm_shapes(shapes, reps):
    """Several GEMM shapes one after the other, each with its own tensors (freed before the
    next shape is allocated)."""
    import torch
    for M, K, N, epi in shapes:
        gemm_case(M, K, N, epi, reps)
        torch.cuda.synchronize()
        torch.cuda.empty_cache()


def attn_case(B, H, d, length, reps, topk=0):
    import torch
    import fg_synth
    from bit_compressed_throughput_gb300 import fg
    cap = (length + 15) // 16 * 16
    kc, vc, ka, va = fg_synth.random_q4_cache_torch(B, H, cap, d, seed=3)
    cache = fg.KVCacheQ4.__new__(fg.KVCacheQ4)
    cache.B, cache.cap, cache.h, cache.H, cache.d = B, cap, H * d, H, d
    cache.k_codes, cache.v_codes, cache.k_ab, cache.v_ab = kc, vc, ka, va
    q = torch.randn((B, H * d), device="cuda").half()
    out = torch.empty_like(q)
    wsb = fg.fg_decode_attn_workspace_bytes(cache, length)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda") if wsb else None
    tws = torch.empty(fg.fg_decode_attn_topk_workspace_bytes(cache, length), dtype=torch.uint8,
                      device="cuda") if topk else None
    for _ in range(1 + reps):
        if topk:
            fg.fg_decode_attn_q4kv_topk(q, H * d, cache, length, topk, 1.0 / math.sqrt(d), out,
                                        tws)
        else:
            fg.fg_decode_attn_q4kv(q, H * d, cache, length, 1.0 / math.sqrt(d), out, ws)
    torch.cuda.synchronize()


def prefill_case(nseq, s, H, d, reps):
    import torch
    from bit_compressed_throughput_gb300 import fg
    g = torch.Generator(device="cuda")
    g.manual_seed(7)
    qkv = torch.randn((nseq * s, 3 * H * d), generator=g, device="cuda").half()
    out = torch.empty((nseq * s, H * d), dtype=torch.float16, device="cuda")
    for _ in range(1 + reps):
        fg.fg_prefill_attn(qkv, nseq, s, H, d, 1.0 / math.sqrt(d), out)
    fg.fg_check_device_error()


def layer_prefill_case(h, H, f, g, s, reps):
    """One decoder layer's prefill over one GPU batch (g sequences of s tokens): the layer
    restores its weights to fp16 once, then runs LN, the four projections (the CTA-pair GEMM
    in its fp16-weight mode), the K/V append and prefill attention."""
    import torch
    from bit_compressed_throughput_gb300 import fg
    gen = torch.Generator(device="cuda")
    gen.manual_seed(9)
    params = {}
    for name, (K, N) in {"wqkv": (h, 3 * h), "wo": (h, h), "w1": (h, f), "w2": (f, h)}.items():
        params[name] = (torch.randn((K, N), generator=gen, device="cuda") * 0.02).half()
    params.update({"bqkv": torch.zeros(3 * h), "bo": torch.zeros(h), "ln1_g": torch.ones(h),
                   "ln1_b": torch.zeros(h), "ln2_g": torch.ones(h), "ln2_b": torch.zeros(h),
                   "b1": torch.zeros(f), "b2": torch.zeros(h)})
    layer = fg.LayerQ4.from_fp16(params, H)
    del params
    torch.cuda.empty_cache()
    eng = fg.StackEngine([layer], g, 1, s, s)
    x = torch.randn((g, s, h), generator=gen, device="cuda").half()
    y = torch.empty_like(x)
    for _ in range(1 + reps):
        eng.prefill(x, y, s)
    fg.fg_check_device_error()


CASES = {
    # 6.7B prefill FC1 of one GPU batch: M = 16*512, K = 4096, N = 16384, ReLU
    "gemm-fc1-opt67b": lambda r: gemm_case(8192, 4096, 16384, 1, r),
    # 6.7B prefill QKV: N = 3*4096
    "gemm-qkv-opt67b": lambda r: gemm_case(8192, 4096, 12288, 0, r),
    # OPT-175B prefill projections of one GPU batch (36 sequences x 512 = 18432 tokens):
    # QKV, O, FC1 (ReLU), FC2 in layer order, at most 2.6 GB on the device at a time
    "gemm-prefill-opt175b": lambda r: gemm_shapes(((18432, 12288, 36864, 0),
                                                   (18432, 12288, 12288, 0),
                                                   (18432, 12288, 49152, 1),
                                                   (18432, 49152, 12288, 0)), r),
    # one OPT-175B layer's prefill over one GPU batch (36 x 512 tokens): ~9 GB on the device
    "layer-prefill-opt175b": lambda r: layer_prefill_case(12288, 96, 49152, 36, 512, r),
    # one opt-6.7b layer's prefill over one GPU batch (16 x 512 tokens): ~2 GB on the device,
    # for multi-pass captures of the fp16-weight GEMM (launches QKV, O, FC1, FC2 in order)
    "layer-prefill-opt67b": lambda r: layer_prefill_case(4096, 32, 16384, 16, 512, r),
    # 6.7B decode FC1 (M = B = 64, split K)
    "gemm-fc1-decode-opt67b": lambda r: gemm_case(64, 4096, 16384, 1, r),
    # 6.7B decode attention at the last step: 64 sequences x 32 heads x 543 positions
    "decode-attn-opt67b": lambda r: attn_case(64, 32, 128, 543, r),
    # KV-dominated workload: 512 sequences x 56 heads x 1056 positions (4.3 GB of cache)
    "decode-attn-kv": lambda r: attn_case(512, 56, 128, 1056, r),
    # a quarter of it (128 sequences, 1.1 GB of cache): the same per-warp work, capture-sized
    "decode-attn-kv-quarter": lambda r: attn_case(128, 56, 128, 1056, r),
    # top-K sparse attention on the quarter KV workload: the top 10% (106 of 1056 positions)
    "decode-attn-topk-kv-quarter": lambda r: attn_case(128, 56, 128, 1056, r, topk=106),
    # 6.7B prefill attention of one GPU batch: 16 sequences x 32 heads x 512 (201 MB of QKV)
    "prefill-attn-opt67b": lambda r: prefill_case(16, 512, 32, 128, r),
    # KV-workload prefill attention, a quarter of one GPU batch: 32 x 56 heads x 1024 (1.3 GB)
    "prefill-attn-kv-quarter": lambda r: prefill_case(32, 1024, 56, 128, r),
    # top-K on the full KV workload (launch lists only: 4.3 GB of cache)
    "decode-attn-topk-kv": lambda r: attn_case(512, 56, 128, 1056, r, topk=106),
}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("case", choices=sorted(CASES))
    ap.add_argument("--reps", type=int, default=2)
    a = ap.parse_args()
    import torch
    import __graft_entry__
    __graft_entry__.build()
    CASES[a.case](a.reps)
    torch.cuda.synchronize()
    print(f"{a.case}: ok")


if __name__ == "__main__":
    main()
