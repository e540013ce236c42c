"""Kernel-level parity of libfg against the CPU oracle, through the C ABI.

Integer outputs (codes, group statistics) must be bit-exact; floating outputs must meet
max |err| <= 2e-2 * max |ref| + 1e-3.  Cases span several tiles, ragged tails, the
degenerate sizes and, on sampled rows / sequences, the full workload sizes.
"""
import math

import numpy as np
import pytest
import torch

import fg_synth
from oracle import layer as OL
from oracle import quant as OQ
from parity_util import assert_close, cache_codes_to_rows, dev, f16, host, lib, rows_to_cache

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fg():
    return lib()


def gpu_quantize(fg, x16):
    x = dev(x16)
    R, Cc = x16.shape
    codes = torch.empty((R, Cc // 2), dtype=torch.uint8, device="cuda")
    ab = torch.empty((R, Cc // 64), dtype=torch.int32, device="cuda")
    fg.fg_quantize_g64(x, codes, ab)
    return codes, ab


def oracle_packed(x16):
    q, a, b = OQ.quantize_g64(x16)
    return OQ.pack_nibbles(q), OQ.ab_pack_u32(a, b)


# ----------------------------------------------------------------------------- quantise


@pytest.mark.parametrize("shape,scale", [((1, 64), 1.0), ((7, 192), 0.02), ((300, 4160), 3.0),
                                         ((1025, 128), 1e-4), ((33, 64 * 37), 100.0)])
def test_quantize_bit_exact(fg, shape, scale):
    x16 = fg_synth.random_fp16(shape, seed=shape[0] * 7 + shape[1], scale=scale, offset=scale / 3)
    codes, ab = gpu_quantize(fg, x16)
    c_ref, ab_ref = oracle_packed(x16)
    assert np.array_equal(host(codes), c_ref)
    assert np.array_equal(host(ab).view(np.uint32), ab_ref)


def test_quantize_adversarial_groups(fg):
    x16 = fg_synth.adversarial_groups_fp16()
    codes, ab = gpu_quantize(fg, x16)
    c_ref, ab_ref = oracle_packed(x16)
    assert np.array_equal(host(codes), c_ref)
    assert np.array_equal(host(ab).view(np.uint32), ab_ref)


def test_quantize_empty_is_noop(fg):
    codes = torch.full((4, 32), 7, dtype=torch.uint8, device="cuda")
    ab = torch.zeros((4, 1), dtype=torch.int32, device="cuda")
    fg.fg_quantize_g64(torch.empty((0, 64), dtype=torch.float16, device="cuda"), codes, ab)
    torch.cuda.synchronize()
    assert int(codes.min()) == 7


@pytest.mark.parametrize("wl_name,which", [("opt-30b", "w1"), ("opt-175b", "w1")])
def test_quantize_full_size_sampled_rows(fg, wl_name, which):
    """A full weight of the workload (30B: with outlier input channels), quantised on the
    device; sampled rows checked bit-exact against the oracle."""
    wl = fg_synth.WORKLOADS[wl_name]
    w = fg_synth.weight_fp16(wl.h, wl.f, wl, 0, fg_synth.T_W1)
    codes, ab = gpu_quantize(fg, w)
    rows = np.unique(np.r_[0, wl.h - 1, np.random.Generator(np.random.PCG64(1)).integers(
        0, wl.h, 30)])
    c_ref, ab_ref = oracle_packed(w[rows])
    assert np.array_equal(host(codes[torch.from_numpy(rows).cuda()]), c_ref)
    assert np.array_equal(host(ab[torch.from_numpy(rows).cuda()]).view(np.uint32), ab_ref)


def test_dequant_bit_exact(fg):
    x16 = np.concatenate([fg_synth.random_fp16((40, 256), 5, 2.0),
                          fg_synth.adversarial_groups_fp16().reshape(4, 256)])
    codes, ab = gpu_quantize(fg, x16)
    y = torch.empty(x16.shape, dtype=torch.float16, device="cuda")
    fg.fg_dequant_g64(codes, ab, x16.shape[0], x16.shape[1], y)
    q, a, b = OQ.quantize_g64(x16)
    ref = OQ.dequant_g64(q, a, b)
    assert np.array_equal(host(y).view(np.uint16), ref.view(np.uint16))


# ----------------------------------------------------------------------------- KV append


@pytest.mark.parametrize("B,T,pos,h,H,cap", [(3, 5, 2, 256, 4, 9), (2, 1, 15, 512, 4, 16),
                                              (4, 33, 0, 1024, 8, 40)])
def test_kv_append_bit_exact(fg, B, T, pos, h, H, cap):
    qkv16 = fg_synth.random_fp16((B * T, 3 * h), seed=B * 100 + T, scale=2.0)
    qkv = dev(qkv16)
    cache = fg.KVCacheQ4(B, cap, h, H)
    fg.fg_kv_append_q4(qkv[:, h:], qkv[:, 2 * h:], 3 * h, T, pos, cache)
    for src, codes_t, ab_t in ((qkv16[:, h:2 * h], cache.k_codes, cache.k_ab),
                               (qkv16[:, 2 * h:], cache.v_codes, cache.v_ab)):
        c_ref, ab_ref = oracle_packed(np.ascontiguousarray(src))
        got_c = cache_codes_to_rows(host(codes_t))
        got_ab = cache_codes_to_rows(host(ab_t)).view(np.uint32)
        assert np.array_equal(got_c[:, pos:pos + T].reshape(B * T, h // 2), c_ref)
        assert np.array_equal(got_ab[:, pos:pos + T].reshape(B * T, h // 64), ab_ref)
        untouched = np.ones(cache.cap, bool)
        untouched[pos:pos + T] = False
        assert not got_c[:, untouched].any() and not got_ab[:, untouched].any()


# ----------------------------------------------------------------------------- LayerNorm


@pytest.mark.parametrize("rows,h", [(1, 256), (37, 4096), (5, 7168), (3, 12288), (2, 16384)])
def test_layernorm(fg, rows, h):
    x16 = fg_synth.random_fp16((rows, h), seed=rows + h, scale=3.0, offset=1.0)
    g16 = fg_synth.random_fp16((h,), seed=h + 1, scale=0.1, offset=1.0)
    b16 = fg_synth.random_fp16((h,), seed=h + 2, scale=0.1)
    y = torch.empty((rows, h), dtype=torch.float16, device="cuda")
    fg.fg_layernorm(dev(x16), dev(g16), dev(b16), 1e-5, y)
    ref = OL.layernorm(x16, g16, b16, 1e-5)
    assert_close(f16(y), ref, f"layernorm {rows}x{h}")


# ----------------------------------------------------------------------------- GEMM


def gemm_case(fg, M, K, N, epi, with_bias, seed, alias=False):
    x16 = fg_synth.random_fp16((M, K), seed, 1.0)
    w16 = fg_synth.random_fp16((K, N), seed + 1, 0.02)
    bias16 = fg_synth.random_fp16((N,), seed + 2, 0.1) if with_bias else None
    res16 = fg_synth.random_fp16((M, N), seed + 3, 1.0) if epi == 2 else None
    W = fg.Q4Weight.from_fp16(dev(w16))
    # the device quantiser is bit-exact with the oracle (checked above); re-check here
    c_ref, ab_ref = oracle_packed(w16)
    assert np.array_equal(host(W.codes), c_ref)
    X = dev(x16)
    bias = dev(bias16) if with_bias else None
    res = dev(res16) if res16 is not None else None
    Y = res if alias else torch.empty((M, N), dtype=torch.float16, device="cuda")
    wsb = fg.fg_gemm_workspace_bytes(M, K, N)
    ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device="cuda") if wsb else None
    fg.fg_dequant_gemm_q4(X, W, bias, epi, res, Y, ws)
    fg.fg_check_device_error()
    q, a, b = OQ.quantize_g64(w16)
    what = OQ.dequant_g64(q, a, b).astype(np.float64)
    ref = x16.astype(np.float64) @ what
    if with_bias:
        ref += bias16.astype(np.float64)
    if epi == 1:
        ref = np.maximum(ref, 0)
    elif epi == 2:
        ref += res16.astype(np.float64)
    got = f16(Y)
    assert_close(got, ref, f"gemm M={M} K={K} N={N} epi={epi}")
    # a tighter statistical check: relative RMS error at fp16 output precision
    rms = np.sqrt(np.mean((got - ref) ** 2)) / max(np.sqrt(np.mean(ref ** 2)), 1e-30)
    assert rms < 3e-3, f"relative rms error {rms:.3g}"
    return wsb


@pytest.mark.parametrize("M,K,N,epi,bias", [
    (1, 64, 256, 0, False),         # single row, single tile
    (4, 256, 768, 0, True),         # tiny decode QKV (split K)
    (32, 256, 1024, 1, True),       # tiny prefill FC1
    (200, 1024, 768, 2, True),      # ragged M, three n tiles
    (130, 80, 512, 0, False),       # K ragged inside a 64-block
    (300, 512, 2048, 1, False),     # several m tiles in one raster group
    (1100, 256, 256, 0, True),      # 9 m tiles (two raster groups)
    (48, 320, 512, 1, True),        # odd k-block count split over two MMA issuers
    (64, 1344, 256, 2, True),       # split K with an odd number of k-blocks per split
])
def test_gemm_small(fg, M, K, N, epi, bias):
    gemm_case(fg, M, K, N, epi, bias, seed=M * 31 + K + N)


@pytest.mark.parametrize("M,K,N,epi,bias", [
    (128, 4096, 4096, 2, True),     # largest token tile of the streaming kernel, split K
    (127, 208, 512, 1, True),       # ragged M and K (three k-blocks and 16 rows)
    (16, 16, 256, 0, False),        # a single partial k-block
    (64, 2048, 12288, 0, True),     # decode QKV width: 96 channel tiles, K split in three
    (8, 16384, 1024, 2, False),     # long K over few tiles: sixteen splits
])
def test_gemm_stream(fg, M, K, N, epi, bias):
    """M <= 128 runs the weight-streaming kernel (restored weights in tensor memory)."""
    fg.fg_prof_reset()
    fg.fg_prof_enable(True)
    try:
        gemm_case(fg, M, K, N, epi, bias, seed=M * 7 + K + N)
    finally:
        fg.fg_prof_enable(False)
    assert fg.fg_prof_query(fg.K_GEMM_STREAM)["launches"] == 1
    assert fg.fg_prof_query(fg.K_GEMM)["launches"] == 0


# QKV projection with the KV quantise-and-append in the GEMM epilogue.  The codes and (a, b)
# are bit-exact against the oracle's quantiser applied to the K/V columns of the kernel's own
# fp16 output (Y); Y itself matches the plain GEMM bit for bit and the oracle GEMM within
# the float tolerance.  Cases cover the streaming kernel unsplit and split-K (the reduce
# kernel appends), and the tiled kernel with ragged token tiles; d = 64 and 128.
@pytest.mark.parametrize("M,K,N,epi,bias", [
    (256, 64, 256, 0, False),       # one 2-CTA tile: one pair, one k-block
    (512, 320, 512, 1, True),       # two token tiles x two pairs, five k-blocks
    (1000, 256, 768, 2, True),      # ragged last token tile (the odd CTA's half past M), 3 pairs
    (2048, 1024, 1024, 0, True),    # 8 tiles x 4 pairs
    (4352, 512, 2304, 1, False),    # 17 tiles x 9 pairs: several tiles per pair, two raster groups
    (512, 8192, 256, 2, True),      # few tiles: K split over the pairs, then the reduce
    (144, 12288, 4096, 1, True),    # decode M = 144: one 256 x 144 tile per pair, 4-k-block stages
    (144, 16384, 1024, 2, True),    # M = 144, few pairs: K split in whole 4-k-block stages
    (130, 80, 512, 0, False),       # 72 tokens per CTA, K ragged inside a k-block (1-k-block stages)
    (200, 1024, 768, 2, True),      # 104 tokens per CTA, three pairs
])
def test_gemm_pair(fg, M, K, N, epi, bias):
    """M > 128 runs on CTA pairs (2-CTA tensor-core tiles of 256 channels x up to 256
    tokens)."""
    fg.fg_prof_reset()
    fg.fg_prof_enable(True)
    try:
        gemm_case(fg, M, K, N, epi, bias, seed=M * 13 + K + N)
    finally:
        fg.fg_prof_enable(False)
    assert fg.fg_prof_query(fg.K_GEMM_PAIR)["launches"] == 1
    assert fg.fg_prof_query(fg.K_GEMM)["launches"] == 0


@pytest.mark.parametrize("B,T,pos,h,H,K,cap,path", [
    (64, 1, 7, 512, 4, 256, 16, "stream"),          # decode: one new token per sequence
    (16, 1, 0, 256, 4, 4096, 16, "split"),         # long K: split-K, appended by the reduce
    (5, 1, 31, 768, 6, 1024, 32, "any"),           # six heads of 128, last cache slot
    (40, 5, 3, 256, 4, 256, 16, "tiled"),          # 200 rows: tiled kernel, ragged tile
    (3, 100, 0, 512, 8, 512, 112, "tiled"),        # prefill rows, d = 64
])
def test_gemm_kv_append(fg, B, T, pos, h, H, K, cap, path):
    M, N = B * T, 3 * h
    seed = B * 1000 + T * 10 + h
    x16 = fg_synth.random_fp16((M, K), seed, 1.0)
    w16 = fg_synth.random_fp16((K, N), seed + 1, 0.02)
    bias16 = fg_synth.random_fp16((N,), seed + 2, 0.1)
    W = fg.Q4Weight.from_fp16(dev(w16))
    X, bias = dev(x16), dev(bias16)
    wsb = fg.fg_gemm_workspace_bytes(M, K, N)
    ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device="cuda") if wsb else None
    cache = fg.KVCacheQ4(B, cap, h, H)
    Y = torch.empty((M, N), dtype=torch.float16, device="cuda")
    fg.fg_prof_reset()
    fg.fg_prof_enable(True)
    try:
        fg.fg_dequant_gemm_q4_kv(X, W, bias, Y, cache, T, pos, ws)
        fg.fg_check_device_error()
    finally:
        fg.fg_prof_enable(False)
    n_stream = fg.fg_prof_query(fg.K_GEMM_STREAM)["launches"]
    n_reduce = fg.fg_prof_query(fg.K_GEMM_REDUCE)["launches"]
    assert fg.fg_prof_query(fg.K_KV_APPEND)["launches"] == 0
    if path == "stream":
        assert n_stream == 1 and n_reduce == 0
    elif path == "split":
        assert n_reduce == 1
    elif path == "tiled":
        assert n_stream == 0 and fg.fg_prof_query(fg.K_GEMM)["launches"] == 1
    y16 = host(Y).view(np.float16)
    # Y: bit-identical to the plain GEMM when that runs the same kernel (the plain GEMM of
    # more than 32 rows runs on CTA pairs, which sum in another order: then within the
    # float tolerance), and within tolerance of the oracle GEMM
    Y2 = torch.empty_like(Y)
    fg.fg_prof_reset()
    fg.fg_prof_enable(True)
    try:
        fg.fg_dequant_gemm_q4(X, W, bias, 0, None, Y2, ws)
        fg.fg_check_device_error()
    finally:
        fg.fg_prof_enable(False)
    if fg.fg_prof_query(fg.K_GEMM_PAIR)["launches"] == 0:
        assert torch.equal(Y, Y2)
    else:
        assert_close(f16(Y2), y16.astype(np.float64), f"plain vs fused M={M} N={N}")
    q, a, b = OQ.quantize_g64(w16)
    ref = x16.astype(np.float64) @ OQ.dequant_g64(q, a, b).astype(np.float64) + bias16
    assert_close(y16.astype(np.float64), ref, f"qkv+append M={M} N={N}")
    # the cache: codes and (a, b) of the output's K and V columns, nothing else written
    for src, codes_t, ab_t in ((y16[:, h:2 * h], cache.k_codes, cache.k_ab),
                               (y16[:, 2 * h:], cache.v_codes, cache.v_ab)):
        c_ref, ab_ref = oracle_packed(np.ascontiguousarray(src))
        got_c = cache_codes_to_rows(host(codes_t))
        got_ab = cache_codes_to_rows(host(ab_t)).view(np.uint32)
        assert np.array_equal(got_c[:, pos:pos + T].reshape(M, h // 2), c_ref)
        assert np.array_equal(got_ab[:, pos:pos + T].reshape(M, h // 64), ab_ref)
        untouched = np.ones(cap, bool)
        untouched[pos:pos + T] = False
        assert not got_c[:, untouched].any() and not got_ab[:, untouched].any()


@pytest.mark.parametrize("B,K,path", [(64, 256, "stream"), (16, 4096, "split"), (200, 256, "tiled")])
def test_gemm_kv_append_ties(fg, B, K, path):
    """Codes exactly at half-integers go to the exact division in every epilogue path.

    X = 0 makes Y = bias exactly; the K and V columns of the bias hold groups whose minimum
    is 0 and maximum 15 * 2^-e, the other values (k + 1/2) * 2^-e, so (x - a) * 15 / (b - a)
    is a tie k + 1/2 that rounds to the even neighbour."""
    h, H = 256, 2
    M, N = B, 3 * h
    r = np.random.default_rng(B + K)
    bias16 = r.standard_normal(N).astype(np.float16)
    for g0 in range(h, N, 64):
        e = float(2.0 ** -int(r.integers(0, 4)))
        vals = (r.integers(0, 15, size=64) + 0.5) * e
        vals[r.choice(64, 2, replace=False)] = [0.0, 15.0 * e]
        bias16[g0:g0 + 64] = vals.astype(np.float16)
    W = fg.Q4Weight.from_fp16(dev(fg_synth.random_fp16((K, N), B, 0.02)))
    X = torch.zeros((M, K), dtype=torch.float16, device="cuda")
    wsb = fg.fg_gemm_workspace_bytes(M, K, N)
    ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device="cuda") if wsb else None
    cache = fg.KVCacheQ4(B, 16, h, H)
    Y = torch.empty((M, N), dtype=torch.float16, device="cuda")
    fg.fg_prof_reset()
    fg.fg_prof_enable(True)
    try:
        fg.fg_dequant_gemm_q4_kv(X, W, dev(bias16), Y, cache, 1, 5, ws)
        fg.fg_check_device_error()
    finally:
        fg.fg_prof_enable(False)
    n_red = fg.fg_prof_query(fg.K_GEMM_REDUCE)["launches"]
    n_stream = fg.fg_prof_query(fg.K_GEMM_STREAM)["launches"]
    assert (path == "split") == (n_red == 1) and (path == "tiled") == (n_stream == 0)
    y16 = host(Y).view(np.float16)
    assert np.array_equal(y16, np.broadcast_to(bias16, (M, N)))
    for src, codes_t, ab_t in ((y16[:, h:2 * h], cache.k_codes, cache.k_ab),
                               (y16[:, 2 * h:], cache.v_codes, cache.v_ab)):
        c_ref, ab_ref = oracle_packed(np.ascontiguousarray(src))
        assert np.array_equal(cache_codes_to_rows(host(codes_t))[:, 5], c_ref)
        assert np.array_equal(cache_codes_to_rows(host(ab_t)).view(np.uint32)[:, 5], ab_ref)


def test_gemm_kv_append_rejects_bad_shapes(fg):
    h, H, B = 256, 2, 4
    W = fg.Q4Weight.from_fp16(torch.zeros((256, 3 * h), dtype=torch.float16, device="cuda"))
    X = torch.zeros((B, 256), dtype=torch.float16, device="cuda")
    Y = torch.empty((B, 3 * h), dtype=torch.float16, device="cuda")
    cache = fg.KVCacheQ4(B, 16, h, H)
    with pytest.raises(fg.FgError, match=r"\(-6\)"):                       # FG_ERR_CAPACITY
        fg.fg_dequant_gemm_q4_kv(X, W, None, Y, cache, 1, 16, None)      # pos + T > cap
    with pytest.raises(fg.FgError):
        fg.fg_dequant_gemm_q4_kv(X[:3], W, None, Y, cache, 1, 0, None)   # M != B * T
    W2 = fg.Q4Weight.from_fp16(torch.zeros((256, 2 * h), dtype=torch.float16, device="cuda"))
    with pytest.raises(fg.FgError):
        fg.fg_dequant_gemm_q4_kv(X, W2, None, Y, cache, 1, 0, None)      # N != 3h
    assert not host(cache.k_codes).any()


# GEMM + LayerNorm of its output rows: Y bit-identical to the plain GEMM, Y_ln within the
# float tolerance of the oracle's LayerNorm of Y as stored, and within one fp16 step of the
# standalone LayerNorm kernel on the same Y (the statistics are summed in another order).
# Split plans run the fused reduce (no LayerNorm launch); unsplit ones the GEMM then the
# LayerNorm kernel.
@pytest.mark.parametrize("M,K,N,epi,fused", [
    (64, 4096, 4096, 2, True),       # decode O projection + residual, then LN2
    (16, 4096, 8192, 1, True),       # FC1-wide rows: four chunks of 8 per thread
    (7, 16384, 768, 0, True),        # FC2-long K split 16 ways; 96 chunks for 256 threads
    (300, 512, 1024, 2, False),      # many rows: unsplit GEMM, then the LayerNorm kernel
])
def test_gemm_layernorm(fg, M, K, N, epi, fused):
    seed = M * 13 + K + N
    x16 = fg_synth.random_fp16((M, K), seed, 1.0)
    w16 = fg_synth.random_fp16((K, N), seed + 1, 0.02)
    bias16 = fg_synth.random_fp16((N,), seed + 2, 0.1)
    res16 = fg_synth.random_fp16((M, N), seed + 3, 1.0, offset=0.5) if epi == 2 else None
    g16 = fg_synth.random_fp16((N,), seed + 4, 0.1, offset=1.0)
    b16 = fg_synth.random_fp16((N,), seed + 5, 0.1)
    W = fg.Q4Weight.from_fp16(dev(w16))
    X, bias, g, b = dev(x16), dev(bias16), dev(g16), dev(b16)
    res = dev(res16) if res16 is not None else None
    wsb = fg.fg_gemm_workspace_bytes(M, K, N)
    ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device="cuda") if wsb else None
    Y = torch.empty((M, N), dtype=torch.float16, device="cuda")
    Yln = torch.empty_like(Y)
    fg.fg_prof_reset()
    fg.fg_prof_enable(True)
    try:
        fg.fg_dequant_gemm_q4_ln(X, W, bias, epi, res, Y, g, b, 1e-5, Yln, ws)
        fg.fg_check_device_error()
    finally:
        fg.fg_prof_enable(False)
    n_ln = fg.fg_prof_query(fg.K_LAYERNORM)["launches"]
    n_red = fg.fg_prof_query(fg.K_GEMM_REDUCE)["launches"]
    assert (n_ln, n_red) == ((0, 1) if fused else (1, 0))
    Y2 = torch.empty_like(Y)
    fg.fg_dequant_gemm_q4(X, W, bias, epi, res, Y2, ws)
    assert torch.equal(Y, Y2)
    y16 = host(Y).view(np.float16)
    ref = OL.layernorm(y16, g16, b16, 1e-5)
    assert_close(f16(Yln), ref, f"gemm+ln M={M} N={N}")
    Y3 = torch.empty_like(Y)
    fg.fg_layernorm(Y, g, b, 1e-5, Y3)
    d = np.abs(f16(Yln) - f16(Y3))
    assert d.max() <= np.abs(f16(Y3)).max() * 2.0 ** -10


def test_gemm_layernorm_rejects_aliasing(fg):
    W = fg.Q4Weight.from_fp16(torch.zeros((64, 256), dtype=torch.float16, device="cuda"))
    X = torch.zeros((4, 64), dtype=torch.float16, device="cuda")
    Y = torch.empty((4, 256), dtype=torch.float16, device="cuda")
    g = torch.ones(256, dtype=torch.float16, device="cuda")
    with pytest.raises(fg.FgError):
        fg.fg_dequant_gemm_q4_ln(X, W, None, 0, None, Y, g, g, 1e-5, Y, None)


def test_gemm_split_k(fg):
    wsb = gemm_case(fg, 64, 4096, 512, 2, True, seed=77)
    assert wsb > 0                                        # the split-K path ran


def test_gemm_inplace_residual(fg):
    gemm_case(fg, 96, 512, 768, 2, True, seed=91, alias=True)


@pytest.mark.parametrize("M,K,N,epi", [
    (8192, 4096, 12288, 0),        # 6.7B prefill QKV, one GPU batch (g*s = 16*512)
    (64, 4096, 16384, 1),          # 6.7B decode FC1 (M = B)
    (144, 28672, 7168, 2),         # 30B decode FC2
    (18432, 12288, 4096, 0),       # 175B prefill, one GPU batch, N reduced to 4096
])
def test_gemm_full_size_sampled(fg, M, K, N, epi):
    """Workload-sized launches; the oracle computes sampled rows only."""
    seed = M + K + N
    x16 = fg_synth.random_fp16((M, K), seed, 1.0)
    w16 = fg_synth.random_fp16((K, N), seed + 1, 0.02)
    res16 = fg_synth.random_fp16((M, N), seed + 3, 1.0) if epi == 2 else None
    W = fg.Q4Weight.from_fp16(dev(w16))
    Y = torch.empty((M, N), dtype=torch.float16, device="cuda")
    wsb = fg.fg_gemm_workspace_bytes(M, K, N)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda") if wsb else None
    res = dev(res16) if res16 is not None else None
    fg.fg_dequant_gemm_q4(dev(x16), W, None, epi, res, Y, ws)
    fg.fg_check_device_error()
    rows = np.unique(np.r_[0, M - 1, np.random.Generator(np.random.PCG64(seed)).integers(0, M, 6)])
    q, a, b = OQ.quantize_g64(w16)
    what = OQ.dequant_g64(q, a, b).astype(np.float32)
    ref = (x16[rows].astype(np.float32) @ what).astype(np.float64)
    if epi == 1:
        ref = np.maximum(ref, 0)
    elif epi == 2:
        ref += res16[rows].astype(np.float64)
    got = f16(Y[torch.from_numpy(rows).cuda()])
    assert_close(got, ref, f"gemm full M={M} K={K} N={N}")


@pytest.mark.parametrize("M,K,N,epi", [
    (8192, 4096, 4096, 2),         # prefill O projection with residual (CTA pairs)
    (18432, 12288, 4096, 0),       # long K: 192 k-blocks per tile (CTA pairs)
    (144, 12288, 4096, 1),         # decode M = 144: one-CTA tiled kernel
    (64, 16384, 4096, 2),          # decode FC2: split K + reduce
    (512, 8192, 256, 2),           # CTA pairs with split K
])
def test_gemm_repeat_bit_identical(fg, M, K, N, epi):
    """The pipelined GEMM is deterministic: repeated launches on the same inputs give the
    same bits, which a race between its shared-memory producers and consumers would break."""
    seed = 7 * M + K + N
    X = dev(fg_synth.random_fp16((M, K), seed, 1.0))
    W = fg.Q4Weight.from_fp16(dev(fg_synth.random_fp16((K, N), seed + 1, 0.02)))
    res = dev(fg_synth.random_fp16((M, N), seed + 3, 1.0)) if epi == 2 else None
    wsb = fg.fg_gemm_workspace_bytes(M, K, N)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda") if wsb else None
    outs = []
    for _ in range(3):
        Y = torch.empty((M, N), dtype=torch.float16, device="cuda")
        fg.fg_dequant_gemm_q4(X, W, None, epi, res, Y, ws)
        outs.append(Y)
    fg.fg_check_device_error()
    for Y in outs[1:]:
        assert torch.equal(Y.view(torch.int16), outs[0].view(torch.int16))


# ----------------------------------------------------------------------------- decode attention


def oracle_cache_from_rows(fg, k16, v16, cap, H):
    """Quantise K/V rows [B][T][h] with the oracle and place the codes in a device cache."""
    B, T, h = k16.shape
    cache = fg.KVCacheQ4(B, cap, h, H)
    hats = []
    for src, codes_t, ab_t in ((k16, cache.k_codes, cache.k_ab), (v16, cache.v_codes, cache.v_ab)):
        q, a, b = OQ.quantize_g64(src.reshape(B * T, h))
        codes = OQ.pack_nibbles(q).reshape(B, T, h // 2)
        abw = OQ.ab_pack_u32(a, b).reshape(B, T, h // 64).view(np.int32)
        codes_t[:, :, :T] = dev(rows_to_cache(codes, H))
        ab_t[:, :, :T] = dev(rows_to_cache(abw, H))
        hats.append(OQ.dequant_g64(q, a, b).reshape(B, T, h))
    return cache, hats[0], hats[1]


@pytest.mark.parametrize("B,H,d,T,length,stride3", [
    (3, 4, 128, 100, 1, False), (3, 4, 128, 100, 17, True), (3, 4, 128, 100, 100, False),
    (2, 4, 64, 40, 37, True), (1, 2, 128, 600, 600, False), (64, 32, 128, 530, 530, True)])
def test_decode_attention(fg, B, H, d, T, length, stride3):
    h = H * d
    k16 = fg_synth.random_fp16((B, T, h), seed=B * 1000 + T, scale=1.5)
    v16 = fg_synth.random_fp16((B, T, h), seed=B * 1000 + T + 1, scale=1.0, offset=0.2)
    cache, khat, vhat = oracle_cache_from_rows(fg, k16, v16, T + 3, H)
    # positions the call must not read (or must mask): garbage codes, NaN statistics
    cache.k_codes[:, :, T:] = 0x5A
    cache.v_codes[:, :, T:] = 0xA5
    cache.k_ab[:, :, T:] = 0x7E007E00
    cache.v_ab[:, :, T:] = 0x7E007E00
    qbuf16 = fg_synth.random_fp16((B, 3 * h if stride3 else h), seed=T + 5, scale=1.5)
    q16 = qbuf16[:, :h]
    out = torch.empty((B, h), dtype=torch.float16, device="cuda")
    wsb = fg.fg_decode_attn_workspace_bytes(cache, length)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda") if wsb else None
    scale = 1.0 / math.sqrt(d)
    fg.fg_decode_attn_q4kv(dev(qbuf16), qbuf16.shape[1], cache, length, scale, out, ws)
    ref = OL.decode_attention(q16, khat[:, :length], vhat[:, :length], H, d)
    assert_close(f16(out), ref, f"decode attn B={B} H={H} d={d} len={length}")


def test_decode_attention_full_kv_workload_sampled(fg):
    """The KV-dominated workload's cache (512 sequences x 56 heads x 1056 positions) filled
    with seeded random codes on the device; two sequences checked against the oracle."""
    wl = fg_synth.WORKLOADS["kv-decode"]
    B, H, d, cap = wl.B, wl.H, wl.d, wl.cap
    kc, vc, ka, va = fg_synth.random_q4_cache_torch(B, H, cap, d, seed=4)
    cache = fg.KVCacheQ4.__new__(fg.KVCacheQ4)
    cache.B, cache.cap, cache.h, cache.H, cache.d = B, cap, wl.h, H, d
    cache.k_codes, cache.v_codes, cache.k_ab, cache.v_ab = kc, vc, ka, va
    q16 = fg_synth.random_fp16((B, wl.h), seed=44, scale=1.5)
    out = torch.empty((B, wl.h), dtype=torch.float16, device="cuda")
    wsb = fg.fg_decode_attn_workspace_bytes(cache, cap)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda") if wsb else None
    fg.fg_decode_attn_q4kv(dev(q16), wl.h, cache, cap, 1.0 / math.sqrt(d), out, ws)
    for b in (0, B - 1):
        hats = []
        for codes_t, ab_t in ((kc, ka), (vc, va)):
            codes = cache_codes_to_rows(host(codes_t[b:b + 1]))[0]          # [cap][h/2]
            abw = cache_codes_to_rows(host(ab_t[b:b + 1]))[0].view(np.uint32)
            q = OQ.unpack_nibbles(codes)
            a = (abw & 0xFFFF).astype(np.uint16).view(np.float16)
            bb = (abw >> 16).astype(np.uint16).view(np.float16)
            hats.append(OQ.dequant_g64(q, a, bb))
        ref = OL.decode_attention(q16[b:b + 1], hats[0][None], hats[1][None], H, d)
        assert_close(f16(out[b:b + 1]), ref, f"kv workload seq {b}")


# ----------------------------------------------------------------------------- top-K attention


def _topk_check(q16, khat, vhat, H, d, k, got, sel_gpu, label):
    """The GPU's selection is a valid top-k of the oracle's scores (near-equal scores at the
    k-th place may fall either way) and its output is the oracle's weighted sum over it."""
    S = q16.shape[0]
    qh = q16.astype(np.float64).reshape(S, H, 1, d)
    kh = khat.astype(np.float64).reshape(S, -1, H, d).transpose(0, 2, 1, 3)
    sc = ((qh @ kh.transpose(0, 1, 3, 2)) / math.sqrt(d))[:, :, 0, :]       # [S][H][T]
    kth = -np.sort(-sc, axis=-1)[:, :, k - 1:k]
    eps = 2e-3 * np.abs(sc).max() + 1e-4
    picked = np.zeros(sc.shape, dtype=bool)
    np.put_along_axis(picked, sel_gpu.astype(np.int64), True, axis=-1)
    assert (np.sort(sel_gpu, axis=-1)[:, :, 1:] > np.sort(sel_gpu, axis=-1)[:, :, :-1]).all(), \
        f"{label}: repeated position"
    assert (sc[picked] >= np.broadcast_to(kth, sc.shape)[picked] - eps).all(), f"{label}: low pick"
    assert (sc[~picked] <= np.broadcast_to(kth, sc.shape)[~picked] + eps).all(), f"{label}: missed"
    ref, oracle_sel = OL.decode_attention_topk(q16, khat, vhat, H, d, k, selected=sel_gpu)
    assert_close(got, ref, label)
    same = np.mean([len(set(a) & set(b)) / k for a, b in
                    zip(sel_gpu.reshape(-1, k).tolist(),
                        OL.decode_attention_topk(q16, khat, vhat, H, d, k)[1].reshape(-1, k).tolist())])
    assert same > 0.95, f"{label}: only {same:.3f} of the oracle's selection"


@pytest.mark.parametrize("B,H,d,T,length,k,stride3", [
    (3, 4, 128, 100, 100, 10, False), (2, 4, 64, 40, 37, 4, True), (2, 2, 128, 600, 600, 60, False),
    (2, 2, 64, 50, 50, 1, False), (64, 32, 128, 543, 543, 55, True)])
def test_decode_attention_topk(fg, B, H, d, T, length, k, stride3):
    h = H * d
    k16 = fg_synth.random_fp16((B, T, h), seed=B * 77 + T, scale=1.5)
    v16 = fg_synth.random_fp16((B, T, h), seed=B * 77 + T + 1, scale=1.0, offset=0.2)
    cache, khat, vhat = oracle_cache_from_rows(fg, k16, v16, T + 3, H)
    cache.k_codes[:, :, T:] = 0x5A                  # never read: garbage past the end
    cache.v_codes[:, :, T:] = 0xA5
    cache.k_ab[:, :, T:] = 0x7E007E00
    cache.v_ab[:, :, T:] = 0x7E007E00
    qbuf16 = fg_synth.random_fp16((B, 3 * h if stride3 else h), seed=T + 9, scale=1.5)
    q16 = qbuf16[:, :h]
    out = torch.empty((B, h), dtype=torch.float16, device="cuda")
    sel = torch.empty((B, H, k), dtype=torch.int32, device="cuda")
    ws = torch.empty(fg.fg_decode_attn_topk_workspace_bytes(cache, length), dtype=torch.uint8,
                     device="cuda")
    fg.fg_decode_attn_q4kv_topk(dev(qbuf16), qbuf16.shape[1], cache, length, k,
                                1.0 / math.sqrt(d), out, ws, sel)
    fg.fg_check_device_error()
    _topk_check(q16, khat[:, :length], vhat[:, :length], H, d, k, f16(out), host(sel),
                f"topk B={B} H={H} d={d} len={length} k={k}")


def test_decode_attention_topk_all_positions_is_dense(fg):
    """k = len keeps every value: the dense kernel's result."""
    B, H, d, T = 4, 4, 128, 300
    h = H * d
    k16 = fg_synth.random_fp16((B, T, h), seed=31, scale=1.5)
    v16 = fg_synth.random_fp16((B, T, h), seed=32, scale=1.0)
    cache, _, _ = oracle_cache_from_rows(fg, k16, v16, T, H)
    q = dev(fg_synth.random_fp16((B, h), seed=33, scale=1.5))
    dense = torch.empty((B, h), dtype=torch.float16, device="cuda")
    wsb = fg.fg_decode_attn_workspace_bytes(cache, T)
    fg.fg_decode_attn_q4kv(q, h, cache, T, 0.1, dense,
                           torch.empty(wsb, dtype=torch.uint8, device="cuda") if wsb else None)
    top = torch.empty_like(dense)
    ws = torch.empty(fg.fg_decode_attn_topk_workspace_bytes(cache, T), dtype=torch.uint8,
                     device="cuda")
    fg.fg_decode_attn_q4kv_topk(q, h, cache, T, T, 0.1, top, ws)
    fg.fg_check_device_error()
    assert_close(f16(top), f16(dense).astype(np.float64), "topk k=len vs dense")


def test_decode_attention_topk_kv_workload_sampled(fg):
    """The KV-dominated workload's cache with the pages' top 10% (106 of 1056 positions);
    two sequences checked against the oracle."""
    wl = fg_synth.WORKLOADS["kv-decode"]
    B, H, d, cap = wl.B, wl.H, wl.d, wl.cap
    k = OL.topk_count(cap)
    kc, vc, ka, va = fg_synth.random_q4_cache_torch(B, H, cap, d, seed=5)
    cache = fg.KVCacheQ4.__new__(fg.KVCacheQ4)
    cache.B, cache.cap, cache.h, cache.H, cache.d = B, cap, wl.h, H, d
    cache.k_codes, cache.v_codes, cache.k_ab, cache.v_ab = kc, vc, ka, va
    q16 = fg_synth.random_fp16((B, wl.h), seed=45, scale=1.5)
    out = torch.empty((B, wl.h), dtype=torch.float16, device="cuda")
    sel = torch.empty((B, H, k), dtype=torch.int32, device="cuda")
    ws = torch.empty(fg.fg_decode_attn_topk_workspace_bytes(cache, cap), dtype=torch.uint8,
                     device="cuda")
    fg.fg_decode_attn_q4kv_topk(dev(q16), wl.h, cache, cap, k, 1.0 / math.sqrt(d), out, ws, sel)
    fg.fg_check_device_error()
    for b in (0, B - 1):
        hats = []
        for codes_t, ab_t in ((kc, ka), (vc, va)):
            codes = cache_codes_to_rows(host(codes_t[b:b + 1]))[0]
            abw = cache_codes_to_rows(host(ab_t[b:b + 1]))[0].view(np.uint32)
            qq = OQ.unpack_nibbles(codes)
            a = (abw & 0xFFFF).astype(np.uint16).view(np.float16)
            bb = (abw >> 16).astype(np.uint16).view(np.float16)
            hats.append(OQ.dequant_g64(qq, a, bb))
        _topk_check(q16[b:b + 1], hats[0][None], hats[1][None], H, d, k, f16(out[b:b + 1]),
                    host(sel[b:b + 1]), f"topk kv workload seq {b}")


# ----------------------------------------------------------------------------- prefill attention


@pytest.mark.parametrize("nseq,s,H,d,mag", [
    (2, 16, 4, 64, 1.5), (3, 100, 2, 128, 1.5), (1, 513, 2, 128, 1.5), (2, 64, 3, 64, 1.5),
    (1, 1, 2, 128, 1.5),
    (2, 384, 2, 128, 1.5),       # a full 256-row block and a half one, key tiles shared by both
    (3, 300, 3, 64, 1.5),        # d = 64, ragged second block
    (1, 1024, 1, 128, 1.5),      # four blocks, up to eight key tiles per Q tile
    (2, 640, 2, 128, 4.0),       # large scores: the reference maximum moves many times
    # more blocks than SMs: every persistent CTA takes several blocks (next block's loads and
    # first products during the previous block's output), ragged last blocks
    (3, 700, 24, 128, 1.5),
    (4, 520, 20, 64, 1.5),
])
def test_prefill_attention(fg, nseq, s, H, d, mag):
    h = H * d
    qkv16 = fg_synth.random_fp16((nseq * s, 3 * h), seed=nseq * 10 + s, scale=mag)
    out = torch.empty((nseq * s, h), dtype=torch.float16, device="cuda")
    fg.fg_prefill_attn(dev(qkv16), nseq, s, H, d, 1.0 / math.sqrt(d), out)
    x = qkv16.reshape(nseq, s, 3 * h)
    ref = OL.causal_attention(x[..., :h], x[..., h:2 * h], x[..., 2 * h:], H, d)
    assert_close(f16(out).reshape(nseq, s, h), ref, f"prefill attn {nseq}x{s} H={H} d={d}")
