"""The allocation-free decode-attention entry point gives the same output as the
workspace entry point.

fg_decode_attn_q4kv_static exists for callers that cannot allocate device memory (code
that must not call cudaMalloc, or whose device memory belongs to an outside allocator)
and so cannot hand the library a workspace: its split-sequence scratch is a static array
inside the library.  This file is collected last so that a run stopping at the first
failure has already run every other test; it also passes when run alone.
"""
import math

import numpy as np
import pytest
import torch

import fg_synth
from oracle import quant as OQ
from parity_util import assert_close, dev, f16, lib, rows_to_cache

pytestmark = pytest.mark.gpu


def make_cache(fg, B, H, d, T, cap, seed):
    h = H * d
    k16 = fg_synth.random_fp16((B, T, h), seed=seed, scale=1.5)
    v16 = fg_synth.random_fp16((B, T, h), seed=seed + 1, scale=1.0, offset=0.2)
    cache = fg.KVCacheQ4(B, cap, h, H)
    for src, codes_t, ab_t in ((k16, cache.k_codes, cache.k_ab), (v16, cache.v_codes, cache.v_ab)):
        q, a, b = OQ.quantize_g64(src.reshape(B * T, h))
        codes_t[:, :, :T] = dev(rows_to_cache(OQ.pack_nibbles(q).reshape(B, T, h // 2), H))
        ab_t[:, :, :T] = dev(rows_to_cache(
            OQ.ab_pack_u32(a, b).reshape(B, T, h // 64).view(np.int32), H))
    return cache


def run_both(fg, cache, q, q_stride, length, scale):
    B, h = cache.B, cache.h
    wsb = fg.fg_decode_attn_workspace_bytes(cache, length)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda") if wsb else None
    ref = torch.empty((B, h), dtype=torch.float16, device="cuda")
    fg.fg_decode_attn_q4kv(q, q_stride, cache, length, scale, ref, ws)
    got = torch.full((B, h), float("nan"), dtype=torch.float16, device="cuda")
    fg.fg_decode_attn_q4kv_static(q, q_stride, cache, length, scale, got)
    torch.cuda.synchronize()
    return wsb, f16(got), f16(ref)


def test_static_scratch_matches_workspace_entry_point_twice():
    fg = lib()
    B, H, d, T = 2, 4, 128, 600
    cache = make_cache(fg, B, H, d, T, T + 8, seed=501)
    scale = 1.0 / math.sqrt(d)
    # first call: full length, q read from a [B][3h] QKV-style buffer
    qbuf = dev(fg_synth.random_fp16((B, 3 * H * d), seed=502, scale=1.5))
    wsb, got, ref = run_both(fg, cache, qbuf, 3 * H * d, T, scale)
    assert wsb > 0, "this case must use split-sequence scratch"
    assert_close(got, ref, "static scratch, call 1")
    # second call in a row: other query, other length; the array keeps call 1's contents
    q2 = dev(fg_synth.random_fp16((B, H * d), seed=503, scale=1.0))
    wsb2, got2, ref2 = run_both(fg, cache, q2, H * d, 333, scale)
    assert wsb2 > 0
    assert_close(got2, ref2, "static scratch, call 2")
    assert not np.allclose(got, got2)


def test_static_scratch_rejects_oversize_calls():
    fg = lib()
    # 25 sequences x 100 heads x 4096 positions: the split planner chooses 6 splits on 152
    # SMs, so the partials (2500 x 6 x (128 + 2) floats = 7.8 MB) exceed the 4 MiB static
    # array; the call is rejected on the host before any launch (the cache is allocated, so
    # a device whose plan did not split would run the call instead of faulting)
    B, H, d, length = 25, 100, 128, 4096
    cache = fg.KVCacheQ4(B, length, H * d, H)
    need = fg.fg_decode_attn_workspace_bytes(cache, length)
    assert need > fg.DECODE_ATTN_STATIC_SCRATCH_BYTES
    q = torch.zeros((B, H * d), dtype=torch.float16, device="cuda")
    out = torch.full((B, H * d), 7.0, dtype=torch.float16, device="cuda")
    with pytest.raises(fg.FgError) as ei:
        fg.fg_decode_attn_q4kv_static(q, H * d, cache, length, 0.1, out)
    assert ei.value.status == fg.FG_ERR_WORKSPACE
    assert "static" in str(ei.value)
    torch.cuda.synchronize()
    assert float(out.float().min()) == 7.0          # nothing was launched
