"""The allocation-free decode-attention entry point gives the same output as the
workspace entry point and as the oracle.

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
from oracle import layer as OL
from oracle import quant as OQ
from parity_util import assert_close, dev, f16, lib, rows_to_cache

pytestmark = pytest.mark.gpu


def make_cache(fg, B, H, d, T, cap, seed):
    """A cache holding the oracle's codes of seeded K/V rows; returns it with the oracle's
    restored K^, V^ [B][T][h]."""
    h = H * d
    k16 = fg_synth.random_fp16((B, T, h), seed=seed, scale=1.5)
    v16 = fg_synth.random_fp16((B, T, h), seed=seed + 1, scale=1.0, offset=0.2)
    cache = fg.KVCacheQ4(B, cap, h, H)
    hats = []
    for src, codes_t, ab_t in ((k16, cache.k_codes, cache.k_ab), (v16, cache.v_codes, cache.v_ab)):
        q, a, b = OQ.quantize_g64(src.reshape(B * T, h))
        codes_t[:, :, :T] = dev(rows_to_cache(OQ.pack_nibbles(q).reshape(B, T, h // 2), H))
        ab_t[:, :, :T] = dev(rows_to_cache(
            OQ.ab_pack_u32(a, b).reshape(B, T, h // 64).view(np.int32), H))
        hats.append(OQ.dequant_g64(q, a, b).reshape(B, T, h))
    return cache, hats[0], hats[1]


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


@pytest.mark.parametrize("d", [128, 64])
def test_static_scratch_matches_workspace_entry_point_twice(d):
    """Two calls in a row with split scratch (the array keeps the first call's contents),
    each against the workspace entry point and the oracle."""
    fg = lib()
    B, H, T = 2, 4 if d == 128 else 8, 600
    cache, khat, vhat = make_cache(fg, B, H, d, T, T + 8, seed=501 + d)
    scale = 1.0 / math.sqrt(d)
    h = H * d
    # first call: full length, q read from a [B][3h] QKV-style buffer
    qbuf16 = fg_synth.random_fp16((B, 3 * h), seed=502, scale=1.5)
    wsb, got, ref = run_both(fg, cache, dev(qbuf16), 3 * h, T, scale)
    assert wsb > 0, "this case must use split-sequence scratch"
    assert_close(got, ref, f"static scratch d={d}, call 1 vs workspace entry")
    assert_close(got, OL.decode_attention(qbuf16[:, :h], khat, vhat, H, d),
                 f"static scratch d={d}, call 1 vs oracle")
    # second call in a row: other query, other length
    q2 = fg_synth.random_fp16((B, h), seed=503, scale=1.0)
    wsb2, got2, ref2 = run_both(fg, cache, dev(q2), h, 333, scale)
    assert wsb2 > 0
    assert_close(got2, ref2, f"static scratch d={d}, call 2 vs workspace entry")
    assert_close(got2, OL.decode_attention(q2, khat[:, :333], vhat[:, :333], H, d),
                 f"static scratch d={d}, call 2 vs oracle")
    assert not np.allclose(got, got2)


def test_static_scratch_unsplit_call():
    """A short cache over many heads needs no split scratch (the workspace query returns 0):
    the static entry point passes the array but the kernel does not use it."""
    fg = lib()
    B, H, d, T = 16, 32, 128, 40
    cache, khat, vhat = make_cache(fg, B, H, d, T, T + 8, seed=611)
    assert fg.fg_decode_attn_workspace_bytes(cache, T) == 0
    q16 = fg_synth.random_fp16((B, H * d), seed=612, scale=1.5)
    for length in (T, 17):
        wsb, got, ref = run_both(fg, cache, dev(q16), H * d, length, 1.0 / math.sqrt(d))
        assert wsb == 0
        assert_close(got, ref, f"unsplit static len={length} vs workspace entry")
        assert_close(got, OL.decode_attention(q16, khat[:, :length], vhat[:, :length], H, d),
                     f"unsplit static len={length} vs oracle")


def test_static_scratch_rejects_oversize_calls():
    fg = lib()
    # 25 sequences x 100 heads x 4096 positions: the split scratch that
    # fg_decode_attn_workspace_bytes reports (planned for up to 192 SMs) exceeds the 4 MiB
    # static array, and that query is the threshold: the call is rejected on the host
    # before any launch
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
