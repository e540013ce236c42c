"""The C-ABI library builds, loads and exports every symbol include/fg.h declares, and
its host-side argument validation rejects bad calls before touching CUDA (so these run
on a machine without a GPU)."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def fg():
    import __graft_entry__ as g
    g.build()
    from bit_compressed_throughput_gb300 import fg as mod
    return mod


def declared_symbols():
    hdr = open(os.path.join(ROOT, "include", "fg.h")).read()
    return sorted(set(re.findall(r"^\s*(?:int|size_t|const char\*)\s+(fg_\w+)\s*\(", hdr, re.M)))


def test_exports_every_declared_symbol(fg):
    names = declared_symbols()
    assert len(names) >= 19
    missing = [n for n in names if not hasattr(fg.lib, n)]
    assert missing == []
    # the boundary's calls by the names the scope table gives them
    for n in ("fg_quantize_g64", "fg_dequant_gemm_q4", "fg_kv_append_q4", "fg_decode_attn_q4kv",
              "fg_layer_prefill", "fg_layer_decode", "fg_workspace_bytes", "fg_status_string"):
        assert n in names, n


def test_workspace_bytes_names_agree(fg):
    for h, H, f, g, m, s in ((256, 4, 1024, 2, 2, 20), (4096, 32, 16384, 16, 4, 544),
                             (7168, 56, 0, 128, 4, 1056)):
        dm = fg.fg_dims(h, H, h // H, f, 1e-5)
        a = fg.lib.fg_workspace_bytes(fg.C.byref(dm), g, m, s)
        assert a > 0 and a == fg.lib.fg_layer_workspace_bytes(fg.C.byref(dm), g, m, s)
    bad = fg.fg_dims(100, 4, 25, 0, 1e-5)
    assert fg.lib.fg_workspace_bytes(fg.C.byref(bad), 2, 2, 16) == 0


def test_status_strings(fg):
    for s in range(0, -8, -1):
        assert fg.lib.fg_status_string(s).decode() not in ("", "unknown status")
    assert fg.lib.fg_status_string(-99).decode() == "unknown status"


FAKE = 0x10000          # aligned, never dereferenced: validation fails before any use
MISALIGNED = 0x10008
FAKE2 = 0x20000         # a second aligned, never dereferenced address


def q4(K, N, codes=FAKE, ab=FAKE):
    from bit_compressed_throughput_gb300 import fg
    return fg.fg_q4mat(codes, ab, K, N)


def test_quantize_validation(fg):
    L = fg.lib
    assert L.fg_quantize_g64(FAKE, 4, 63, FAKE, FAKE, None) == fg.FG_ERR_SHAPE
    assert L.fg_quantize_g64(FAKE, -1, 64, FAKE, FAKE, None) == fg.FG_ERR_SHAPE
    assert L.fg_quantize_g64(None, 4, 64, FAKE, FAKE, None) == fg.FG_ERR_ARG
    assert L.fg_quantize_g64(MISALIGNED, 4, 64, FAKE, FAKE, None) == fg.FG_ERR_ARG
    assert L.fg_quantize_g64(None, 0, 64, None, None, None) == fg.FG_OK     # empty: no-op
    assert L.fg_dequant_g64(FAKE, FAKE, 4, 96, FAKE, None) == fg.FG_ERR_SHAPE


def test_gemm_validation(fg):
    L = fg.lib
    call = lambda W, M=8, bias=None, epi=0, res=None, ws=None, wsb=0, X=FAKE, Y=FAKE: \
        L.fg_dequant_gemm_q4(X, M, C.byref(W), bias, epi, res, Y, ws, wsb, None)
    assert call(q4(40, 256)) == fg.FG_ERR_SHAPE                 # K % 16
    assert call(q4(64, 96)) == fg.FG_ERR_SHAPE                  # N % 64
    assert call(q4(64, 320)) == fg.FG_ERR_SHAPE                 # N % 256
    assert call(q4(64, 256, codes=None)) == fg.FG_ERR_ARG
    assert call(q4(64, 256), epi=3) == fg.FG_ERR_ARG
    assert call(q4(64, 256), epi=fg.FG_EPI_RESIDUAL) == fg.FG_ERR_ARG   # residual missing
    assert call(q4(64, 256), X=MISALIGNED) == fg.FG_ERR_ARG
    assert call(q4(64, 256), M=0, X=None, Y=None) == fg.FG_OK
    need = fg.fg_gemm_workspace_bytes(64, 4096, 256)
    assert need > 0                                  # one tile of 256: split K
    assert call(q4(4096, 256), M=64, ws=FAKE, wsb=need - 1) == fg.FG_ERR_WORKSPACE
    # full grid, no split: only the 256-byte unit counter of the many-token plan
    assert fg.fg_gemm_workspace_bytes(8192, 4096, 12288) == 256
    assert fg.fg_gemm_workspace_bytes(200, 64, 49152) == 0         # one token tile, no split
    # with split partials too: the counter follows them at a 256-byte boundary
    for M, K, N in ((512, 8192, 256), (18432, 49152, 12288), (300, 512, 2048)):
        wsb = fg.fg_gemm_workspace_bytes(M, K, N)
        assert wsb >= 256 and wsb % 256 == 0, (M, K, N, wsb)


def test_fused_gemm_validation(fg):
    """The QKV + K/V-append and GEMM + LayerNorm entries reject bad calls on the host."""
    L = fg.lib
    kv = kvs(B=4, cap=16, h=256, H=2)
    w3 = q4(256, 768)
    kvcall = lambda W=w3, M=4, T=1, pos=0, k=kv, X=FAKE, Y=FAKE: \
        L.fg_dequant_gemm_q4_kv(X, M, C.byref(W), None, Y, C.byref(k), T, pos, None, 0, None)
    assert kvcall(W=q4(256, 512)) == fg.FG_ERR_SHAPE            # N != 3h
    assert kvcall(M=3) == fg.FG_ERR_SHAPE                       # M != B*T
    assert kvcall(T=0, M=0) == fg.FG_ERR_SHAPE
    assert kvcall(pos=16) == fg.FG_ERR_CAPACITY                 # pos + T > cap
    assert kvcall(k=kvs(B=1 << 16, cap=1 << 14, h=256, H=2), M=1 << 16) == fg.FG_ERR_SHAPE
    assert kvcall(X=MISALIGNED) == fg.FG_ERR_ARG
    lncall = lambda M=4, Y=FAKE, Yln=FAKE2, g=FAKE, eps=1e-5, epi=0: \
        L.fg_dequant_gemm_q4_ln(FAKE, M, C.byref(q4(256, 256)), None, epi, None, Y, g, FAKE,
                                eps, Yln, None, 0, None)
    assert lncall(Yln=FAKE) == fg.FG_ERR_ARG                    # Y_ln aliases Y
    assert lncall(g=None) == fg.FG_ERR_ARG
    assert lncall(eps=0.0) == fg.FG_ERR_ARG
    assert lncall(epi=fg.FG_EPI_RESIDUAL) == fg.FG_ERR_ARG      # residual missing
    assert L.fg_dequant_gemm_q4_ln(FAKE, 4, C.byref(q4(256, 16640)), None, 0, None, FAKE, FAKE,
                                   FAKE, 1e-5, FAKE2, None, 0, None) == fg.FG_ERR_SHAPE  # N > 16384
    tk = kvs(B=2, cap=64, h=256, H=2)
    topk = lambda length=32, k=4, ws=FAKE, wsb=1 << 30: \
        L.fg_decode_attn_q4kv_topk(FAKE, 256, C.byref(tk), length, k, 0.1, FAKE, None, ws, wsb,
                                   None)
    assert topk(k=0) == fg.FG_ERR_SHAPE
    assert topk(k=33) == fg.FG_ERR_SHAPE                        # k > len
    assert topk(length=65) == fg.FG_ERR_CAPACITY
    assert topk(wsb=L.fg_decode_attn_topk_workspace_bytes(C.byref(tk), 32) - 1) \
        == fg.FG_ERR_WORKSPACE


def kvs(B=2, cap=32, h=256, H=2):
    from bit_compressed_throughput_gb300 import fg
    return fg.fg_kvcache(FAKE, FAKE, FAKE, FAKE, B, cap, h, H)


def test_kv_and_attention_validation(fg):
    L = fg.lib
    kv = kvs()
    assert L.fg_kv_append_q4(FAKE, FAKE, 256, 4, 30, C.byref(kv), None) == fg.FG_ERR_CAPACITY
    assert L.fg_kv_append_q4(FAKE, FAKE, 100, 1, 0, C.byref(kv), None) == fg.FG_ERR_SHAPE
    bad = kvs(h=256, H=8)                                        # d = 32
    assert L.fg_kv_append_q4(FAKE, FAKE, 256, 1, 0, C.byref(bad), None) == fg.FG_ERR_SHAPE
    assert L.fg_decode_attn_q4kv(FAKE, 256, C.byref(kv), 33, 0.1, FAKE, None, 0, None) \
        == fg.FG_ERR_CAPACITY
    assert L.fg_decode_attn_q4kv(FAKE, 256, C.byref(kv), 0, 0.1, FAKE, None, 0, None) \
        == fg.FG_ERR_SHAPE
    assert L.fg_decode_attn_q4kv(FAKE, 256, C.byref(kv), 4, -1.0, FAKE, None, 0, None) \
        == fg.FG_ERR_ARG
    small = kvs(B=1, cap=1024, h=256, H=2)
    need = L.fg_decode_attn_workspace_bytes(C.byref(small), 1024)
    assert need > 0                                   # 2 heads: split the sequence
    assert L.fg_decode_attn_q4kv(FAKE, 256, C.byref(small), 1024, 0.1, FAKE, FAKE, need - 1,
                                 None) == fg.FG_ERR_WORKSPACE
    assert L.fg_prefill_attn(FAKE, 2, 16, 4, 32, 0.1, FAKE, None) == fg.FG_ERR_SHAPE
    assert L.fg_layernorm(FAKE, 4, 100, FAKE, FAKE, 1e-5, FAKE, None) == fg.FG_ERR_SHAPE


def test_layer_validation(fg):
    L = fg.lib
    dm = fg.fg_dims(256, 4, 64, 1024, 1e-5)
    lay = fg.fg_layer(q4(256, 768), q4(256, 256), q4(256, 1024), q4(1024, 256),
                      None, None, None, None, FAKE, FAKE, FAKE, FAKE)
    kv = kvs(B=4, cap=32, h=256, H=4)
    wsb = L.fg_layer_workspace_bytes(C.byref(dm), 2, 2, 32)
    assert wsb > 0
    pre = lambda g=2, m=2, s=16, ws=FAKE, n=wsb, d=dm, k=kv: L.fg_layer_prefill(
        C.byref(d), C.byref(lay), C.byref(k), FAKE, FAKE, g, m, s, ws, n, None)
    assert pre(n=wsb // 4) == fg.FG_ERR_WORKSPACE
    assert pre(g=3) == fg.FG_ERR_SHAPE                       # kv.B != g*m
    assert pre(s=33) == fg.FG_ERR_CAPACITY
    assert pre(k=kvs(B=4, cap=20, h=256, H=4)) == fg.FG_ERR_SHAPE      # cap % 16
    assert pre(d=fg.fg_dims(256, 4, 64, 1000, 1e-5)) == fg.FG_ERR_SHAPE
    assert pre(d=fg.fg_dims(256, 4, 64, 960, 1e-5)) == fg.FG_ERR_SHAPE     # f % 256
    assert pre(d=fg.fg_dims(256, 2, 128, 1024, 1e-5)) == fg.FG_ERR_SHAPE   # kv.H mismatch
    lay_bad = fg.fg_layer(q4(256, 512), q4(256, 256), q4(256, 1024), q4(1024, 256),
                          None, None, None, None, FAKE, FAKE, FAKE, FAKE)
    assert L.fg_layer_prefill(C.byref(dm), C.byref(lay_bad), C.byref(kv), FAKE, FAKE, 2, 2, 16,
                              FAKE, wsb, None) == fg.FG_ERR_SHAPE
    assert L.fg_layer_decode(C.byref(dm), C.byref(lay), C.byref(kv), FAKE, FAKE, 2, 2, 32,
                             FAKE, wsb, None) == fg.FG_ERR_CAPACITY


def test_workspace_sizes_monotone(fg):
    L = fg.lib
    dm = fg.fg_dims(4096, 32, 128, 16384, 1e-5)
    a = L.fg_layer_workspace_bytes(C.byref(dm), 16, 4, 512)
    b = L.fg_layer_workspace_bytes(C.byref(dm), 16, 4, 544)
    assert 0 < a <= b
    # prefill buffers of one GPU batch: LN, QKV, attention, h1 and the FFN activation
    assert a >= 16 * 512 * (4096 * 6 + 16384) * 2




def test_decode_attention_workspace_for_long_few_sequences(fg):
    """A long sequence over few heads is split (partials in the workspace); the query sizes
    for the largest planned SM count, so it covers any GB300 launch."""
    L = fg.lib
    kv = fg.fg_kvcache(FAKE, FAKE, FAKE, FAKE, 1, 8192, 256, 2)
    assert L.fg_decode_attn_workspace_bytes(C.byref(kv), 8192) > 0
