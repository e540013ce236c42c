"""ctypes binding of libfg (include/fg.h): argument marshalling only.

Every function here checks the status the C call returns and raises ``FgError`` on
failure.  Tensors are torch CUDA tensors (device memory and streams only); nothing is
computed in Python.  Importing this module loads ``libfg.so`` from this package and
raises ``ImportError`` if it has not been built -- there is no fallback path.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Optional

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfg.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"libfg.so is not built ({LIB_PATH}); run "
                      "`python -c 'import __graft_entry__ as g; g.build()'` first")
lib = C.CDLL(LIB_PATH)

FG_OK, FG_ERR_ARG, FG_ERR_SHAPE, FG_ERR_WORKSPACE = 0, -1, -2, -3
FG_ERR_CUDA, FG_ERR_ARCH, FG_ERR_CAPACITY, FG_ERR_TIMEOUT = -4, -5, -6, -7
FG_EPI_NONE, FG_EPI_RELU, FG_EPI_RESIDUAL = 0, 1, 2
KINDS = ["q4g64_quantize", "q4g64_dequant", "q4_dequant_gemm_tc", "gemm_splitk_reduce",
         "q4kv_append", "q4kv_decode_attn", "decode_attn_combine", "prefill_attn", "layernorm",
         "q4_dequant_gemm_stream", "q4kv_decode_attn_topk", "q4_dequant_gemm_pair",
         "gemm_f16w_pair"]
K_QUANT, K_DEQUANT, K_GEMM, K_GEMM_REDUCE, K_KV_APPEND, K_DECODE_ATTN, K_DECODE_COMBINE, \
    K_PREFILL_ATTN, K_LAYERNORM, K_GEMM_STREAM, K_DECODE_ATTN_TOPK, K_GEMM_PAIR, \
    K_GEMM_PAIR_F16W = range(13)


class fg_q4mat(C.Structure):
    _fields_ = [("codes", C.c_void_p), ("ab", C.c_void_p), ("K", C.c_int64), ("N", C.c_int64)]


class fg_kvcache(C.Structure):
    _fields_ = [("k_codes", C.c_void_p), ("v_codes", C.c_void_p), ("k_ab", C.c_void_p),
                ("v_ab", C.c_void_p), ("B", C.c_int32), ("cap", C.c_int32), ("h", C.c_int32),
                ("H", C.c_int32)]


class fg_dims(C.Structure):
    _fields_ = [("h", C.c_int32), ("H", C.c_int32), ("d", C.c_int32), ("f", C.c_int32),
                ("ln_eps", C.c_float)]


class fg_layer(C.Structure):
    _fields_ = [("wqkv", fg_q4mat), ("wo", fg_q4mat), ("w1", fg_q4mat), ("w2", fg_q4mat),
                ("bqkv", C.c_void_p), ("bo", C.c_void_p), ("b1", C.c_void_p), ("b2", C.c_void_p),
                ("ln1_g", C.c_void_p), ("ln1_b", C.c_void_p), ("ln2_g", C.c_void_p),
                ("ln2_b", C.c_void_p)]


_P, _I64, _I32, _F, _SZ = C.c_void_p, C.c_int64, C.c_int32, C.c_float, C.c_size_t
_SIGS = {
    "fg_quantize_g64": ([_P, _I64, _I64, _P, _P, _P], C.c_int),
    "fg_dequant_g64": ([_P, _P, _I64, _I64, _P, _P], C.c_int),
    "fg_dequant_gemm_q4": ([_P, _I64, C.POINTER(fg_q4mat), _P, C.c_int, _P, _P, _P, _SZ, _P],
                           C.c_int),
    "fg_gemm_workspace_bytes": ([_I64, _I64, _I64], _SZ),
    "fg_dequant_gemm_q4_kv": ([_P, _I64, C.POINTER(fg_q4mat), _P, _P, C.POINTER(fg_kvcache),
                               _I32, _I32, _P, _SZ, _P], C.c_int),
    "fg_dequant_gemm_q4_ln": ([_P, _I64, C.POINTER(fg_q4mat), _P, C.c_int, _P, _P, _P, _P, _F,
                               _P, _P, _SZ, _P], C.c_int),
    "fg_kv_append_q4": ([_P, _P, _I64, _I32, _I32, C.POINTER(fg_kvcache), _P], C.c_int),
    "fg_decode_attn_q4kv": ([_P, _I64, C.POINTER(fg_kvcache), _I32, _F, _P, _P, _SZ, _P],
                            C.c_int),
    "fg_decode_attn_workspace_bytes": ([C.POINTER(fg_kvcache), _I32], _SZ),
    "fg_decode_attn_q4kv_static": ([_P, _I64, C.POINTER(fg_kvcache), _I32, _F, _P, _P], C.c_int),
    "fg_decode_attn_q4kv_topk": ([_P, _I64, C.POINTER(fg_kvcache), _I32, _I32, _F, _P, _P, _P,
                                  _SZ, _P], C.c_int),
    "fg_decode_attn_topk_workspace_bytes": ([C.POINTER(fg_kvcache), _I32], _SZ),
    "fg_prefill_attn": ([_P, _I32, _I32, _I32, _I32, _F, _P, _P], C.c_int),
    "fg_layernorm": ([_P, _I64, _I32, _P, _P, _F, _P, _P], C.c_int),
    "fg_layer_prefill": ([C.POINTER(fg_dims), C.POINTER(fg_layer), C.POINTER(fg_kvcache), _P, _P,
                          _I32, _I32, _I32, _P, _SZ, _P], C.c_int),
    "fg_layer_decode": ([C.POINTER(fg_dims), C.POINTER(fg_layer), C.POINTER(fg_kvcache), _P, _P,
                         _I32, _I32, _I32, _P, _SZ, _P], C.c_int),
    "fg_workspace_bytes": ([C.POINTER(fg_dims), _I32, _I32, _I32], _SZ),
    "fg_layer_workspace_bytes": ([C.POINTER(fg_dims), _I32, _I32, _I32], _SZ),
    "fg_status_string": ([C.c_int], C.c_char_p),
    "fg_last_error": ([], C.c_char_p),
    "fg_check_device_error": ([_P], C.c_int),
    "fg_prof_enable": ([C.c_int], C.c_int),
    "fg_prof_reset": ([], C.c_int),
    "fg_prof_query": ([C.c_int, C.POINTER(C.c_int64), C.POINTER(C.c_double),
                       C.POINTER(C.c_double)], C.c_int),
    "fg_kernel_name": ([C.c_int], C.c_char_p),
}
for _name, (_args, _res) in _SIGS.items():
    _fn = getattr(lib, _name)
    _fn.argtypes = _args
    _fn.restype = _res


class FgError(RuntimeError):
    def __init__(self, fn: str, status: int):
        msg = lib.fg_status_string(status).decode()
        detail = lib.fg_last_error().decode()
        super().__init__(f"{fn}: {msg} ({status})" + (f": {detail}" if detail else ""))
        self.status = status


def _check(fn: str, status: int):
    if status != FG_OK:
        raise FgError(fn, status)


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream=None) -> Optional[int]:
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


# ----------------------------------------------------------------------------- containers


class Q4Weight:
    """A 4-bit weight W[K][N] on the device: ``codes`` uint8 [K][N/2], ``ab`` int32
    [K][N/64] (a in the low 16 bits, b in the high 16 bits)."""

    def __init__(self, codes, ab, K: int, N: int):
        self.codes, self.ab, self.K, self.N = codes, ab, int(K), int(N)

    @classmethod
    def from_fp16(cls, w, stream=None) -> "Q4Weight":
        import torch
        K, N = w.shape
        codes = torch.empty((K, N // 2), dtype=torch.uint8, device=w.device)
        ab = torch.empty((K, N // 64), dtype=torch.int32, device=w.device)
        fg_quantize_g64(w, codes, ab, stream)
        return cls(codes, ab, K, N)

    def struct(self) -> fg_q4mat:
        return fg_q4mat(_ptr(self.codes), _ptr(self.ab), self.K, self.N)


class KVCacheQ4:
    """One layer's 4-bit KV cache: codes [B][H][cap][d/2] uint8, ab [B][H][cap][d/64]
    int32, for K and V.  ``cap`` is rounded up to a multiple of 16 positions."""

    def __init__(self, B: int, cap: int, h: int, H: int, device="cuda"):
        import torch
        cap = (int(cap) + 15) // 16 * 16
        d = h // H
        self.B, self.cap, self.h, self.H, self.d = B, cap, h, H, d
        self.k_codes = torch.zeros((B, H, cap, d // 2), dtype=torch.uint8, device=device)
        self.v_codes = torch.zeros_like(self.k_codes)
        self.k_ab = torch.zeros((B, H, cap, d // 64), dtype=torch.int32, device=device)
        self.v_ab = torch.zeros_like(self.k_ab)

    def struct(self) -> fg_kvcache:
        return fg_kvcache(_ptr(self.k_codes), _ptr(self.v_codes), _ptr(self.k_ab),
                          _ptr(self.v_ab), self.B, self.cap, self.h, self.H)


class LayerQ4:
    """One decoder layer's device parameters (4-bit weights, fp16 vectors)."""

    def __init__(self, h: int, H: int, f: int, wqkv: Q4Weight, wo: Q4Weight,
                 w1: Optional[Q4Weight], w2: Optional[Q4Weight], vec: dict, ln_eps=1e-5):
        self.h, self.H, self.d, self.f, self.ln_eps = h, H, h // H, f, ln_eps
        self.wqkv, self.wo, self.w1, self.w2, self.vec = wqkv, wo, w1, w2, vec

    @classmethod
    def from_fp16(cls, params: dict, H: int, ln_eps=1e-5, device="cuda", stream=None):
        """Quantise fp16 parameters (numpy or torch, W[K][N] layout) on the device."""
        import torch

        def dev(a):
            t = a if isinstance(a, torch.Tensor) else torch.from_numpy(a)
            return t.to(device=device, dtype=torch.float16).contiguous()

        h = params["wo"].shape[0]
        f = params["w1"].shape[1] if "w1" in params else 0
        wq = Q4Weight.from_fp16(dev(params["wqkv"]), stream)
        wo = Q4Weight.from_fp16(dev(params["wo"]), stream)
        w1 = Q4Weight.from_fp16(dev(params["w1"]), stream) if f else None
        w2 = Q4Weight.from_fp16(dev(params["w2"]), stream) if f else None
        vec = {k: dev(v) for k, v in params.items() if k not in ("wqkv", "wo", "w1", "w2")}
        return cls(h, H, f, wq, wo, w1, w2, vec, ln_eps)

    def dims(self) -> fg_dims:
        return fg_dims(self.h, self.H, self.d, self.f, self.ln_eps)

    def struct(self) -> fg_layer:
        z = fg_q4mat(None, None, 0, 0)
        v = self.vec
        return fg_layer(self.wqkv.struct(), self.wo.struct(),
                        self.w1.struct() if self.w1 else z, self.w2.struct() if self.w2 else z,
                        _ptr(v.get("bqkv")), _ptr(v.get("bo")), _ptr(v.get("b1")),
                        _ptr(v.get("b2")), _ptr(v["ln1_g"]), _ptr(v["ln1_b"]),
                        _ptr(v.get("ln2_g")), _ptr(v.get("ln2_b")))


# ----------------------------------------------------------------------------- calls


def fg_quantize_g64(x, codes, ab, stream=None):
    rows, cols = x.shape
    _check("fg_quantize_g64", lib.fg_quantize_g64(_ptr(x), rows, cols, _ptr(codes), _ptr(ab),
                                                  _stream(stream)))


def fg_dequant_g64(codes, ab, rows: int, cols: int, y, stream=None):
    _check("fg_dequant_g64", lib.fg_dequant_g64(_ptr(codes), _ptr(ab), rows, cols, _ptr(y),
                                                _stream(stream)))


def fg_gemm_workspace_bytes(M: int, K: int, N: int) -> int:
    return int(lib.fg_gemm_workspace_bytes(M, K, N))


def fg_dequant_gemm_q4(X, W: Q4Weight, bias, epilogue: int, residual, Y, ws=None, stream=None):
    M = X.shape[0]
    wsb = 0 if ws is None else ws.numel() * ws.element_size()
    st = W.struct()
    _check("fg_dequant_gemm_q4",
           lib.fg_dequant_gemm_q4(_ptr(X), M, C.byref(st), _ptr(bias), epilogue, _ptr(residual),
                                  _ptr(Y), _ptr(ws), wsb, _stream(stream)))


def fg_dequant_gemm_q4_kv(X, W: Q4Weight, bias, Y, cache: KVCacheQ4, T: int, pos: int, ws=None,
                          stream=None):
    M = X.shape[0]
    wsb = 0 if ws is None else ws.numel() * ws.element_size()
    st, kst = W.struct(), cache.struct()
    _check("fg_dequant_gemm_q4_kv",
           lib.fg_dequant_gemm_q4_kv(_ptr(X), M, C.byref(st), _ptr(bias), _ptr(Y), C.byref(kst),
                                     T, pos, _ptr(ws), wsb, _stream(stream)))


def fg_dequant_gemm_q4_ln(X, W: Q4Weight, bias, epilogue: int, residual, Y, gamma, beta,
                          eps: float, Y_ln, ws=None, stream=None):
    M = X.shape[0]
    wsb = 0 if ws is None else ws.numel() * ws.element_size()
    st = W.struct()
    _check("fg_dequant_gemm_q4_ln",
           lib.fg_dequant_gemm_q4_ln(_ptr(X), M, C.byref(st), _ptr(bias), epilogue, _ptr(residual),
                                     _ptr(Y), _ptr(gamma), _ptr(beta), eps, _ptr(Y_ln), _ptr(ws),
                                     wsb, _stream(stream)))


def fg_kv_append_q4(k_new, v_new, row_stride: int, T: int, pos: int, cache: KVCacheQ4,
                    stream=None):
    st = cache.struct()
    _check("fg_kv_append_q4", lib.fg_kv_append_q4(_ptr(k_new), _ptr(v_new), row_stride, T, pos,
                                                  C.byref(st), _stream(stream)))


def fg_decode_attn_workspace_bytes(cache: KVCacheQ4, length: int) -> int:
    st = cache.struct()
    return int(lib.fg_decode_attn_workspace_bytes(C.byref(st), length))


def fg_decode_attn_q4kv(q, q_stride: int, cache: KVCacheQ4, length: int, scale: float, out,
                        ws=None, stream=None):
    st = cache.struct()
    wsb = 0 if ws is None else ws.numel() * ws.element_size()
    _check("fg_decode_attn_q4kv",
           lib.fg_decode_attn_q4kv(_ptr(q), q_stride, C.byref(st), length, scale, _ptr(out),
                                   _ptr(ws), wsb, _stream(stream)))


def fg_decode_attn_topk_workspace_bytes(cache: KVCacheQ4, length: int) -> int:
    st = cache.struct()
    return int(lib.fg_decode_attn_topk_workspace_bytes(C.byref(st), length))


def fg_decode_attn_q4kv_topk(q, q_stride: int, cache: KVCacheQ4, length: int, k: int,
                             scale: float, out, ws, sel=None, stream=None):
    """Top-K sparse decode attention: softmax over all positions' scores, values of the k
    highest-scoring positions only; ``sel`` (optional int32 [B][H][k]) receives them."""
    st = cache.struct()
    wsb = 0 if ws is None else ws.numel() * ws.element_size()
    _check("fg_decode_attn_q4kv_topk",
           lib.fg_decode_attn_q4kv_topk(_ptr(q), q_stride, C.byref(st), length, k, scale,
                                        _ptr(out), _ptr(sel), _ptr(ws), wsb, _stream(stream)))


DECODE_ATTN_STATIC_SCRATCH_BYTES = 4 << 20


def fg_decode_attn_q4kv_static(q, q_stride: int, cache: KVCacheQ4, length: int, scale: float,
                               out, stream=None):
    """Decode attention for callers that cannot allocate: the split scratch is the
    library's own static device array (4 MiB), so no workspace is passed."""
    st = cache.struct()
    _check("fg_decode_attn_q4kv_static",
           lib.fg_decode_attn_q4kv_static(_ptr(q), q_stride, C.byref(st), length, scale,
                                          _ptr(out), _stream(stream)))


def fg_prefill_attn(qkv, nseq: int, s: int, H: int, d: int, scale: float, out, stream=None):
    _check("fg_prefill_attn", lib.fg_prefill_attn(_ptr(qkv), nseq, s, H, d, scale, _ptr(out),
                                                  _stream(stream)))


def fg_layernorm(x, gamma, beta, eps: float, y, stream=None):
    rows, h = x.shape
    _check("fg_layernorm", lib.fg_layernorm(_ptr(x), rows, h, _ptr(gamma), _ptr(beta), eps,
                                            _ptr(y), _stream(stream)))


def fg_workspace_bytes(layer: LayerQ4, g: int, m: int, s_max: int) -> int:
    """Scratch bytes of fg_layer_prefill / fg_layer_decode for this layer's dims."""
    dm = layer.dims()
    return int(lib.fg_workspace_bytes(C.byref(dm), g, m, s_max))


fg_layer_workspace_bytes = fg_workspace_bytes


def fg_layer_prefill(layer: LayerQ4, cache: KVCacheQ4, x, y, g: int, m: int, s: int, ws,
                     stream=None):
    dm, L, kv = layer.dims(), layer.struct(), cache.struct()
    _check("fg_layer_prefill",
           lib.fg_layer_prefill(C.byref(dm), C.byref(L), C.byref(kv), _ptr(x), _ptr(y), g, m, s,
                                _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def fg_layer_decode(layer: LayerQ4, cache: KVCacheQ4, x, y, g: int, m: int, pos: int, ws,
                    stream=None):
    dm, L, kv = layer.dims(), layer.struct(), cache.struct()
    _check("fg_layer_decode",
           lib.fg_layer_decode(C.byref(dm), C.byref(L), C.byref(kv), _ptr(x), _ptr(y), g, m, pos,
                               _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def fg_check_device_error(stream=None):
    _check("fg_check_device_error", lib.fg_check_device_error(_stream(stream)))


def fg_prof_enable(on: bool = True):
    lib.fg_prof_enable(1 if on else 0)


def fg_prof_reset():
    lib.fg_prof_reset()


def fg_prof_query(kind: int):
    n, ms, work = C.c_int64(), C.c_double(), C.c_double()
    _check("fg_prof_query", lib.fg_prof_query(kind, C.byref(n), C.byref(ms), C.byref(work)))
    return {"kernel": lib.fg_kernel_name(kind).decode(), "launches": n.value, "ms": ms.value,
            "work": work.value}


# ----------------------------------------------------------------------------- stack


class StackEngine:
    """A stack of layers over one block of B = g*m sequences: prefill over the prompt,
    then decode steps, each running every layer over the whole block before the next
    (the block schedule).  Orchestration only -- each layer step is one C call."""

    def __init__(self, layers, g: int, m: int, cap: int, s_max: int, device="cuda"):
        import torch
        self.layers, self.g, self.m, self.cap = layers, g, m, cap
        L0 = layers[0]
        self.B = g * m
        self.caches = [KVCacheQ4(self.B, cap, L0.h, L0.H, device) for _ in layers]
        wsb = max(fg_workspace_bytes(L, g, m, max(s_max, cap)) for L in layers)
        self.ws = torch.empty((wsb + 255) // 256 * 256, dtype=torch.uint8, device=device)

    def prefill(self, x, y, s: int, stream=None):
        """x, y: [B][s][h] fp16 (may alias); runs every layer over the prompt."""
        cur = x
        for L, c in zip(self.layers, self.caches):
            fg_layer_prefill(L, c, cur, y, self.g, self.m, s, self.ws, stream)
            cur = y
        return y

    def decode(self, x, y, pos: int, stream=None):
        """One decode step: x, y [B][h]; appends at ``pos`` in every layer's cache."""
        cur = x
        for L, c in zip(self.layers, self.caches):
            fg_layer_decode(L, c, cur, y, self.g, self.m, pos, self.ws, stream)
            cur = y
        return y
