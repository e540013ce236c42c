"""One pre-LN OPT decoder layer over INT4 weights and an INT4 KV cache (oracle).

Test infrastructure only.  Plain numpy, float64 by default (``dt`` may be float32 for
the large sampled workloads), no blocking, fusion or reordering.

What the pages fix:
* the layer is QKV projections, attention, output projection and an MLP; one layer's
  FP16 weights are 8*h1^2 + 4*h1*h2 bytes, i.e. four h x h matrices and two h x h2 ones
  (FlexGen paper explainer, "Cost Model and Policy Search", the dtoc_g term);
* weights and K/V are stored 4-bit group-wise and dequantised to FP16 before compute
  (FlexGen review, jaehun.me, section "4-bit 압축은 정수 연산 가속과 같은가");
* generation is a prefill over the prompt that builds the KV cache, then decode steps
  that each add one token per sequence and read the cache (FlexGen paper explainer,
  "Problem Formulation", Figure 2; "论文阅读：FlexGen", §1);
* the cost model charges one prefill and n-1 decode steps per layer
  (FlexGen paper explainer, "Analytical Cost Model", T = Tpre*l + Tgen*(n-1)*l).

Readings where the pages are silent (the workload definition fixes pre-LN and ReLU):
R5  prefill attends over the fp16 K/V the projection produced; decode attends over the
    dequantised cache including the token just appended.
R6  h1 = x + Attn(LN1(x)) Wo + bo ;  y = h1 + ReLU(LN2(h1) W1 + b1) W2 + b2, with
    Q,K,V = LN1(x) Wqkv + bqkv; LayerNorm with population variance and eps 1e-5;
    scores scaled by 1/sqrt(d); causal mask lets position i see j <= i; softmax in the
    usual max-subtracted form.  f == 0 means an attention block without the MLP.
R7  K and V are rounded to fp16 where they enter the quantiser (the quantiser is defined
    on fp16 values); every other intermediate stays in ``dt``.
R9  a run is a prefill followed by n-1 decode steps; the cache holds s+n positions.
R10 the input of each decode step is a fresh hidden state per sequence (no embedding or
    LM head in a layer stack).
"""
from __future__ import annotations

from typing import Dict, List, Optional

import numpy as np

from .quant import quantize_g64, dequant_g64

F64 = np.float64


def layernorm(x, gamma, beta, eps: float, dt=F64):
    """LayerNorm over the last axis: (x - mean) / sqrt(var + eps) * gamma + beta with the
    population variance.  Parity: pinned by a pure-Python loop and by the mean-0 /
    variance-1 property at gamma = 1, beta = 0."""
    x = np.asarray(x, dtype=dt)
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    return (x - mu) / np.sqrt(var + dt(eps)) * np.asarray(gamma, dt) + np.asarray(beta, dt)


def relu(x):
    return np.maximum(x, 0)


def _heads(x, H, d):
    S_, T, _ = x.shape
    return x.reshape(S_, T, H, d).transpose(0, 2, 1, 3)


def causal_attention(q, k, v, H: int, d: int, dt=F64):
    """softmax(Q K^T / sqrt(d) + causal mask) V per head; q, k, v [S][T][h] -> [S][T][h].
    Parity: pinned by a pure-Python loop, one-token = v, equal scores = running mean."""
    q, k, v = (np.asarray(t, dtype=dt) for t in (q, k, v))
    S_, T, h = q.shape
    qh, kh, vh = _heads(q, H, d), _heads(k, H, d), _heads(v, H, d)
    sc = (qh @ kh.transpose(0, 1, 3, 2)) / np.sqrt(dt(d))
    sc = np.where(np.triu(np.ones((T, T), dtype=bool), 1), -np.inf, sc)
    sc = sc - sc.max(axis=-1, keepdims=True)
    p = np.exp(sc)
    p = p / p.sum(axis=-1, keepdims=True)
    o = p @ vh
    return o.transpose(0, 2, 1, 3).reshape(S_, T, h)


def decode_attention(q, K, V, H: int, d: int, dt=F64):
    """One query per sequence over T cached positions: q [S][h], K, V [S][T][h] -> [S][h].
    Parity: pinned by a pure-Python loop and the one-position / equal-score cases."""
    q, K, V = (np.asarray(t, dtype=dt) for t in (q, K, V))
    S_, T, h = K.shape
    qh = q.reshape(S_, H, 1, d)
    kh, vh = _heads(K, H, d), _heads(V, H, d)
    sc = (qh @ kh.transpose(0, 1, 3, 2)) / np.sqrt(dt(d))     # [S][H][1][T]
    sc = sc - sc.max(axis=-1, keepdims=True)
    p = np.exp(sc)
    p = p / p.sum(axis=-1, keepdims=True)
    return (p @ vh).reshape(S_, h)


def decode_attention_topk(q, K, V, H: int, d: int, k: int, dt=F64, selected=None):
    """Top-K sparse decode attention: the scores of all T positions come from K, the
    softmax runs over all of them, and only the k positions with the highest scores
    contribute their values: o = sum_{t in top-k} p_t v_t, without renormalising
    [论文阅读：FlexGen, §3.4 "4-bit 压缩权重和 KV cache": optional sparse attention that
    loads only the top 10% of the value cache; FlexGen paper explainer, §3.3 "Roadmap for
    the Deep Dive": Top-K sparse attention, an approximate method that cuts I/O volume].  Readings: p is the full softmax (loading fewer values
    drops terms, it does not change the others); equal scores at the k-th place go to the
    lower position.  q [S][h], K, V [S][T][h] -> ([S][h], top-k positions [S][H][k] in
    decreasing score order).

    ``selected`` ([S][H][k] positions), when given, replaces the selection: the output is
    then the same weighted sum over those positions (used to evaluate another
    implementation's choice among near-equal scores).  Parity: pinned by k = T reducing to
    dense decode attention, k = 1 to the single largest term, and a pure-Python loop."""
    q, K, V = (np.asarray(t, dtype=dt) for t in (q, K, V))
    S_, T, h = K.shape
    qh = q.reshape(S_, H, 1, d)
    kh, vh = _heads(K, H, d), _heads(V, H, d)
    sc = ((qh @ kh.transpose(0, 1, 3, 2)) / np.sqrt(dt(d)))[:, :, 0, :]      # [S][H][T]
    e = np.exp(sc - sc.max(axis=-1, keepdims=True))
    p = e / e.sum(axis=-1, keepdims=True)
    if selected is None:
        # stable sort on -score: among equal scores the lower position comes first
        selected = np.argsort(-sc, axis=-1, kind="stable")[:, :, :k]
    sel = np.asarray(selected)
    w = np.take_along_axis(p, sel, axis=-1)                                   # [S][H][k]
    vs = np.take_along_axis(vh, sel[..., None], axis=2)                       # [S][H][k][d]
    o = (w[..., None] * vs).sum(axis=2)
    return o.reshape(S_, h), sel


def topk_count(T: int, frac: float = 0.1) -> int:
    """Positions kept by a top-fraction rule: ceil(frac * T), at least one."""
    return max(1, int(np.ceil(frac * T - 1e-9)))


class QuantLayer:
    """A layer's weights quantised once (R1-R3) and restored to fp16 (R4).

    ``q[name]``, ``a[name]``, ``b[name]`` hold codes (unpacked) and group statistics of
    each weight W[K][N] (groups of 64 along the output channel N); ``w_hat[name]`` is
    the fp16 matrix every product uses."""

    WEIGHTS = ("wqkv", "wo", "w1", "w2")

    def __init__(self, params: Dict[str, np.ndarray], H: int, d: int, eps: float = 1e-5,
                 keep_codes: bool = True):
        self.H, self.d, self.eps = H, d, eps
        self.h = params["wo"].shape[0]
        self.f = params["w1"].shape[1] if "w1" in params else 0
        self.q: Dict[str, np.ndarray] = {}
        self.a: Dict[str, np.ndarray] = {}
        self.b: Dict[str, np.ndarray] = {}
        self.w_hat: Dict[str, np.ndarray] = {}
        for name in self.WEIGHTS:
            if name not in params:
                continue
            q, a, b = quantize_g64(params[name])
            self.w_hat[name] = dequant_g64(q, a, b)
            if keep_codes:
                self.q[name], self.a[name], self.b[name] = q, a, b
        self.vec = {k: np.asarray(v, dtype=np.float16) for k, v in params.items()
                    if k not in self.WEIGHTS}


class KVCache:
    """Per-layer INT4 cache for S sequences: codes [S][cap][h] (unpacked), a and b
    [S][cap][h/64], groups of 64 along the hidden dimension."""

    def __init__(self, S: int, cap: int, h: int):
        self.S, self.cap, self.h = S, cap, h
        self.qk = np.zeros((S, cap, h), np.uint8)
        self.qv = np.zeros((S, cap, h), np.uint8)
        g = h // 64
        self.ak = np.zeros((S, cap, g), np.float16)
        self.bk = np.zeros((S, cap, g), np.float16)
        self.av = np.zeros((S, cap, g), np.float16)
        self.bv = np.zeros((S, cap, g), np.float16)
        self.length = 0

    def append(self, k16: np.ndarray, v16: np.ndarray, pos: int):
        """Quantise K/V rows [S][T][h] (fp16) into positions pos .. pos+T-1."""
        S_, T, h = k16.shape
        assert pos + T <= self.cap, "cache capacity exceeded"
        for src, qd, ad, bd in ((k16, self.qk, self.ak, self.bk),
                                (v16, self.qv, self.av, self.bv)):
            q, a, b = quantize_g64(src.reshape(S_ * T, h))
            qd[:, pos:pos + T] = q.reshape(S_, T, h)
            ad[:, pos:pos + T] = a.reshape(S_, T, h // 64)
            bd[:, pos:pos + T] = b.reshape(S_, T, h // 64)
        self.length = max(self.length, pos + T)

    def dequant(self, upto: int):
        """fp16 K^, V^ [S][upto][h] of positions 0 .. upto-1 (R4)."""
        S_, h = self.S, self.h
        out = []
        for q, a, b in ((self.qk, self.ak, self.bk), (self.qv, self.av, self.bv)):
            x = dequant_g64(q[:, :upto].reshape(S_ * upto, h),
                            a[:, :upto].reshape(S_ * upto, h // 64),
                            b[:, :upto].reshape(S_ * upto, h // 64))
            out.append(x.reshape(S_, upto, h))
        return out[0], out[1]


def _mlp_and_residual(L: QuantLayer, h1, dt):
    if L.f == 0:
        return h1
    v = L.vec
    u = layernorm(h1, v["ln2_g"], v["ln2_b"], L.eps, dt)
    mid = relu(u @ L.w_hat["w1"].astype(dt) + v["b1"].astype(dt))
    return h1 + mid @ L.w_hat["w2"].astype(dt) + v["b2"].astype(dt)


def layer_prefill(L: QuantLayer, x, cache: KVCache, dt=F64):
    """Prefill of one layer over prompts x [S][s][h]; writes K/V of positions 0..s-1
    into ``cache`` and returns the layer output [S][s][h] (R5-R7)."""
    v = L.vec
    h = L.h
    x = np.asarray(x, dtype=dt)
    a = layernorm(x, v["ln1_g"], v["ln1_b"], L.eps, dt)
    qkv = a @ L.w_hat["wqkv"].astype(dt) + v["bqkv"].astype(dt)
    q, k, vv = qkv[..., :h], qkv[..., h:2 * h], qkv[..., 2 * h:]
    k16, v16 = k.astype(np.float16), vv.astype(np.float16)
    cache.append(k16, v16, 0)
    attn = causal_attention(q, k16, v16, L.H, L.d, dt)
    h1 = x + attn @ L.w_hat["wo"].astype(dt) + v["bo"].astype(dt)
    return _mlp_and_residual(L, h1, dt)


def layer_decode(L: QuantLayer, x, cache: KVCache, pos: int, dt=F64):
    """One decode step of one layer: x [S][h] is the new token of each sequence, ``pos``
    the cache length before the step.  Appends its K/V at ``pos`` and attends over
    positions 0..pos (R5-R7).  Returns [S][h]."""
    v = L.vec
    h = L.h
    x = np.asarray(x, dtype=dt)
    a = layernorm(x, v["ln1_g"], v["ln1_b"], L.eps, dt)
    qkv = a @ L.w_hat["wqkv"].astype(dt) + v["bqkv"].astype(dt)
    q, k, vv = qkv[..., :h], qkv[..., h:2 * h], qkv[..., 2 * h:]
    cache.append(k.astype(np.float16)[:, None, :], vv.astype(np.float16)[:, None, :], pos)
    K, V = cache.dequant(pos + 1)
    attn = decode_attention(q, K, V, L.H, L.d, dt)
    h1 = x + attn @ L.w_hat["wo"].astype(dt) + v["bo"].astype(dt)
    return _mlp_and_residual(L, h1, dt)


def run_stack(layers: List[QuantLayer], x_prompt, x_steps, cap: Optional[int] = None,
              dt=F64, keep_layer_outputs: bool = False):
    """The generation loop over a layer stack for S sequences (R9, R10).

    x_prompt [S][s][h]; x_steps [n-1][S][h].  Prefill runs every layer over the prompt;
    then each decode step t = 1 .. n-1 runs every layer on x_steps[t-1] with the cache
    length pos = s + t - 1.  Returns a dict with the final prefill output [S][s][h], the
    decode outputs [n-1][S][h] and the per-layer caches."""
    S_, s, h = x_prompt.shape
    n_dec = x_steps.shape[0]
    cap = s + n_dec + 1 if cap is None else cap
    caches = [KVCache(S_, cap, h) for _ in layers]
    per_layer = []
    y = np.asarray(x_prompt, dtype=dt)
    for L, c in zip(layers, caches):
        y = layer_prefill(L, y, c, dt)
        if keep_layer_outputs:
            per_layer.append(y.copy())
    prefill = y
    steps = np.zeros((n_dec, S_, h), dtype=dt)
    for t in range(1, n_dec + 1):
        y = np.asarray(x_steps[t - 1], dtype=dt)
        for L, c in zip(layers, caches):
            y = layer_decode(L, y, c, s + t - 1, dt)
        steps[t - 1] = y
    out = {"prefill": prefill, "steps": steps, "caches": caches}
    if keep_layer_outputs:
        out["prefill_layers"] = per_layer
    return out
